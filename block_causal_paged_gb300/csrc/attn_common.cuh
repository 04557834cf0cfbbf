// Parts shared by the attention kernels (attention.cu: one CTA per SM;
// attention_pair.cu: CTA pairs with two-SM tensor-core MMAs): the record
// ring that carries work items and KV tiles from the planner warp to the
// other roles, bounded barrier waits, and the planner itself.
//
// The visibility rule ("Inference for Interpretable Text-Diffusion Models",
// "Background"; "Inference: Fewer, smaller forwards", "Advancement 13") is
// evaluated per row as a key-position limit: a query at position q sees key
// position k iff k < lim(q), lim(q) = P0 if q < P0 else P0 + D*(floor((q-P0)/D)+1).
// Each KV tile is classified against an item's rows ("FlexAttention with
// Aligned Tiles"): fully included (no mask arithmetic), partially included
// (elementwise mask) or fully excluded (not emitted: no load, no math).
#pragma once

#include <climits>
#include <cstdint>

#include "bca_internal.h"
#include "ptx_sm103.cuh"

namespace bca {
namespace attn {

constexpr int kNumRec = 8;      // record ring entries
constexpr int kMailSlots = 4;   // item-index mailbox of a CTA pair
constexpr int kErrTimeout = -18;
constexpr int kErrPageOob = -16;
constexpr int kErrBadLength = -17;
constexpr int kErrWorkspace = -4;

enum RecKind : int { kRecItem = 0, kRecTile = 1, kRecEnd = 2 };

// Record ring entry (128 bytes).  Item fields:
enum : int {
  I_KIND = 0, I_NT = 1, I_NM = 2, I_QMODE = 3, I_QTOK = 4 /*2*/, I_QHEAD = 6 /*2*/,
  I_NTOK = 8 /*2*/, I_QBASE = 10 /*2*/, I_P0 = 12, I_DBLK = 13, I_SPLIT = 14
};
// Tile fields (one coordinate and one position offset per 16-key chunk):
enum : int {
  T_KIND = 0, T_SRC = 1, T_FULL = 2, T_NVALID = 3, T_HEAD = 4, T_KMODE = 5, T_KBASE = 6,
  T_COORD = 8 /*8*/, T_KOFF = 16 /*8*/
};
struct __align__(16) Rec {
  int32_t w[32];
};

__device__ __forceinline__ void record_error(const AttnParams& p, int code) {
  atomicCAS(&p.hdr->status, 0, code);
}

// A wait ran out of time (or another role of this CTA gave up first): stop
// every role of the CTA, record the timeout, and -- for the first wait of
// the launch that really timed out -- which CTA, warp and barrier it was.
template <class Ctx>
__device__ __forceinline__ void give_up(const Ctx& c, const AttnParams& p, const uint64_t* bar,
                                        uint32_t parity) {
  const bool first = *c.abort_flag == 0;
  *c.abort_flag = 1;
  record_error(p, kErrTimeout);
  if (first && atomicCAS(&p.hdr->wait_fail[0], 0, 1) == 0) {
    p.hdr->wait_fail[1] = (int32_t)blockIdx.x;
    p.hdr->wait_fail[2] = (int32_t)(threadIdx.x >> 5);
    p.hdr->wait_fail[3] = (int32_t)(reinterpret_cast<uintptr_t>(bar) -
                                    reinterpret_cast<uintptr_t>(c.smem));
    p.hdr->wait_fail[4] = (int32_t)parity;
  }
}

template <class Ctx>
__device__ __forceinline__ bool wait_bar(const Ctx& c, const AttnParams& p, uint64_t* bar,
                                         uint32_t parity) {
  if (mbar_wait(bar, parity, c.abort_flag, kWaitTimeoutCycles)) return true;
  give_up(c, p, bar, parity);
  return false;
}

// Wait on a barrier that threads of the other CTA of a pair arrive on
// (acquire at cluster scope).
template <class Ctx>
__device__ __forceinline__ bool wait_bar_cluster(const Ctx& c, const AttnParams& p, uint64_t* bar,
                                                 uint32_t parity) {
  if (mbar_wait_cluster(bar, parity, c.abort_flag, kWaitTimeoutCycles)) return true;
  give_up(c, p, bar, parity);
  return false;
}
template <class Ctx>
__device__ __forceinline__ bool wait_bar_warp_cluster(const Ctx& c, const AttnParams& p,
                                                      uint64_t* bar, uint32_t parity) {
  const bool ok = wait_bar_cluster(c, p, bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Whole-warp wait with a warp-uniform outcome.
template <class Ctx>
__device__ __forceinline__ bool wait_bar_warp(const Ctx& c, const AttnParams& p, uint64_t* bar,
                                              uint32_t parity) {
  const bool ok = wait_bar(c, p, bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Key-position limit of a query at position q (block rule).
__device__ __forceinline__ int row_limit(int q, int P0, int D) {
  if (q < P0) return P0;
  return P0 + D * ((q - P0) / D + 1);
}

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ long long warp_excl_scan_ll(long long v, int lane) {
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x - v;
}

// ============================================================================
// planner (warp 3)
// ============================================================================
template <class Ctx, bool kPair>
struct Planner {
  const AttnParams& p;
  const Ctx& c;
  int lane;
  uint32_t idx = 0;   // records written
  bool ok = true;
  unsigned long long n_full = 0, n_partial = 0, n_skip = 0;
  int page_err = 0;

  __device__ Planner(const AttnParams& p_, const Ctx& c_, int lane_) : p(p_), c(c_), lane(lane_) {}

  // Wait for a free ring entry; returns it (all lanes get the pointer).
  __device__ __forceinline__ Rec* acquire() {
    const uint32_t slot = idx % kNumRec;
    if (!wait_bar_warp(c, p, &c.bar.rec_empty[slot], ((idx / kNumRec) & 1) ^ 1)) {
      ok = false;
      return nullptr;
    }
    return &c.ring[slot];
  }
  __device__ void publish() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.bar.rec_full[idx % kNumRec]);
    __syncwarp();
    ++idx;
  }
  __device__ void emit_end() {
    Rec* r = acquire();
    if (!r) return;
    if (lane == 0) r->w[I_KIND] = kRecEnd;
    publish();
  }

  // Emit one tile record.  coord[i]: per 16-key chunk, pool row / dense token
  // coordinate (already out of range for chunks with no valid key).
  __device__ __forceinline__ void emit_tile(int src, int full, int nvalid, int head, int kmode,
                                            int kbase, const int (&coord)[kChunksPerTile],
                                            const int (&koff)[kChunksPerTile]) {
    Rec* r = acquire();
    if (!r) return;
    // the MMA warp never reads tile records: release this one on its behalf
    // (counts toward the phase that frees the entry again); a pair's second
    // CTA has no MMA warp among the ring's consumers
    if (lane == 0 && lead()) mbar_arrive(&c.bar.rec_empty[idx % kNumRec]);
    if (lane == 0) {
      r->w[T_KIND] = kRecTile;
      r->w[T_SRC] = src;
      r->w[T_FULL] = full;
      r->w[T_NVALID] = nvalid;
      r->w[T_HEAD] = head;
      r->w[T_KMODE] = kmode;
      r->w[T_KBASE] = kbase;
#pragma unroll
      for (int i = 0; i < kChunksPerTile; ++i) {
        r->w[T_COORD + i] = coord[i];
        r->w[T_KOFF + i] = koff[i];
      }
    }
    publish();
    if (full) ++n_full; else ++n_partial;
  }

  __device__ __forceinline__ void emit_item(int n_tiles, int n_m, int qmode, const int (&qtok)[2],
                            const int (&qhead)[2], const int (&ntok)[2], const int (&qbase)[2],
                            int P0, int Dblk, int split) {
    Rec* r = acquire();
    if (!r) return;
    if (lane == 0) {
      r->w[I_KIND] = kRecItem;
      r->w[I_NT] = n_tiles;
      r->w[I_NM] = n_m;
      r->w[I_QMODE] = qmode;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        r->w[I_QTOK + m] = qtok[m];
        r->w[I_QHEAD + m] = qhead[m];
        r->w[I_NTOK + m] = ntok[m];
        r->w[I_QBASE + m] = qbase[m];
      }
      r->w[I_P0] = P0;
      r->w[I_DBLK] = Dblk;
      r->w[I_SPLIT] = split;
    }
    publish();
  }

  // Page id of logical key position k of sequence b (all lanes call with
  // their own k); returns -1 for an out-of-range id and flags the error.
  __device__ int page_of(int b, int k) {
    const int pidx = k / p.S;
    int page = -1;
    if (pidx >= 0 && pidx < p.max_pages) page = __ldg(p.page_table + (size_t)b * p.max_pages + pidx);
    if (page < 0 || page >= p.num_pages) {
      page_err = 1;
      page = -1;
    }
    return page;
  }

  // Raw page-table entry for chunk (lane % 8) of tile tg + lane / 8 of
  // sequence b (INT_MIN: no key there), and its pool row coordinate for KV
  // head g (out of range -- zero fill -- for no key or a bad page id, which
  // is flagged).  The load and its use are split so that the load of the
  // next group of tiles is in flight while the current group is emitted.
  __device__ __forceinline__ int group_page_raw(int b, int P, int tg, int t1) const {
    const int t = tg + lane / kChunksPerTile;
    const int k = t * kTileKeys + (lane % kChunksPerTile) * kChunkKeys;
    if (t >= t1 || k >= P) return INT_MIN;
    const int pidx = k / p.S;
    if (pidx >= p.max_pages) return -1;
    return __ldg(p.page_table + (size_t)b * p.max_pages + pidx);
  }
  __device__ __forceinline__ int group_coord(int raw, int g, int tg) {
    if (raw == INT_MIN) return p.pool_rows;
    if (raw < 0 || raw >= p.num_pages) {
      page_err = 1;
      return p.pool_rows;
    }
    const int t = tg + lane / kChunksPerTile;
    const int k = t * kTileKeys + (lane % kChunksPerTile) * kChunkKeys;
    return (raw * p.Hkv + g) * p.S + (k % p.S);
  }

  // Emit the prefix tiles [t0, t1) of a decode/paged stream, keys 0..P-1 of
  // sequence b, KV head g.  Page-table entries for 4 tiles (32 chunks, one
  // per lane) are fetched at once, one group ahead of the group emitted.
  __device__ void emit_pool_tiles_contig(int b, int g, int P, int t0, int t1) {
    constexpr int kTilesPerGroup = 32 / kChunksPerTile;
    int raw_next = group_page_raw(b, P, t0, t1);
    for (int tg = t0; tg < t1 && ok; tg += kTilesPerGroup) {
      const int raw = raw_next;
      if (tg + kTilesPerGroup < t1) raw_next = group_page_raw(b, P, tg + kTilesPerGroup, t1);
      const int coord = group_coord(raw, g, tg);
      const int ntile = min(kTilesPerGroup, t1 - tg);
      for (int j = 0; j < ntile && ok; ++j) {
        int cd[kChunksPerTile], ko[kChunksPerTile];
#pragma unroll
        for (int i = 0; i < kChunksPerTile; ++i) {
          cd[i] = __shfl_sync(0xffffffffu, coord, kChunksPerTile * j + i);
          ko[i] = 0;
        }
        const int tt = tg + j;
        const int nvalid = min(kTileKeys, P - tt * kTileKeys);
        emit_tile(0, nvalid == kTileKeys, nvalid, g, 0, tt * kTileKeys, cd, ko);
      }
    }
  }

  // Dense tile: keys are tokens tok0.. of a dense [tokens, Hkv, d] tensor; key
  // i has position kbase + i (kmode 0) or live_pos[kbase + i] (kmode 2).
  __device__ __forceinline__ void emit_dense_tile(int g, int tok0, int nvalid, int kmode,
                                                  int kbase, int full) {
    int cd[kChunksPerTile], ko[kChunksPerTile];
#pragma unroll
    for (int i = 0; i < kChunksPerTile; ++i) {
      cd[i] = (i * kChunkKeys < nvalid) ? tok0 + i * kChunkKeys : p.dense_tokens;
      ko[i] = 0;
    }
    emit_tile(1, full, nvalid, g, kmode, kbase, cd, ko);
  }

  // --------------------------------------------------------------------------
  // Next work item from the shared counter (zero at launch: the last CTA of
  // the previous launch reset it, as does the plan kernel).
  // Work units (CTAs, or CTA pairs) take their first item by their own
  // index, without the counter's latency, and the rest from the counter,
  // offset by the number of units: every item is handed out exactly once.
  bool grabbed = false;
  __device__ int units() const {
    return kPair ? (int)(gridDim.x / 2) : (int)gridDim.x;
  }
  __device__ int next_index() {
    if (!grabbed) {
      grabbed = true;
      return kPair ? (int)(blockIdx.x / 2) : (int)blockIdx.x;
    }
    return units() + atomicAdd(&p.hdr->work_next, 1);
  }
  __device__ int grab() {
    if constexpr (kPair) {
      return grab_pair();
    } else {
      int idx = 0;
      if (lane == 0) idx = next_index();
      return __shfl_sync(0xffffffffu, idx, 0);
    }
  }

  // The CTA that owns the counters and the tile-record release on the MMA
  // warp's behalf: every CTA, or the first of a pair.
  __device__ __forceinline__ bool lead() const {
    if constexpr (kPair) return c.rank == 0;
    else return true;
  }

  // A CTA pair works on the same items: the first CTA takes the next index
  // (its own pair index first, then from the counter) and posts it into a
  // four-entry mailbox in the second CTA's shared memory; the second CTA
  // reads its mailbox and frees the entry.
  uint32_t n_grab = 0;
  __device__ int grab_pair() {
    const uint32_t k = n_grab++;
    const uint32_t slot = k % kMailSlots, par = (k / kMailSlots) & 1u;
    int idx = INT_MAX;  // on a failed wait: no more items
    if (c.rank == 0) {
      if (!wait_bar_warp_cluster(c, p, &c.bar.mail_empty[slot], par ^ 1u)) {
        ok = false;
      } else {
        if (lane == 0) {
          idx = next_index();
          st_shared_cluster_u32(mapa_shared(smem_u32(&c.mail[slot]), 1), (uint32_t)idx);
          mbar_arrive_remote(mapa_shared(smem_u32(&c.bar.mail_full[slot]), 1));
        }
        idx = __shfl_sync(0xffffffffu, idx, 0);
      }
    } else {
      if (!wait_bar_warp_cluster(c, p, &c.bar.mail_full[slot], par)) {
        ok = false;
      } else {
        idx = *reinterpret_cast<volatile int*>(&c.mail[slot]);
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&c.bar.mail_empty[slot]), 0));
      }
    }
    return idx;
  }

  // --------------------------------------------------------------------------
  // Decode with at most kFusedPlanMax sequences: the planner warp of every CTA
  // computes the plan itself, by the same rules as the plan kernel (chunk of
  // about `waves` items per CTA, never below ch_min tiles and within the
  // workspace; sequences longest first, ties by index; split slots in
  // sequence order), holding sequences 2l and 2l+1 in lane l.  Every CTA gets
  // the same plan; CTA 0 also writes the split tables the epilogue reads.
  __device__ void run_decode_fused() {
    const int B = p.B, D = p.Dblk, per_seq = p.Hkv * p.n_rb;
    int P[2], nt[2], bad = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int b = 2 * lane + k;
      P[k] = 0;
      nt[k] = 0;  // no sequence
      if (b < B) {
        int v = __ldg(p.lens + b);
        if (v < 0 || (!p.causal && v % D != 0) || (long long)v + D > (long long)p.max_pages * p.S) {
          bad = 1;  // treated as an empty prefix, reported in the status word
          v = 0;
        }
        P[k] = v;
        nt[k] = ceil_div(v, kTileKeys) + ceil_div(D, kTileKeys);
      }
    }
    if (__any_sync(0xffffffffu, bad) && blockIdx.x == 0 && lane == 0)
      record_error(p, kErrBadLength);
    const long long tot = warp_sum_ll(nt[0] + nt[1]) * per_seq;
    // work units that run at once: CTAs, or CTA pairs
    const long long units = p.pair ? (long long)gridDim.x / 2 : (long long)gridDim.x;
    const long long target = units * (p.waves > 0 ? p.waves : 1);
    long long ch = (tot + target - 1) / target;
    if (ch < p.ch_min) ch = p.ch_min;
    if (ch < 1) ch = 1;
    int CH = 1, nch[2] = {0, 0};
    for (int guard = 0; guard < 40; ++guard) {
      CH = (int)(ch < (1ll << 30) ? ch : (1ll << 30));
      nch[0] = ceil_div(nt[0], CH);
      nch[1] = ceil_div(nt[1], CH);
      const long long ns =
          warp_sum_ll((nch[0] > 1 ? nch[0] : 0) + (nch[1] > 1 ? nch[1] : 0)) * per_seq;
      const long long ni = warp_sum_ll(nch[0] + nch[1]) * per_seq;
      if (ns <= p.split_cap && ni <= p.items_cap) break;
      ch *= 2;
    }
    // schedule position (rank) of each sequence, then its first item
    int rank[2] = {0, 0}, base[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < kFusedPlanMax; ++j) {
      const int ntj = __shfl_sync(0xffffffffu, nt[j & 1], j >> 1);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = 2 * lane + k;
        rank[k] += (j < B) & ((ntj > nt[k]) | ((ntj == nt[k]) & (j < i)));
      }
    }
#pragma unroll
    for (int j = 0; j < kFusedPlanMax; ++j) {
      const int rj = __shfl_sync(0xffffffffu, rank[j & 1], j >> 1);
      const int itj = __shfl_sync(0xffffffffu, nch[j & 1], j >> 1) * per_seq;
#pragma unroll
      for (int k = 0; k < 2; ++k) base[k] += ((j < B) & (rj < rank[k])) ? itj : 0;
    }
    const long long n_all = warp_sum_ll(nch[0] + nch[1]) * per_seq;
    const int n_items = (int)(n_all < p.items_cap ? n_all : p.items_cap);
    // split slots, sequence order
    const int sz0 = nch[0] > 1 ? nch[0] * per_seq : 0, sz1 = nch[1] > 1 ? nch[1] * per_seq : 0;
    const int sb0 = (int)warp_excl_scan_ll(sz0 + sz1, lane);
    const int sb[2] = {sb0, sb0 + sz0};
    const long long n_slots = warp_sum_ll(sz0 + sz1);
    // The split slots' table, read only by the epilogue kernel: sequence b's
    // entries are written by CTA b (modulo the grid), its lanes in parallel,
    // so that no CTA's first item waits for the whole table
    for (int bb = blockIdx.x; bb < B; bb += gridDim.x) {
      const int o = bb >> 1, kk = bb & 1;  // the lane and register holding sequence bb
      const int nchb = __shfl_sync(0xffffffffu, kk ? nch[1] : nch[0], o);
      const int sbb = __shfl_sync(0xffffffffu, kk ? sb[1] : sb[0], o);
      if (lane == 0) p.split_base[bb] = sbb;
      if (nchb > 1) {
        for (int e = lane; e < per_seq * nchb; e += 32) {
          const int gr = e / nchb, cc = e % nchb;
          const int first = sbb + gr * nchb;
          if (first + cc < p.split_cap)
            p.slot_info[first + cc] =
                make_int4(bb, ((gr / p.n_rb) << 16) | (gr % p.n_rb), first, nchb);
        }
      }
    }
    if (blockIdx.x == 0 && lane == 0) {
      p.hdr->chunk_tiles = CH;
      p.hdr->n_items = n_items;
      p.hdr->n_split_slots = (int)(n_slots < p.split_cap ? n_slots : p.split_cap);
      if (n_slots > p.split_cap || n_all > p.items_cap) record_error(p, kErrWorkspace);
    }
    while (ok) {
      const int idx = grab();
      if (idx >= n_items) break;
      const bool in0 = nch[0] > 0 && base[0] <= idx && idx < base[0] + nch[0] * per_seq;
      const bool in1 = nch[1] > 0 && base[1] <= idx && idx < base[1] + nch[1] * per_seq;
      const unsigned owners = __ballot_sync(0xffffffffu, in0 || in1);
      const int o = __ffs(owners) - 1;
      const int k = __shfl_sync(0xffffffffu, in1 ? 1 : 0, o);
      const int b = 2 * o + k;
      const int Pb = __shfl_sync(0xffffffffu, k ? P[1] : P[0], o);
      const int ntb = __shfl_sync(0xffffffffu, k ? nt[1] : nt[0], o);
      const int nchb = __shfl_sync(0xffffffffu, k ? nch[1] : nch[0], o);
      const int sbb = __shfl_sync(0xffffffffu, k ? sb[1] : sb[0], o);
      const int l = idx - __shfl_sync(0xffffffffu, k ? base[1] : base[0], o);
      const int c = l / per_seq, rest = l % per_seq;
      const int g = rest / p.n_rb, rb = rest % p.n_rb;
      const int t0 = c * CH, t1 = min(ntb, t0 + CH);
      const int split = nchb > 1 ? sbb + (g * p.n_rb + rb) * nchb + c : -1;
      decode_item(b, Pb, g, rb, t0, t1, split);
    }
  }

  // Decode items come from the plan kernel's list, longest sequences first:
  // {b, g, rb, split slot} {first tile, end tile, prefix length, chunks}.
  __device__ void run_decode() {
    const int n_items = *reinterpret_cast<volatile int*>(&p.hdr->n_items);
    while (ok) {
      const int idx = grab();
      if (idx >= n_items) break;
      const int4 a = p.items[2 * idx], e = p.items[2 * idx + 1];
      decode_item(a.x, e.z, a.y, a.z, e.x, e.y, a.w);
    }
  }

  __device__ void decode_item(int b, int P, int g, int rb, int t0, int t1, int split) {
    const int D = p.Dblk;
    int qtok[2], qhead[2], ntok[2], qbase[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int tok = rb * 2 * p.tpm + m * p.tpm;
      ntok[m] = max(0, min(p.tpm, D - tok));
      qtok[m] = b * D + tok;
      qhead[m] = g * p.G;
      qbase[m] = P + tok;
    }
    const int n_m = ntok[1] > 0 ? 2 : 1;
    // mask block: the D tokens form one block, or one block each (causal)
    emit_item(t1 - t0, n_m, 0, qtok, qhead, ntok, qbase, P, p.causal ? 1 : D, split);
    const int n_pre = ceil_div(P, kTileKeys);
    // prefix tiles through the page table
    if (t0 < n_pre) emit_pool_tiles_contig(b, g, P, t0, min(t1, n_pre));
    // the block's own keys, dense
    for (int t = max(t0, n_pre); t < t1 && ok; ++t) {
      const int o = (t - n_pre) * kTileKeys;
      const int nvalid = min(kTileKeys, D - o);
      emit_dense_tile(g, b * D + o, nvalid, 0, P + o, !p.causal && nvalid == kTileKeys);
    }
  }

  // --------------------------------------------------------------------------
  // Prefill items: index space (query tile, sequence, KV head, head pair),
  // query tiles from the last (longest key range) down; empty ones skipped.
  __device__ void run_prefill() {
    const int per_qt = p.B * p.Hkv * p.n_hp;
    const int n_items = p.n_qt_max * per_qt;
    int bad = 0;
    while (ok) {
      const int idx = grab();
      if (idx >= n_items) break;
      const int qt = p.n_qt_max - 1 - idx / per_qt;
      const int rest = idx % per_qt;
      const int b = rest / (p.Hkv * p.n_hp);
      const int g = (rest / p.n_hp) % p.Hkv, hp = rest % p.n_hp;
      const int start = __ldg(p.lens + b), end = __ldg(p.lens + b + 1);
      int T = end - start;
      if (start < 0 || T < 0 || end > p.dense_tokens) {
        bad = 1;
        T = 0;
      }
      if (qt * kRowsPerMTile >= T) continue;
      prefill_item(start, T, qt, g, hp, p.Dblk);
    }
    if (bad && lane == 0) record_error(p, kErrBadLength);
  }

  __device__ void prefill_item(int start, int T, int qt, int g, int hp, int D) {
    const int q0 = qt * kRowsPerMTile;
    const int nq = min(kRowsPerMTile, T - q0);
    const int min_lim = min(row_limit(q0, 0, D), T);
    const int max_lim = min(row_limit(q0 + nq - 1, 0, D), T);
    const int n_tiles = ceil_div(max_lim, kTileKeys);
    int qtok[2], qhead[2], ntok[2], qbase[2];
    const int h0 = 2 * hp;
    for (int m = 0; m < 2; ++m) {
      qtok[m] = start + q0;
      qhead[m] = g * p.G + h0 + m;
      ntok[m] = (h0 + m < p.G) ? nq : 0;
      qbase[m] = q0;
    }
    const int n_m = ntok[1] > 0 ? 2 : 1;
    emit_item(n_tiles, n_m, 0, qtok, qhead, ntok, qbase, 0, D, -1);
    n_skip += (unsigned long long)(ceil_div(T, kTileKeys) - n_tiles);
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int k0 = t * kTileKeys;
      const int nvalid = min(kTileKeys, T - k0);
      const int full = (nvalid == kTileKeys) && (k0 + kTileKeys - 1 < min_lim);
      emit_dense_tile(g, start + k0, nvalid, 0, k0, full);
    }
  }

  // --------------------------------------------------------------------------
  __device__ int live_position(int b, int r) const {
    return p.live_pos ? __ldg(p.live_pos + (size_t)b * p.max_live + r) : p.prompt_len + r;
  }

  // Multicanvas items: index space (sequence, KV head, row block), row
  // blocks innermost, so that the items running at once share the keys of a
  // few (sequence, KV head) groups and their tiles are read from L2.
  __device__ void run_multicanvas() {
    const int rows_per_item = 2 * p.tpm;
    const int n_items = p.n_rb_max * p.B * p.Hkv;
    int bad = 0;
    while (ok) {
      const int idx = grab();
      if (idx >= n_items) break;
      const int rb = idx % p.n_rb_max;
      const int b = idx / (p.n_rb_max * p.Hkv), g = (idx / p.n_rb_max) % p.Hkv;
      int n_live = p.lens ? __ldg(p.lens + b) : p.max_live;
      int A = __ldg(p.arena_len + b);
      if (n_live < 0 || n_live > p.max_live || A < 0 ||
          (long long)A > (long long)p.max_pages * p.S) {
        bad = 1;
        continue;
      }
      if (rb * rows_per_item >= n_live) continue;
      multicanvas_item(b, n_live, A, g, rb);
    }
    if (bad && lane == 0) record_error(p, kErrBadLength);
  }

  // Class of arena tile a (entries [128a, 128a+128) of sequence b; 0 past
  // the last) from the plan kernel's {min, max} of its key positions.
  __device__ int arena_class(int b, int A, int a, int n_at, int min_lim, int max_lim, int min_lo,
                             int max_lo) const {
    if (a >= n_at) return 0;
    const int2 s = __ldcg(p.tile_kv + (size_t)b * p.n_at_max + a);
    return classify(s.x, s.y, min(kTileKeys, A - a * kTileKeys), min_lim, max_lim, min_lo,
                    max_lo);
  }

  // A tile of keys with positions in [kmin, kmax] against rows whose keys must
  // lie in [lo(q), lim(q)): skipped (0) when no row sees any of them, full (2)
  // when every row sees all of them and the tile holds 128 keys, else partial.
  __device__ static int classify(int kmin, int kmax, int nvalid, int min_lim, int max_lim,
                                 int min_lo, int max_lo) {
    if (kmin >= max_lim || kmax < min_lo) return 0;
    if (kmax < min_lim && kmin >= max_lo && nvalid == kTileKeys) return 2;
    return 1;
  }

  // Classes of live tiles l0 .. l0+3 (0 past the last), two bits each; the
  // positions of all four tiles are loaded before any is reduced.
  __device__ uint32_t live_classes4(int b, int n_live, int l0, int min_lim, int max_lim,
                                    int min_lo, int max_lo) {
    constexpr int kPer = kTileKeys / 32;
    int pos[4][kPer];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int h = 0; h < kPer; ++h) {
        const int r = (l0 + t) * kTileKeys + 32 * h + lane;
        pos[t][h] = r < n_live ? live_position(b, r) : INT_MAX;
      }
    uint32_t cls = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      int kmin = INT_MAX, kmax = INT_MIN;
#pragma unroll
      for (int h = 0; h < kPer; ++h) {
        const int r = (l0 + t) * kTileKeys + 32 * h + lane;
        kmin = min(kmin, pos[t][h]);
        kmax = r < n_live ? max(kmax, pos[t][h]) : kmax;
      }
      kmin = warp_min(kmin);
      kmax = warp_max(kmax);
      const int nvalid = n_live - (l0 + t) * kTileKeys;
      if (nvalid > 0)
        cls |= (uint32_t)classify(kmin, kmax, min(kTileKeys, nvalid), min_lim, max_lim, min_lo,
                                  max_lo) << (2 * t);
    }
    return cls;
  }

  __device__ void multicanvas_item(int b, int n_live, int A, int g, int rb) {
    const int r0 = rb * 2 * p.tpm;
    const int nrows = min(2 * p.tpm, n_live - r0);
    int lo = INT_MAX, hi = INT_MIN, qlo = INT_MAX, qhi = INT_MIN;
    for (int r = lane; r < nrows; r += 32) {
      const int q = live_position(b, r0 + r);
      const int lim = row_limit(q, p.prompt_len, p.Dblk);
      lo = min(lo, lim);
      hi = max(hi, lim);
      qlo = min(qlo, q);
      qhi = max(qhi, q);
    }
    const int min_lim = warp_min(lo), max_lim = warp_max(hi);
    // sliding-window band: the keys of row q start at q - window + 1
    const int min_lo = p.window > 0 ? warp_min(qlo) - p.window + 1 : INT_MIN;
    const int max_lo = p.window > 0 ? warp_max(qhi) - p.window + 1 : INT_MIN;
    const int n_at = ceil_div(A, kTileKeys), n_lt = ceil_div(n_live, kTileKeys);
    // pass 1: count the tiles that are not fully excluded (arena tiles 32 at a
    // time, one summary per lane; live tiles 4 at a time)
    int n_tiles = 0;
    for (int a0 = 0; a0 < n_at; a0 += 32)
      n_tiles += __popc(__ballot_sync(
          0xffffffffu, arena_class(b, A, a0 + lane, n_at, min_lim, max_lim, min_lo, max_lo) != 0));
    for (int l0 = 0; l0 < n_lt; l0 += 4) {
      const uint32_t c4 = live_classes4(b, n_live, l0, min_lim, max_lim, min_lo, max_lo);
      n_tiles += __popc((c4 | (c4 >> 1)) & 0x55u);
    }
    int qtok[2], qhead[2], ntok[2], qbase[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int r = r0 + m * p.tpm;
      ntok[m] = max(0, min(p.tpm, n_live - r));
      qtok[m] = b * p.max_live + r;
      qhead[m] = g * p.G;
      qbase[m] = p.live_pos ? b * p.max_live + r : p.prompt_len + r;
    }
    const int n_m = ntok[1] > 0 ? 2 : 1;
    emit_item(n_tiles, n_m, p.live_pos ? 1 : 0, qtok, qhead, ntok, qbase, p.prompt_len, p.Dblk,
              -1);
    n_skip += (unsigned long long)(n_at + n_lt - n_tiles);
    // pass 2: emit.  Arena tiles: the chunk pages of the next four kept tiles
    // are fetched at once (lane 8j + i: chunk i of the j-th).
    constexpr int kTilesPerGroup = 32 / kChunksPerTile;
    for (int a0 = 0; a0 < n_at && ok; a0 += 32) {
      const int cls = arena_class(b, A, a0 + lane, n_at, min_lim, max_lim, min_lo, max_lo);
      uint32_t keep = __ballot_sync(0xffffffffu, cls != 0);
      const uint32_t full = __ballot_sync(0xffffffffu, cls == 2);
      while (keep != 0 && ok) {
        uint32_t mine = keep;
        for (int k = 0; k < lane / kChunksPerTile; ++k) mine &= mine - 1;
        int coord = p.pool_rows, koff = 0;  // out of range -> zero fill
        if (mine != 0) {
          const int e = (a0 + __ffs(mine) - 1) * kTileKeys + (lane % kChunksPerTile) * kChunkKeys;
          if (e < A) {
            const int page = page_of(b, e);
            if (page >= 0) {
              coord = (page * p.Hkv + g) * p.S + (e % p.S);
              koff = page * p.S + (e % p.S);
            }
          }
        }
        const int ntile = min(kTilesPerGroup, __popc(keep));
        for (int j = 0; j < ntile && ok; ++j) {
          const int a = a0 + __ffs(keep) - 1;
          keep &= keep - 1;
          int cd[kChunksPerTile], ko[kChunksPerTile];
#pragma unroll
          for (int i = 0; i < kChunksPerTile; ++i) {
            cd[i] = __shfl_sync(0xffffffffu, coord, kChunksPerTile * j + i);
            ko[i] = __shfl_sync(0xffffffffu, koff, kChunksPerTile * j + i);
          }
          emit_tile(0, (full >> (a - a0)) & 1, min(kTileKeys, A - a * kTileKeys), g, 1, 0, cd, ko);
        }
      }
    }
    const int kmode = p.live_pos ? 2 : 0;
    for (int l0 = 0; l0 < n_lt && ok; l0 += 4) {
      const uint32_t c4 = live_classes4(b, n_live, l0, min_lim, max_lim, min_lo, max_lo);
      for (int t = 0; t < 4 && ok; ++t) {
        const int cls = (c4 >> (2 * t)) & 3, l = l0 + t;
        if (cls == 0) continue;
        const int nvalid = min(kTileKeys, n_live - l * kTileKeys);
        const int kbase = p.live_pos ? b * p.max_live + l * kTileKeys : p.prompt_len + l * kTileKeys;
        emit_dense_tile(g, b * p.max_live + l * kTileKeys, nvalid, kmode, kbase, cls == 2);
      }
    }
  }

  __device__ void run() {
    if (p.mode == kModeDecode) {
      if (p.fused_plan) run_decode_fused();
      else run_decode();
    }
    else if (p.mode == kModePrefill) run_prefill();
    else run_multicanvas();
    if (ok) emit_end();
    if (__any_sync(0xffffffffu, page_err) && lane == 0) record_error(p, kErrPageOob);
    if (lane == 0 && lead()) {
      if (n_full) atomicAdd(&p.hdr->tiles_full, n_full);
      if (n_partial) atomicAdd(&p.hdr->tiles_partial, n_partial);
      if (n_skip) atomicAdd(&p.hdr->tiles_skipped, n_skip);
    }
  }
};

// Consumer side of the record ring (whole-warp roles).
template <class Ctx>
__device__ __forceinline__ const Rec* ring_get(const Ctx& c, const AttnParams& p, uint32_t i) {
  if (!wait_bar_warp(c, p, &c.bar.rec_full[i % kNumRec], (i / kNumRec) & 1)) return nullptr;
  return &c.ring[i % kNumRec];
}
template <class Ctx>
__device__ __forceinline__ void ring_release(const Ctx& c, uint32_t i, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&c.bar.rec_empty[i % kNumRec]);
}

}  // namespace attn
}  // namespace bca
