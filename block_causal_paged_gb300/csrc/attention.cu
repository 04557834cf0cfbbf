// Block-causal attention over a paged KV cache, sm_103a (tcgen05 + TMA).
//
// One persistent CTA per SM takes work items from a shared counter (a small
// plan kernel orders them longest first and resets the counter).  An item is a
// block of up to 256 query rows (two M-tiles of 128 rows) that share one KV
// head, plus the sequence of 128-key tiles those rows attend.  Rows are
// (token, head) pairs: for decode and multicanvas the G query heads of one KV
// head are packed into the rows (rows = tokens x G, so K/V is read once per
// group); for prefill each M-tile is one head over 128 tokens.
//
// The visibility rule ("Inference for Interpretable Text-Diffusion Models",
// "Background"; "Inference: Fewer, smaller forwards", "Advancement 13") is
// evaluated per row as a key-position limit: a query at position q sees key
// position k iff k < lim(q), lim(q) = P0 if q < P0 else P0 + D*(floor((q-P0)/D)+1).
// Each KV tile is classified against the item's rows ("FlexAttention with
// Aligned Tiles"): fully included (no mask arithmetic), partially included
// (elementwise k < lim(q)) or fully excluded (not emitted: no load, no math).
//
// Warp roles (384 threads):
//   warp 3      planner  : enumerates items/tiles, reads page tables and
//                          positions, classifies tiles, writes records into a
//                          small shared-memory ring
//   warp 0      loader   : TMA loads of Q and of K/V page boxes into a ring of
//                          shared-memory stages (ragged 16-key chunks are
//                          copied by the warp's lanes with zero fill)
//   warp 1      MMA      : the whole warp runs the issue loop and one elected
//                          lane issues each tcgen05.mma.  Per M-tile m and
//                          tile j: O_m += P_m V_j with P_m read from TMEM, then
//                          S_m = Q_m K_{j+1}^T into the same TMEM columns; the
//                          two M-tiles alternate, so the tensor core works on
//                          one while the softmax warps work on the other
//   warp 2      TMEM allocation / release
//   warps 4-7   softmax for M-tile 0, warps 8-11 for M-tile 1: read S rows
//               from TMEM, mask, online softmax (lazy rescale of O), write P
//               (bf16) back into the S columns, final normalisation and store.
// Every wait is bounded; on timeout the CTA records BCA_ERR_DEVICE_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include <atomic>
#include <climits>
#include <cstdint>

#include "attn_common.cuh"
#include "bca_internal.h"
#include "ptx_sm103.cuh"

namespace bca {
namespace {
using namespace attn;

constexpr int kRegsLaunch = 168;   // 65536 / 384, rounded down to a multiple of 8
constexpr int kRegsControl = 112;
constexpr int kRegsSoftmax = 184;
static_assert(kRegsControl * 128 + kRegsSoftmax * 256 <= kRegsLaunch * kThreads, "register split");
constexpr int kRecConsumers = 10;  // loader + MMA + 8 softmax warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
template <int HD>
struct Cfg {
  static constexpr int kHalves = HD / 64;                 // 128-byte column blocks of a row
  static constexpr int kQBytes = kHalves * 16384;         // 128 rows of Q
  static constexpr int kHalfBytes = kTileKeys * 128;      // one 64-column half of a KV tile
  static constexpr int kSlotBytes = kHalves * kHalfBytes; // 128 keys of K or V
  static constexpr int kStages = HD == 128 ? 5 : 12;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + 2 * kQBytes;
  static constexpr int kOffRec = kOffKV + kStages * kSlotBytes;
  static constexpr int kNumBars = 2 * kNumRec + 2 * kStages + 12 + 1;
  static constexpr int kOffBar = kOffRec + kNumRec * (int)sizeof(Rec);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  static constexpr int kSmemAlloc = kBytes + 1024;  // base is aligned up to 1024 in the kernel
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S of M-tile m at 128*m (fp32, one column per key); P of
  // M-tile m overwrites the first 64 of them (bf16 pairs); O at 256 + HD*m.
  static constexpr int kColS = 0;
  static constexpr int kColO = 256;
  static_assert(kColO + 2 * HD <= (int)kTmemCols, "TMEM plan");
  static_assert(kSmemAlloc <= 232448, "shared memory plan");
};

struct Bars {
  uint64_t* rec_full;
  uint64_t* rec_empty;
  uint64_t* kv_full;
  uint64_t* kv_empty;
  uint64_t* q_full;    // [2]
  uint64_t* q_empty;   // [2]
  uint64_t* s_full;    // [2]
  uint64_t* p_full;    // [2]
  uint64_t* o_full;    // [2]
  uint64_t* o_empty;   // [2]
  uint64_t* drain;
};

struct Ctx {
  uint8_t* smem;
  Rec* ring;
  Bars bar;
  volatile int* abort_flag;
  uint32_t tmem;
};

// ============================================================================
// loader (warp 0)
// ============================================================================
template <int HD>
__device__ __forceinline__ void run_loader(const Ctx& c, const AttnParams& p, const CUtensorMap* tm_q,
                           const CUtensorMap* tm_kp, const CUtensorMap* tm_vp,
                           const CUtensorMap* tm_kd, const CUtensorMap* tm_vd, int lane) {
  using C = Cfg<HD>;
  const uint32_t q_base = smem_u32(c.smem + C::kOffQ);
  const uint32_t kv_base = smem_u32(c.smem + C::kOffKV);
  // phase bits (bit m): Q loads issued per M-tile (parity) and whether any
  uint32_t ri = 0, u = 0, q_par = 0, q_used = 0;
  bool ok = true;
  const bool box_lane = (lane & 15) < kChunksPerTile * C::kHalves;
  const int my_chunk = box_lane ? (lane & 15) / C::kHalves : 0;
  const int my_half = (lane & 15) % C::kHalves;
  const int my_kv = lane >> 4;  // lanes 0-15 copy K boxes, lanes 16-31 V boxes
  while (ok) {
    const Rec* r = ring_get(c, p, ri);
    if (!r) break;
    const int kind = r->w[0];
    if (kind == kRecEnd) {
      ring_release(c, ri, lane);
      break;
    }
    if (kind == kRecItem) {
      const int n_m = r->w[I_NM];
      const int qh0 = r->w[I_QHEAD], qh1 = r->w[I_QHEAD + 1];
      const int qt0 = r->w[I_QTOK], qt1 = r->w[I_QTOK + 1];
      ring_release(c, ri, lane);
      ++ri;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (m >= n_m) break;
        if (!wait_bar_warp(c, p, &c.bar.q_empty[m], ((q_par >> m) & 1) ^ 1)) { ok = false; break; }
        if (lane == 0) {
          // the Q box holds hpr x tpm rows (126 for G = 3), 128 bytes per row per half
          mbar_arrive_expect_tx(&c.bar.q_full[m], (uint32_t)(C::kHalves * p.hpr * p.tpm * 128));
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_3d(q_base + m * C::kQBytes + h * 16384, tm_q, &c.bar.q_full[m], h * 64,
                        m ? qh1 : qh0, m ? qt1 : qt0);
        }
        __syncwarp();
        q_par ^= 1u << m;
        q_used |= 1u << m;
      }
      continue;
    }
    // fields of a tile record: each box lane reads only its own chunk's coordinate
    const int src = r->w[T_SRC], nvalid = r->w[T_NVALID], head = r->w[T_HEAD];
    const int my_coord = r->w[T_COORD + my_chunk];
    const int ragged = (nvalid % kChunkKeys) != 0 ? nvalid / kChunkKeys : -1;
    const int ragged_coord = ragged >= 0 ? r->w[T_COORD + ragged] : 0;
    ring_release(c, ri, lane);
    ++ri;
    // a KV tile: K into the next stage, V into the one after.  Both stages are
    // acquired first; then one warp instruction issues every box of the tile:
    // lanes 0-15 the K boxes, lanes 16-31 the V boxes (lane l % 16 < 8 * halves
    // copies chunk (l % 16) / halves, half (l % 16) % halves).
    const int my_nv = min(max(nvalid - my_chunk * kChunkKeys, 0), kChunkKeys);
    const bool my_tma = box_lane && (my_nv == 0 || my_nv == kChunkKeys);
    const bool manual = ragged >= 0;
    const uint32_t tma_bytes = (uint32_t)(kChunksPerTile - (manual ? 1 : 0)) * C::kHalves * 2048;
    uint32_t slot[2];
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      slot[kv] = (u + kv) % C::kStages;
      if (ok && !wait_bar_warp(c, p, &c.bar.kv_empty[slot[kv]], (((u + kv) / C::kStages) & 1) ^ 1))
        ok = false;
    }
    if (!ok) break;
    if (manual) {
      // ragged chunk: copy the valid rows with the warp, zero the rest
      const int nv = nvalid - ragged * kChunkKeys;
      const int coord = ragged_coord;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const uint32_t dst = kv_base + slot[kv] * C::kSlotBytes;
        const uint16_t* base = src == 0 ? (kv ? p.v_pool : p.k_pool) : (kv ? p.v_dense : p.k_dense);
        for (int piece = lane; piece < kChunkKeys * C::kHalves * 8; piece += 32) {
          const int rr = piece / (C::kHalves * 8);
          const int h = (piece / 8) % C::kHalves;
          const int cc = piece % 8;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (rr < nv) {
            const size_t row = src == 0 ? (size_t)(coord + rr)
                                        : (size_t)(coord + rr) * p.Hkv + head;
            v = __ldg(reinterpret_cast<const uint4*>(base + row * HD + h * 64 + cc * 8));
          }
          const int krow = ragged * kChunkKeys + rr;
          st_shared_v4(dst + h * C::kHalfBytes + krow * 128 + ((cc ^ (krow & 7)) << 4), v.x, v.y,
                       v.z, v.w);
        }
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(&c.bar.kv_full[slot[0]], tma_bytes);
      mbar_arrive_expect_tx(&c.bar.kv_full[slot[1]], tma_bytes);
    }
    __syncwarp();
    if (my_tma) {
      // the planner made the coordinate out of range for a chunk with no key
      const CUtensorMap* map = src == 0 ? (my_kv ? tm_vp : tm_kp) : (my_kv ? tm_vd : tm_kd);
      const uint32_t sl = my_kv ? slot[1] : slot[0];
      const uint32_t d = kv_base + sl * C::kSlotBytes + my_half * C::kHalfBytes + my_chunk * 2048;
      if (src == 0) tma_load_2d(d, map, &c.bar.kv_full[sl], my_half * 64, my_coord);
      else tma_load_3d(d, map, &c.bar.kv_full[sl], my_half * 64, head, my_coord);
    }
    __syncwarp();
    u += 2;
  }
  // teardown: never leave this CTA with copies in flight
  for (uint32_t k = 0; k < (uint32_t)C::kStages && k < u; ++k) {
    const uint32_t uu = u - 1 - k;
    mbar_wait(&c.bar.kv_full[uu % C::kStages], (uu / C::kStages) & 1, c.abort_flag, kWaitTimeoutCycles);
  }
#pragma unroll
  for (int m = 0; m < 2; ++m)
    if ((q_used >> m) & 1)
      mbar_wait(&c.bar.q_full[m], ((q_par >> m) & 1) ^ 1, c.abort_flag, kWaitTimeoutCycles);
}

// ============================================================================
// MMA issuer (warp 1, one thread)
// ============================================================================
// S_m = Q_m K^T: M = 128 query rows, N = 128 keys, K = head_dim (16 per
// instruction), both operands K-major in 128-byte-swizzled shared memory.
template <int HD>
__device__ __forceinline__ void issue_qk(const Ctx& c, int m, uint32_t slot) {
  using C = Cfg<HD>;
  constexpr uint32_t idesc = make_idesc_bf16(128, kTileKeys, 0, 0);
  const uint32_t qa = smem_u32(c.smem + C::kOffQ + m * C::kQBytes);
  const uint32_t ka = smem_u32(c.smem + C::kOffKV + slot * C::kSlotBytes);
  const uint32_t d = c.tmem + C::kColS + m * kTileKeys;
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    const int h = ks >> 2, kin = ks & 3;
    const uint64_t a = make_sdesc_sw128(qa + h * 16384 + kin * 32, 16, 1024);
    const uint64_t b = make_sdesc_sw128(ka + h * C::kHalfBytes + kin * 32, 16, 1024);
    umma_bf16(d, a, b, idesc, ks > 0 ? 1u : 0u);
  }
}

// O_m (+)= P_m V: M = 128 rows, N = head_dim, K = 128 keys (16 per
// instruction); P_m from TMEM (the S columns, 8 columns per 16 keys), V
// MN-major in shared memory (LBO = the next 64 head-dim columns).
template <int HD>
__device__ __forceinline__ void issue_pv(const Ctx& c, int m, uint32_t slot, bool acc) {
  using C = Cfg<HD>;
  constexpr uint32_t idesc = make_idesc_bf16(128, HD, 0, 1);
  const uint32_t pa = c.tmem + C::kColS + m * kTileKeys;
  const uint32_t va = smem_u32(c.smem + C::kOffKV + slot * C::kSlotBytes);
  const uint32_t d = c.tmem + C::kColO + m * HD;
#pragma unroll
  for (int ks = 0; ks < kTileKeys / 16; ++ks) {
    const uint64_t b = make_sdesc_sw128(va + ks * 2048, C::kHalfBytes, 1024);
    umma_bf16_ts(d, pa + ks * 8, b, idesc, (acc || ks > 0) ? 1u : 0u);
  }
}

// Issue order for an item of n tiles (K(t), V(t) are loads 2t, 2t+1 of the
// item): S_0(0) S_1(0) | PV_0(0) S_0(1) PV_1(0) S_1(1) | PV_0(1) S_0(2) ...
// S_m(t+1) overwrites the TMEM columns holding P_m(t); it is issued after the
// PV that reads them, and tcgen05.mma operations from one thread execute in
// issue order.  Its commit therefore also tells the softmax warps that O_m
// holds every PV before it (needed before they rescale O_m).
template <int HD>
__device__ __forceinline__ void run_mma(const Ctx& c, const AttnParams& p, int lane) {
  using C = Cfg<HD>;
  // phase parities as bits (bit m for M-tile m), so no counter needs memory
  uint32_t ri = 0, u = 0, q_par = 0, p_par = 0, o_par = 0;
  bool ok = true;
  while (ok) {
    const Rec* r = ring_get(c, p, ri);
    if (!r) break;
    const int kind = r->w[I_KIND], n_t = r->w[I_NT], n_m = r->w[I_NM];
    ring_release(c, ri, lane);
    ++ri;
    if (kind == kRecEnd) break;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      if (m < n_m && ok) {
        ok = wait_bar_warp(c, p, &c.bar.q_full[m], (q_par >> m) & 1);
        q_par ^= 1u << m;
      }
    }
    if (!ok) break;
    const uint32_t ub = u;
    u += 2u * (uint32_t)n_t;
    ri += (uint32_t)n_t;  // the item's tile records are released by the planner for this warp
    // tile 0: S for every active M-tile
    uint32_t ks = ub % C::kStages;
    if (!wait_bar_warp(c, p, &c.bar.kv_full[ks], (ub / C::kStages) & 1)) break;
    tc_fence_after();
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      if (m >= n_m) break;
      issue_qk<HD>(c, m, ks);
      umma_commit(&c.bar.s_full[m]);
      if (n_t == 1) umma_commit(&c.bar.q_empty[m]);
    }
    umma_commit(&c.bar.kv_empty[ks]);
    for (int j = 0; j < n_t && ok; ++j) {
      const uint32_t uv = ub + 2u * (uint32_t)j + 1u;
      const uint32_t vs = uv % C::kStages;
      const bool nxt = j + 1 < n_t;
      // V(j) and K(j+1) are checked together, before the wait for P: their
      // loads were issued tiles ago, and a satisfied wait still costs ~150
      // cycles that are better spent while P is being computed
      if (!(ok = wait_bar_warp(c, p, &c.bar.kv_full[vs], (uv / C::kStages) & 1))) break;
      if (nxt) {
        ks = (uv + 1u) % C::kStages;
        if (!(ok = wait_bar_warp(c, p, &c.bar.kv_full[ks], ((uv + 1u) / C::kStages) & 1))) break;
      }
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (m >= n_m || !ok) break;
        if (!(ok = wait_bar_warp(c, p, &c.bar.p_full[m], (p_par >> m) & 1))) break;
        p_par ^= 1u << m;
        if (j == 0 && !(ok = wait_bar_warp(c, p, &c.bar.o_empty[m], ((o_par >> m) & 1) ^ 1))) break;
        tc_fence_after();
        issue_pv<HD>(c, m, vs, j > 0);
        if (nxt) {
          issue_qk<HD>(c, m, ks);
          umma_commit(&c.bar.s_full[m]);
          if (j + 2 == n_t) umma_commit(&c.bar.q_empty[m]);  // last read of Q
        } else {
          umma_commit(&c.bar.o_full[m]);
          o_par ^= 1u << m;
        }
      }
      if (!ok) break;
      umma_commit(&c.bar.kv_empty[vs]);
      if (nxt) umma_commit(&c.bar.kv_empty[ks]);
    }
  }
  // teardown: wait until every MMA issued by this warp has completed
  umma_commit(c.bar.drain);
  mbar_wait(c.bar.drain, 0, c.abort_flag, kWaitTimeoutCycles);
}

// ============================================================================
// softmax / epilogue (warps 4..11)
// ============================================================================
// kBand: the multicanvas sliding-window band (a per-row lower key bound);
// a separate instantiation, so that the other modes keep their registers.
template <int HD, bool kBand>
__device__ __forceinline__ void run_softmax(const Ctx& c, const AttnParams& p, int m, int wq,
                                            int lane) {
  using C = Cfg<HD>;
  const int r = 32 * wq + lane;  // row within the M-tile == TMEM lane
  const uint32_t lane_addr = static_cast<uint32_t>(32 * wq) << 16;
  const uint32_t t_s = c.tmem + lane_addr + C::kColS + m * kTileKeys;  // S, then P
  const uint32_t t_o = c.tmem + lane_addr + C::kColO + m * HD;
  const float sl2 = p.scale_log2;
  uint32_t ri = 0, s_par = 0, o_par = 0;
  while (true) {
    const Rec* rec = ring_get(c, p, ri);
    if (!rec) return;
    const int kind = rec->w[I_KIND];
    const int n_t = rec->w[I_NT], n_m = rec->w[I_NM], qmode = rec->w[I_QMODE];
    const int qtok = rec->w[I_QTOK + m], qhead = rec->w[I_QHEAD + m];
    const int ntok = rec->w[I_NTOK + m], qbase = rec->w[I_QBASE + m];
    const int P0 = rec->w[I_P0], Dblk = rec->w[I_DBLK], split = rec->w[I_SPLIT];
    ring_release(c, ri, lane);
    ++ri;
    if (kind == kRecEnd) return;
    const bool active = m < n_m;
    const int tok = r / p.hpr;
    const bool valid = active && r < p.hpr * p.tpm && tok < ntok;
    int lim = INT_MAX, lo = INT_MIN;  // row q sees key positions in [lo, lim)
    if (valid) {
      const int qpos = qmode == 0 ? qbase + tok : __ldg(p.live_pos + qbase + tok);
      lim = row_limit(qpos, P0, Dblk);
      if (kBand) lo = qpos - p.window + 1;
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < n_t; ++j) {
      const Rec* t = ring_get(c, p, ri);
      if (!t) return;
      const int full = t->w[T_FULL], nvalid = t->w[T_NVALID], kmode = t->w[T_KMODE];
      const int kbase = t->w[T_KBASE];
      // Partial tile: lane l fetches the positions of keys 4l .. 4l+3 now, so
      // that the load is in flight while S is computed.  Keys are consecutive
      // from kbase (kmode 0), 16 consecutive kv_pos entries per chunk from
      // the chunk's offset (arena slots, kmode 1) or consecutive live_pos
      // entries (kmode 2); keys at or past nvalid get INT_MAX (never seen).
      int kp[4] = {INT_MAX, INT_MAX, INT_MAX, INT_MAX};
      if (!full && active) {
        const int k4 = 4 * lane;
        if (kmode == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) kp[i] = k4 + i < nvalid ? kbase + k4 + i : INT_MAX;
        } else if (k4 < nvalid) {
          const int32_t* src = kmode == 1
                                   ? p.kv_pos + t->w[T_KOFF + k4 / kChunkKeys] + k4 % kChunkKeys
                                   : p.live_pos + kbase + k4;
          if (k4 + 4 <= nvalid && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
            const int4 v4 = __ldg(reinterpret_cast<const int4*>(src));
            kp[0] = v4.x;
            kp[1] = v4.y;
            kp[2] = v4.z;
            kp[3] = v4.w;
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) kp[i] = k4 + i < nvalid ? __ldg(src + i) : INT_MAX;
          }
        }
      }
      ring_release(c, ri, lane);
      ++ri;
      if (!active) continue;
      if (!wait_bar_warp(c, p, &c.bar.s_full[m], s_par & 1)) return;
      s_par ^= 1u;
      tc_fence_after();
      // Partial tile: visibility of key k for this row is bit k/4 of vis[k%4].
      // Rows with the same key range [lo, lim) share one mask: per distinct
      // range in the warp, four ballots over the lanes' keys build it (rows of
      // one canvas share lim; only the band's lo differs per token).  Built
      // before S is read into registers, while they are free.
      uint32_t vis[4] = {0u, 0u, 0u, 0u};
      if (!full) {
        bool done = !valid;  // rows past the item's tokens see nothing
        while (true) {
          const uint32_t pend = __ballot_sync(0xffffffffu, !done);
          if (pend == 0u) break;
          const int leader = __ffs(pend) - 1;
          const int L = __shfl_sync(0xffffffffu, lim, leader);
          const int Lo = kBand ? __shfl_sync(0xffffffffu, lo, leader) : INT_MIN;
          uint32_t bl[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            bl[i] = __ballot_sync(0xffffffffu, kBand ? (kp[i] < L && kp[i] >= Lo) : kp[i] < L);
          if (!done && lim == L && (!kBand || lo == Lo)) {
#pragma unroll
            for (int i = 0; i < 4; ++i) vis[i] = bl[i];
            done = true;
          }
        }
      }
      uint32_t sv[kTileKeys];
      tmem_ld128_sync(t_s, sv);
      if (!full) {
#pragma unroll
        for (int k = 0; k < kTileKeys; ++k)
          if (!((vis[k & 3] >> (k >> 2)) & 1u)) sv[k] = __float_as_uint(-INFINITY);
      }
      // row maximum of the raw scores (the scale is positive), in log2 units:
      // four chains of three-input maxima
      float mx[4] = {__uint_as_float(sv[0]), __uint_as_float(sv[1]), __uint_as_float(sv[2]),
                     __uint_as_float(sv[3])};
#pragma unroll
      for (int k = 4; k < kTileKeys; k += 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mx[i] = fmax3(mx[i], __uint_as_float(sv[k + 2 * i]), __uint_as_float(sv[k + 2 * i + 1]));
      }
      const float mt = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
      const float m_new = fmaxf(m_run, mt);
      bool rescale = false;
      float alpha = 1.0f;
      if (j == 0) {
        m_run = m_new;
      } else if (m_new > m_run + kRescaleThreshold) {
        // lazy rescaling: only when the running maximum grows by more than 2^8
        rescale = true;
        alpha = ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O_m holds all earlier PV products (the S commit came after them)
#pragma unroll 1
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32_sync(t_o + c0, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(t_o + c0, o);
        }
      }
      const float ref = m_run == -INFINITY ? 0.f : m_run;
      // p = 2^(s * scale * log2(e) - ref), two keys per paired FMA / add
      const float2 scale2 = make_float2(sl2, sl2), nref2 = make_float2(-ref, -ref);
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int cq = 0; cq < kTileKeys / 32; ++cq) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 x = ffma2(make_float2(__uint_as_float(sv[32 * cq + 2 * k]),
                                             __uint_as_float(sv[32 * cq + 2 * k + 1])),
                                 scale2, nref2);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          sum2 = fadd2(sum2, pp);
          w[k] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st16(t_s + 16 * cq, w);  // P over the first 64 S columns
      }
      l_run = l_run * alpha + (sum2.x + sum2.y);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.bar.p_full[m]);
    }
    if (!active) continue;
    if (!wait_bar_warp(c, p, &c.bar.o_full[m], o_par & 1)) return;
    o_par ^= 1u;
    tc_fence_after();
    if (split < 0) {
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
      uint16_t* dst = p.out + ((size_t)(qtok + tok) * p.Hq + qhead + (r % p.hpr)) * HD;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t o[32];
        tmem_ld32_sync(t_o + c0, o);
        if (valid) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c0 + 8 * k) = v;
          }
        }
      }
    } else {
      const int R = m * kRowsPerMTile + r;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t o[32];
        tmem_ld32_sync(t_o + c0, o);
        if (valid) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float4 v = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                   __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
            const size_t idx = (((size_t)split * (HD / 4) + (c0 / 4 + k)) * 256 + R) * 4;
            *reinterpret_cast<float4*>(p.part_o + idx) = v;
          }
        }
      }
      if (valid) {
        *reinterpret_cast<float2*>(p.part_ml + ((size_t)split * 256 + R) * 2) =
            make_float2(m_run, l_run);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.bar.o_empty[m]);
  }
}

// ============================================================================
// the kernel
// ============================================================================
template <int HD, bool kBand>
__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_kp,
                     const __grid_constant__ CUtensorMap tm_vp,
                     const __grid_constant__ CUtensorMap tm_kd,
                     const __grid_constant__ CUtensorMap tm_vd,
                     const __grid_constant__ AttnParams p) {
  using C = Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Ctx c;
  c.smem = smem;
  c.ring = reinterpret_cast<Rec*>(smem + C::kOffRec);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  c.bar.rec_full = bars;
  c.bar.rec_empty = bars + kNumRec;
  c.bar.kv_full = bars + 2 * kNumRec;
  c.bar.kv_empty = c.bar.kv_full + C::kStages;
  c.bar.q_full = c.bar.kv_empty + C::kStages;
  c.bar.q_empty = c.bar.q_full + 2;
  c.bar.s_full = c.bar.q_empty + 2;
  c.bar.p_full = c.bar.s_full + 2;
  c.bar.o_full = c.bar.p_full + 2;
  c.bar.o_empty = c.bar.o_full + 2;
  c.bar.drain = c.bar.o_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  c.abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumRec; ++i) {
      mbar_init(&c.bar.rec_full[i], 1);
      mbar_init(&c.bar.rec_empty[i], kRecConsumers);
    }
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&c.bar.kv_full[i], 1);
      mbar_init(&c.bar.kv_empty[i], 1);
    }
    for (int m = 0; m < 2; ++m) {
      mbar_init(&c.bar.q_full[m], 1);
      mbar_init(&c.bar.q_empty[m], 1);
      mbar_init(&c.bar.s_full[m], 1);
      mbar_init(&c.bar.p_full[m], 4);
      mbar_init(&c.bar.o_full[m], 1);
      mbar_init(&c.bar.o_empty[m], 4);
    }
    mbar_init(c.bar.drain, 1);
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kp);
    tma_prefetch_desc(&tm_vp);
    tma_prefetch_desc(&tm_kd);
    tma_prefetch_desc(&tm_vd);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *tmem_slot;
  // Programmatic dependent launch: the prologue above overlapped the plan
  // kernel; nothing it wrote is read before this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Register split: the control warpgroup (warps 0-3) gives registers to the
  // two softmax warpgroups for the duration of the roles (each region is
  // entered and left with its own setmaxnreg), then both return to the launch
  // allocation for the common teardown.  The host checks the kernel was
  // compiled with kRegsLaunch registers per thread before launching it.
  // Deadlock freedom: the softmax increase waits only for the control
  // decrease (which never blocks); the barrier after the exchange keeps any
  // control warp from restoring before it; at the end the control increase is
  // served by the softmax decrease, which never waits on a control warp.
  if (warp < 4) {
    regs_dealloc<kRegsControl>();
    // No warp may start (and then finish and take registers back) before the
    // softmax warpgroups' increase has been served from the released pool.
    named_barrier_sync(1, kThreads);
    if (warp == 3) {
      Planner<Ctx, false> pl(p, c, lane);
      pl.run();
    } else if (warp == 0) {
      run_loader<HD>(c, p, &tm_q, &tm_kp, &tm_vp, &tm_kd, &tm_vd, lane);
    } else if (warp == 1) {
      run_mma<HD>(c, p, lane);
    }
    __syncwarp();
    regs_alloc<kRegsLaunch>();
  } else {
    regs_alloc<kRegsSoftmax>();
    named_barrier_sync(1, kThreads);
    run_softmax<HD, kBand>(c, p, (warp - 4) >> 2, warp & 3, lane);
    __syncwarp();
    regs_dealloc<kRegsLaunch>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(c.tmem, C::kTmemCols);
  }
  // The last CTA to leave resets the work counter for the next launch (every
  // CTA has finished taking items by now).
  if (threadIdx.x == 0) {
    __threadfence();
    const int done = atomicAdd(&p.hdr->exit_count, 1);
    if (done == (int)gridDim.x - 1) {
      p.hdr->work_next = 0;
      p.hdr->exit_count = 0;
      __threadfence();
    }
  }
}

template <int HD, bool kBand>
cudaError_t launch_attention_hd(const AttnParams& p, const AttnMaps& maps, int grid,
                                cudaStream_t stream) {
  using C = Cfg<HD>;
  // The shared-memory attribute is a property of the kernel on one device:
  // set it once per device (several host threads may get here at once; a
  // repeated set is harmless).
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (!cached || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attention_kernel<HD, kBand>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits for registers released by setmaxnreg.dec; the
    // split must fit what the block is launched with, or the kernel would stall
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attention_kernel<HD, kBand>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
    if (cached) configured[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attention_kernel<HD, kBand>, maps.q, maps.kp, maps.vp, maps.kd,
                            maps.vd, p);
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, const AttnMaps& maps, int head_dim, int grid,
                             cudaStream_t stream) {
  const bool band = p.mode == kModeMulticanvas && p.window > 0;
  if (head_dim == 128)
    return band ? launch_attention_hd<128, true>(p, maps, grid, stream)
                : launch_attention_hd<128, false>(p, maps, grid, stream);
  return band ? launch_attention_hd<64, true>(p, maps, grid, stream)
              : launch_attention_hd<64, false>(p, maps, grid, stream);
}

}  // namespace bca
