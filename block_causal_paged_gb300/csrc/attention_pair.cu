// Block-causal attention on CTA pairs, sm_103a (tcgen05 cta_group::2 + TMA):
// the decode step and short extend when their query rows fill two M-tiles,
// the prefill and the multicanvas step (with or without the sliding-window
// band), head_dim 128.
//
// A cluster of two CTAs on neighbouring SMs works on one item at a time.  An
// item is up to 256 query rows sharing one KV head -- two M-tiles of 128 rows,
// M-tile r held by CTA r of the pair -- plus the 128-key tiles those rows
// attend ("Inference for Interpretable Text-Diffusion Models", "Background",
// "KV Cache", "Paged Attention"; tiles classified as in "FlexAttention with
// Aligned Tiles").  The pair loads each K/V tile once: CTA r copies keys
// 64r .. 64r+63 of K (both 64-column halves of head_dim) and head_dim columns
// 64r .. 64r+63 of V (all 128 keys), 16 KB of each per tile.  The first CTA
// issues every tcgen05.mma with cta_group::2 (M = 256 across the pair): A is
// read from both CTAs (Q from shared memory, P from TMEM), B is split along N
// between them (K by keys, V by head-dim columns), and each CTA's TMEM
// receives its own 128 rows.
//
// TMEM per CTA (512 columns): S in two buffers (tile j in buffer j % 2, 128
// columns each), so that Q K^T of tile j+2 can be issued as soon as P V of
// tile j has read buffer j % 2, and the tensor core computes S(j+1) while the
// softmax works on S(j); O in two accumulators of 128 columns, O_lo for keys
// 0-63 of every tile and O_hi for keys 64-127.  Softmax warpgroup h handles
// keys 64h .. 64h+63 of each tile with its own running maximum and sum: two
// independent online softmaxes over disjoint key sets, merged once per item
// (O = (2^(m_lo - M) O_lo + 2^(m_hi - M) O_hi) / (2^(m_lo - M) l_lo +
// 2^(m_hi - M) l_hi), M = max(m_lo, m_hi)), so the two warpgroups never wait
// for each other inside a tile.
//
// Warp roles (384 threads, both CTAs):
//   warp 3      planner (the shared planner; the first CTA takes item indices
//               from the counter and posts them into the second CTA's mailbox)
//   warps 0, 2  loaders: this CTA's halves of each K/V tile (alternate tiles)
//               and, warp 0, its Q M-tile; the copies complete on the first
//               CTA's barriers.  Warp 2 also allocates and frees TMEM (both
//               CTAs, cta_group::2) before and after its loader role
//   warp 1      MMA issue (first CTA only)
//   warps 4-7   softmax of keys 0-63, warps 8-11 softmax of keys 64-127
// Every wait is bounded; on timeout a CTA records BCA_ERR_DEVICE_TIMEOUT and
// leaves its roles; the pair meets at a cluster barrier before TMEM is freed.
#include <atomic>
#include <climits>
#include <cstdint>

#include "attn_common.cuh"
#include "bca_internal.h"
#include "ptx_sm103.cuh"

namespace bca {
namespace {
using namespace attn;

constexpr int kHD = 128;
constexpr int kRegsLaunch = 168;   // 65536 / 384, rounded down to a multiple of 8
constexpr int kRegsControl = 112;
constexpr int kRegsSoftmax = 184;
static_assert(kRegsControl * 128 + kRegsSoftmax * 256 <= kRegsLaunch * kThreads, "register split");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
constexpr uint16_t kBoth = 3;              // multicast mask: both CTAs of the pair

struct PCfg {
  static constexpr int kQBytes = 2 * 16384;     // 128 rows x 128 columns, two 64-column halves
  static constexpr int kStageBytes = 16384;     // this CTA's half of a K or V tile
  static constexpr int kStages = 11;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffRec = kOffKV + kStages * kStageBytes;
  static constexpr int kTileSlots = 8;          // tile-full barriers (tiles in flight < 8)
  static constexpr int kNumBars = 2 * kNumRec + kTileSlots + kStages + 9 + 2 * kMailSlots;
  static constexpr int kOffBar = kOffRec + kNumRec * (int)sizeof(Rec);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // TMEM address, abort flag, mailbox
  static constexpr int kOffMl = kOffMisc + 64;              // merge exchange: float2 [2][128]
  static constexpr int kBytes = kOffMl + 2 * 128 * 8;
  static constexpr int kSmemAlloc = kBytes + 1024;  // base is aligned up to 1024 in the kernel
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kColS = 0;     // S buffer b at 128 b (P of keys 64h.. over columns 64h..)
  static constexpr int kColO = 256;   // O_lo at 256, O_hi at 384
  static_assert(kSmemAlloc <= 232448, "shared memory plan");
};

struct PBars {
  uint64_t* rec_full;
  uint64_t* rec_empty;
  uint64_t* tile_full;  // [kTileSlots] first CTA: both CTAs' K and V copies of a tile
  uint64_t* kv_empty;   // [kStages]
  uint64_t* q_full;     // first CTA: both CTAs' Q M-tiles
  uint64_t* q_empty;
  uint64_t* s_full;     // [2] S buffer ready
  uint64_t* p_full;     // [2 S buffers] first CTA: P of both key halves written by both CTAs
  uint64_t* o_full;
  uint64_t* o_empty;    // first CTA: both CTAs have read O
  uint64_t* drain;
  uint64_t* mail_full;  // [kMailSlots] second CTA
  uint64_t* mail_empty; // [kMailSlots] first CTA
};

struct PCtx {
  uint8_t* smem;
  Rec* ring;
  PBars bar;
  volatile int* abort_flag;
  int* mail;
  float2* ml;
  uint32_t tmem;
  uint32_t rank;
};

// ============================================================================
// loaders (warps 0 and 2, both CTAs)
// ============================================================================
// Each 16-row page box is one request to the SM's TMA unit, which takes a
// fixed time per request; one warp waiting for its next record and stages
// between tiles would leave the unit idle.  Two loader warps take alternate
// tiles (loader `which` the tiles t with t % 2 == which, counted over the
// CTA's run), so that one's waits overlap the other's requests; loader 0
// also loads Q.
__device__ __forceinline__ void run_loader(const PCtx& c, const AttnParams& p,
                                           const CUtensorMap* tm_q, const CUtensorMap* tm_kp,
                                           const CUtensorMap* tm_vp, const CUtensorMap* tm_kd,
                                           const CUtensorMap* tm_vd, int which, int lane) {
  using C = PCfg;
  const uint32_t q_base = smem_u32(c.smem + C::kOffQ);
  const uint32_t kv_base = smem_u32(c.smem + C::kOffKV);
  const uint32_t r = c.rank;
  const uint32_t q_full0 = mapa_shared(smem_u32(c.bar.q_full), 0);
  // lanes 0-7: K boxes (chunk 4r + l/2 of the tile, column half l % 2);
  // lanes 8-15: V boxes (chunk l - 8, column half r)
  const bool box = lane < 16;
  const bool is_v = lane >= 8;
  const int chunk = !box ? 0 : is_v ? lane - 8 : 4 * (int)r + (lane >> 1);
  const int half = is_v ? (int)r : (lane & 1);
  const uint32_t dst_off = is_v ? (uint32_t)(lane - 8) * 2048u
                                : (uint32_t)(lane & 1) * 8192u + (uint32_t)(lane >> 1) * 2048u;
  const uint32_t q_bytes = 2u * 2u * (uint32_t)(p.hpr * p.tpm) * 128u;  // both CTAs, both halves
  uint32_t ri = 0, u = 0, q_par = 0;
  bool q_used = false, ok = true;
  while (ok) {
    const Rec* rec = ring_get(c, p, ri);
    if (!rec) break;
    const int kind = rec->w[I_KIND];
    if (kind == kRecEnd) {
      ring_release(c, ri, lane);
      break;
    }
    if (kind == kRecItem) {
      const int qh = rec->w[I_QHEAD + r], qt = rec->w[I_QTOK + r];
      ring_release(c, ri, lane);
      ++ri;
      if (which != 0) continue;
      if (!wait_bar_warp(c, p, c.bar.q_empty, q_par ^ 1u)) break;
      if (lane == 0) {
        if (r == 0) mbar_arrive_expect_tx(c.bar.q_full, q_bytes);
        // the Q box holds hpr x tpm rows; a second M-tile past the item's
        // tokens loads rows nobody stores (or zero fill)
        tma_load_3d_pair(q_base, tm_q, q_full0, 0, qh, qt);
        tma_load_3d_pair(q_base + 16384, tm_q, q_full0, 64, qh, qt);
      }
      __syncwarp();
      q_par ^= 1u;
      q_used = true;
      continue;
    }
    const int src = rec->w[T_SRC], head = rec->w[T_HEAD];
    const int my_coord = rec->w[T_COORD + chunk];
    ring_release(c, ri, lane);
    ++ri;
    if ((int)((u / 2) & 1u) != which) {  // the other loader's tile
      u += 2;
      continue;
    }
    uint32_t slot[2];
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      slot[kv] = (u + kv) % C::kStages;
      if (ok && !wait_bar_warp(c, p, &c.bar.kv_empty[slot[kv]],
                                       (((u + kv) / C::kStages) & 1) ^ 1))
        ok = false;
    }
    if (!ok) break;
    // one barrier for the whole tile: K and V halves of both CTAs
    uint64_t* tfull = &c.bar.tile_full[(u / 2) % C::kTileSlots];
    if (r == 0 && lane == 0) mbar_arrive_expect_tx(tfull, 4u * C::kStageBytes);
    __syncwarp();
    if (box) {
      // every chunk is copied whole: a chunk past the valid keys has an
      // out-of-range coordinate (zero fill) or, from a dense source, holds
      // finite rows of other tokens that the softmax masks
      const uint32_t sl = is_v ? slot[1] : slot[0];
      const uint32_t d = kv_base + sl * C::kStageBytes + dst_off;
      const uint32_t bar = mapa_shared(smem_u32(tfull), 0);
      const CUtensorMap* map = src == 0 ? (is_v ? tm_vp : tm_kp) : (is_v ? tm_vd : tm_kd);
      if (src == 0) tma_load_2d_pair(d, map, bar, half * 64, my_coord);
      else tma_load_3d_pair(d, map, bar, half * 64, head, my_coord);
    }
    __syncwarp();
    u += 2;
  }
  // teardown: both CTAs' copies complete on the first CTA's barriers; the
  // first CTA's loader 0 waits for the last phases (the cluster barrier at
  // the end of the kernel keeps the second CTA resident until then)
  if (r == 0 && which == 0) {
    const uint32_t n_tiles = u / 2;
    for (uint32_t k = 0; k < (uint32_t)C::kTileSlots && k < n_tiles; ++k) {
      const uint32_t t = n_tiles - 1 - k;
      mbar_wait(&c.bar.tile_full[t % C::kTileSlots], (t / C::kTileSlots) & 1, c.abort_flag,
                kWaitTimeoutCycles);
    }
    if (q_used) mbar_wait(c.bar.q_full, q_par ^ 1u, c.abort_flag, kWaitTimeoutCycles);
  }
}

// ============================================================================
// MMA issue (warp 1 of the first CTA)
// ============================================================================
// S(buf) = Q K^T for the pair: M = 256, N = 128 keys (64 from each CTA),
// K = head_dim in steps of 16; operands K-major, 128-byte swizzled.
__device__ __forceinline__ void issue_qk(const PCtx& c, uint32_t buf, uint32_t slot) {
  using C = PCfg;
  constexpr uint32_t idesc = make_idesc_bf16(256, kTileKeys, 0, 0);
  const uint32_t qa = smem_u32(c.smem + C::kOffQ);
  const uint32_t ka = smem_u32(c.smem + C::kOffKV + slot * C::kStageBytes);
  const uint32_t d = c.tmem + C::kColS + buf * kTileKeys;
#pragma unroll
  for (int ks = 0; ks < kHD / 16; ++ks) {
    const int h = ks >> 2, kin = ks & 3;
    const uint64_t a = make_sdesc_sw128(qa + h * 16384 + kin * 32, 16, 1024);
    const uint64_t b = make_sdesc_sw128(ka + h * 8192 + kin * 32, 16, 1024);
    umma_bf16_pair(d, a, b, idesc, ks > 0 ? 1u : 0u);
  }
}

// O_h (+)= P_h V_h for the pair: M = 256, N = head_dim (64 columns from each
// CTA), K = the 64 keys 64h .. 64h+63 of the tile; P from TMEM (8 columns per
// 16 keys), V MN-major in shared memory.
__device__ __forceinline__ void issue_pv(const PCtx& c, uint32_t buf, int h, uint32_t slot,
                                         bool acc) {
  using C = PCfg;
  constexpr uint32_t idesc = make_idesc_bf16(256, kHD, 0, 1);
  const uint32_t pa = c.tmem + C::kColS + buf * kTileKeys + 64 * h;
  const uint32_t va = smem_u32(c.smem + C::kOffKV + slot * C::kStageBytes);
  const uint32_t d = c.tmem + C::kColO + 128 * h;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint64_t b = make_sdesc_sw128(va + (4 * h + kk) * 2048, C::kStageBytes, 1024);
    umma_bf16_ts_pair(d, pa + kk * 8, b, idesc, (acc || kk > 0) ? 1u : 0u);
  }
}

// Issue order for an item of n tiles (K(t), V(t) are loads 2t, 2t+1 of the
// item; buffer b(t) = t % 2 counted over the CTA's whole run):
//   S(0) S(1) | PV_lo(0) PV_hi(0) S(2) | PV_lo(1) PV_hi(1) S(3) | ...
// S(t+2) overwrites buffer b(t), whose P the two P V of tile t read first
// (tcgen05.mma operations from one thread execute in issue order).  Per tile
// the warp waits twice: for the copies of tile t+2 (K and V together; V(t)
// arrived with tile t) and for P of tile t (both key halves, both CTAs).
__device__ __forceinline__ void run_mma(const PCtx& c, const AttnParams& p, int lane) {
  using C = PCfg;
  uint32_t ri = 0, u = 0, q_par = 0, p_par = 0, o_par = 0, tc = 0;
  bool ok = true;
  // wait for both CTAs' copies of this CTA's tile number t
  auto tile_ready = [&](uint32_t t) {
    return wait_bar_warp(c, p, &c.bar.tile_full[t % C::kTileSlots], (t / C::kTileSlots) & 1);
  };
  while (ok) {
    const Rec* r = ring_get(c, p, ri);
    if (!r) break;
    const int kind = r->w[I_KIND], n_t = r->w[I_NT];
    ring_release(c, ri, lane);
    ++ri;
    if (kind == kRecEnd) break;
    if (!(ok = wait_bar_warp(c, p, c.bar.q_full, q_par))) break;
    q_par ^= 1u;
    const uint32_t ub = u;
    u += 2u * (uint32_t)n_t;
    ri += (uint32_t)n_t;  // the item's tile records are released by the planner for this warp
    for (int j = 0; j < 2 && j < n_t && ok; ++j) {
      const uint32_t uk = ub + 2u * (uint32_t)j, ks = uk % C::kStages;
      if (!(ok = tile_ready(uk / 2))) break;
      tc_fence_after();
      const uint32_t buf = (tc + (uint32_t)j) & 1u;
      issue_qk(c, buf, ks);
      umma_commit_pair_mc(&c.bar.s_full[buf], kBoth);
      umma_commit_pair_mc(&c.bar.kv_empty[ks], kBoth);
      if (j == n_t - 1) umma_commit_pair_mc(c.bar.q_empty, kBoth);  // last read of Q
    }
    for (int j = 0; j < n_t && ok; ++j) {
      const uint32_t uv = ub + 2u * (uint32_t)j + 1u, vs = uv % C::kStages;
      const uint32_t buf = (tc + (uint32_t)j) & 1u;
      const bool nxt = j + 2 < n_t;
      // the copies of tile j+2 are checked before the wait for P (they were
      // issued tiles ago)
      uint32_t ks = 0;
      if (nxt) {
        const uint32_t uk = ub + 2u * (uint32_t)(j + 2);
        ks = uk % C::kStages;
        if (!(ok = tile_ready(uk / 2))) break;
      }
      if (!(ok = wait_bar_warp(c, p, &c.bar.p_full[buf], (p_par >> buf) & 1))) break;
      p_par ^= 1u << buf;
      if (j == 0 && !(ok = wait_bar_warp(c, p, c.bar.o_empty, o_par ^ 1u))) break;
      tc_fence_after();
      issue_pv(c, buf, 0, vs, j > 0);
      issue_pv(c, buf, 1, vs, j > 0);
      // (this commit also tells the softmax warps that O holds P V of tile j)
      umma_commit_pair_mc(&c.bar.kv_empty[vs], kBoth);
      if (nxt) {
        issue_qk(c, buf, ks);
        umma_commit_pair_mc(&c.bar.s_full[buf], kBoth);
        umma_commit_pair_mc(&c.bar.kv_empty[ks], kBoth);
        if (j + 2 == n_t - 1) umma_commit_pair_mc(c.bar.q_empty, kBoth);
      }
    }
    if (!ok) break;
    umma_commit_pair_mc(c.bar.o_full, kBoth);
    o_par ^= 1u;
    tc += (uint32_t)n_t;
  }
  // teardown: wait until every MMA issued by this warp has completed
  umma_commit_pair(c.bar.drain);
  mbar_wait(c.bar.drain, 0, c.abort_flag, kWaitTimeoutCycles);
}

// ============================================================================
// softmax and merge (warps 4..11, both CTAs)
// ============================================================================
// Arrive on a barrier of the first CTA (this CTA's own in the first CTA).
__device__ __forceinline__ void arrive_first(const PCtx& c, uint64_t* bar, uint32_t bar0) {
  if (c.rank == 0) mbar_arrive(bar);
  else mbar_arrive_remote_cta(bar0);
}

// kBand: the multicanvas sliding-window band (a per-row lower key bound), a
// separate instantiation.
template <bool kBand>
__device__ __forceinline__ void run_softmax(const PCtx& c, const AttnParams& p, int h, int wq,
                                            int lane) {
  using C = PCfg;
  const int r = 32 * wq + lane;  // row within this CTA's M-tile == TMEM lane
  const uint32_t lane_addr = static_cast<uint32_t>(32 * wq) << 16;
  const uint32_t t_s = c.tmem + lane_addr + C::kColS + 64 * h;  // + 128 * buffer
  const uint32_t t_lo = c.tmem + lane_addr + C::kColO;
  const uint32_t t_hi = t_lo + 128;
  const uint32_t t_own = h ? t_hi : t_lo;
  const uint32_t p_full0[2] = {mapa_shared(smem_u32(&c.bar.p_full[0]), 0),
                               mapa_shared(smem_u32(&c.bar.p_full[1]), 0)};
  const uint32_t o_empty0 = mapa_shared(smem_u32(c.bar.o_empty), 0);
  const int m = (int)c.rank;
  const float sl2 = p.scale_log2;
  uint32_t ri = 0, s_par = 0, o_par = 0, tc = 0;
  while (true) {
    const Rec* rec = ring_get(c, p, ri);
    if (!rec) return;
    const int kind = rec->w[I_KIND];
    const int n_t = rec->w[I_NT], qmode = rec->w[I_QMODE];
    const int qtok = rec->w[I_QTOK + m], qhead = rec->w[I_QHEAD + m];
    const int ntok = rec->w[I_NTOK + m], qbase = rec->w[I_QBASE + m];
    const int P0 = rec->w[I_P0], Dblk = rec->w[I_DBLK], split = rec->w[I_SPLIT];
    ring_release(c, ri, lane);
    ++ri;
    if (kind == kRecEnd) return;
    const int tok = r / p.hpr;
    const bool valid = r < p.hpr * p.tpm && tok < ntok;
    // row q sees key positions in [lo, lim) (rows nobody stores see every
    // valid key: lim = INT_MAX)
    int lim = INT_MAX, lo = INT_MIN;
    if (valid) {
      const int qpos = qmode == 0 ? qbase + tok : __ldg(p.live_pos + qbase + tok);
      lim = row_limit(qpos, P0, Dblk);
      if (kBand) lo = qpos - p.window + 1;
    }
    // band: the range of the warp's lower bounds [lo_min, lo_max] (rows that
    // store nothing excluded); only keys with positions inside it can be
    // seen by some of the warp's rows and not by others
    int lo_min = INT_MAX, lo_max = INT_MIN;
    if (kBand) {
      lo_min = warp_min(valid ? lo : INT_MAX);
      lo_max = warp_max(valid ? lo : INT_MIN);
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < n_t; ++j) {
      const Rec* t = ring_get(c, p, ri);
      if (!t) return;
      const int full = t->w[T_FULL], nvalid = t->w[T_NVALID], kbase = t->w[T_KBASE];
      const int kmode = t->w[T_KMODE];
      // Stored positions (arena keys: kmode 1, 16 consecutive kv_pos entries
      // per chunk from the chunk's offset; live keys: kmode 2, consecutive
      // live_pos entries): lane l fetches keys 64h + 2l, 64h + 2l + 1 now,
      // so that the load is in flight while S is computed; INT_MAX past the
      // valid keys (never seen).
      int kp0 = INT_MAX, kp1 = INT_MAX;
      if (!full && kmode != 0) {
        const int k0 = 64 * h + 2 * lane;
        if (k0 < nvalid) {
          const int32_t* src = kmode == 1
                                   ? p.kv_pos + t->w[T_KOFF + k0 / kChunkKeys] + k0 % kChunkKeys
                                   : p.live_pos + kbase + k0;
          if (k0 + 2 <= nvalid && (reinterpret_cast<uintptr_t>(src) & 7) == 0) {
            const int2 v2 = __ldg(reinterpret_cast<const int2*>(src));
            kp0 = v2.x;
            kp1 = v2.y;
          } else {
            kp0 = __ldg(src);
            if (k0 + 1 < nvalid) kp1 = __ldg(src + 1);
          }
        }
      }
      ring_release(c, ri, lane);
      ++ri;
      const uint32_t buf = tc & 1u;
      if (!wait_bar_warp(c, p, &c.bar.s_full[buf], (s_par >> buf) & 1)) return;
      s_par ^= 1u << buf;
      tc_fence_after();
      uint32_t sa[32], sb[32];  // scores of keys 64h + k: k < 32 in sa, k >= 32 in sb
      tmem_ld64_sync(t_s + 128 * buf, sa, sb);
#define SV(k) ((k) < 32 ? sa[(k)] : sb[(k) - 32])
      if (!full) {
        if (kmode == 0) {
          // key 64h + k is at position kbase + 64h + k: visible iff it is one
          // of the tile's valid keys and in [lo, lim) (lim >= 0 and kbase >= 0,
          // so lim - kbase cannot overflow; lo - kbase is clamped)
          const int hi_cut = max(0, min(64, min(nvalid, lim - kbase) - 64 * h));
          const int lo_cut =
              kBand ? max(0, min(64, (int)max((long long)lo - kbase, -1ll) - 64 * h)) : 0;
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k >= hi_cut || k < lo_cut) SV(k) = __float_as_uint(-INFINITY);
        } else {
          // visibility of key 64h + 2l + i for this row is bit l of vis[i]:
          // rows with the same upper limit share one pair of ballots over the
          // lanes' positions (a warp's rows: a few tokens of one or two
          // canvases)
          uint32_t vis0 = 0u, vis1 = 0u;
          bool done = !valid;  // rows past the item's tokens see nothing
          while (true) {
            const uint32_t pend = __ballot_sync(0xffffffffu, !done);
            if (pend == 0u) break;
            const int leader = __ffs(pend) - 1;
            const int L = __shfl_sync(0xffffffffu, lim, leader);
            const uint32_t b0 = __ballot_sync(0xffffffffu, kp0 < L);
            const uint32_t b1 = __ballot_sync(0xffffffffu, kp1 < L);
            if (!done && lim == L) {
              vis0 = b0;
              vis1 = b1;
              done = true;
            }
          }
          if (kBand) {
            // with the band each token has its own lower bound: keys at or
            // above the warp's largest bound pass every row's, keys below
            // its smallest pass none, and the few in between are tested one
            // by one against this row's bound
            uint32_t m0 = __ballot_sync(0xffffffffu, kp0 >= lo_max);
            uint32_t m1 = __ballot_sync(0xffffffffu, kp1 >= lo_max);
            uint32_t a0 = __ballot_sync(0xffffffffu, kp0 >= lo_min && kp0 < lo_max);
            uint32_t a1 = __ballot_sync(0xffffffffu, kp1 >= lo_min && kp1 < lo_max);
            while (a0 != 0u) {
              const int l = __ffs(a0) - 1;
              if (__shfl_sync(0xffffffffu, kp0, l) >= lo) m0 |= 1u << l;
              a0 &= a0 - 1u;
            }
            while (a1 != 0u) {
              const int l = __ffs(a1) - 1;
              if (__shfl_sync(0xffffffffu, kp1, l) >= lo) m1 |= 1u << l;
              a1 &= a1 - 1u;
            }
            vis0 &= m0;
            vis1 &= m1;
          }
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (!((((k & 1) ? vis1 : vis0) >> (k >> 1)) & 1u)) SV(k) = __float_as_uint(-INFINITY);
        }
        // V rows past the valid keys inside the last partly valid 16-key
        // chunk came in with its box and may hold anything (a pool page's
        // unused slots, another buffer's rows): their P is 0, but 0 * NaN is
        // NaN in P V, so warpgroup 0 zeroes them in this CTA's V stage
        // before P is published
        if (h == 0 && (nvalid & (kChunkKeys - 1)) != 0) {
          const int n_zero = kChunkKeys - (nvalid & (kChunkKeys - 1));
          const uint32_t vrow0 =
              smem_u32(c.smem + C::kOffKV + ((2u * tc + 1u) % C::kStages) * C::kStageBytes) +
              (uint32_t)nvalid * 128u;
          for (int i = r; i < n_zero * 8; i += 128)
            st_shared_v4(vrow0 + (uint32_t)i * 16u, 0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
      }
      // row maximum of the raw scores (the scale is positive), in log2 units
      float mx[4] = {__uint_as_float(SV(0)), __uint_as_float(SV(1)), __uint_as_float(SV(2)),
                     __uint_as_float(SV(3))};
#pragma unroll
      for (int k = 4; k < 60; k += 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mx[i] = fmax3(mx[i], __uint_as_float(SV(k + 2 * i)), __uint_as_float(SV(k + 2 * i + 1)));
      }
      mx[0] = fmax3(mx[0], __uint_as_float(SV(60)), __uint_as_float(SV(61)));
      mx[1] = fmax3(mx[1], __uint_as_float(SV(62)), __uint_as_float(SV(63)));
      const float mt = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
      const float m_new = fmaxf(m_run, mt);
      bool rescale = false;
      float alpha = 1.0f;
      if (j == 0) {
        m_run = m_new;
      } else if (m_new > m_run + kRescaleThreshold) {
        rescale = true;
        alpha = ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O_h holds the P V of the earlier tiles; the last of them (this
        // CTA's tile tc - 1) may still be running.  The MMA warp frees the
        // stage of V(tc - 1) (load 2 tc - 1) right after that P V, so its
        // completion is that stage's phase; the stage's next phase needs the
        // load 11 later consumed (Q K^T of tile tc + 5, after P of tile
        // tc + 3), so no later phase can have completed.
        const uint32_t lv = 2u * tc - 1u;
        if (!wait_bar_warp(c, p, &c.bar.kv_empty[lv % C::kStages], (lv / C::kStages) & 1u)) return;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < kHD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32_sync(t_own + c0, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(t_own + c0, o);
        }
      }
      const float ref = m_run == -INFINITY ? 0.f : m_run;
      // p = 2^(s * scale * log2(e) - ref), two keys per paired FMA / add
      const float2 scale2 = make_float2(sl2, sl2), nref2 = make_float2(-ref, -ref);
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int cq = 0; cq < 2; ++cq) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 x = ffma2(make_float2(__uint_as_float(SV(32 * cq + 2 * k)),
                                             __uint_as_float(SV(32 * cq + 2 * k + 1))),
                                 scale2, nref2);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          sum2 = fadd2(sum2, pp);
          w[k] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st16(t_s + 128 * buf + 16 * cq, w);  // P over the first 32 of this half's columns
      }
#undef SV
      l_run = l_run * alpha + (sum2.x + sum2.y);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_first(c, &c.bar.p_full[buf], buf ? p_full0[1] : p_full0[0]);
      ++tc;
    }
    // ---- end of the item: merge the two halves, store ----
    if (!wait_bar_warp(c, p, c.bar.o_full, o_par & 1)) return;
    o_par ^= 1u;
    tc_fence_after();
    c.ml[h * 128 + r] = make_float2(m_run, l_run);
    named_barrier_sync(2, 256);
    const float2 other = c.ml[(h ^ 1) * 128 + r];
    const float m_lo = h ? other.x : m_run, l_lo = h ? other.y : l_run;
    const float m_hi = h ? m_run : other.x, l_hi = h ? l_run : other.y;
    const float M = fmaxf(m_lo, m_hi);
    const float a_lo = m_lo == -INFINITY ? 0.f : ex2_approx(m_lo - M);
    const float a_hi = m_hi == -INFINITY ? 0.f : ex2_approx(m_hi - M);
    const float L = a_lo * l_lo + a_hi * l_hi;
    // this warpgroup merges head-dim columns 64h .. 64h+63 of both accumulators
    const int cb = 64 * h;
    if (split < 0) {
      const float inv = L > 0.f ? 1.0f / L : 0.f;
      const float s_lo = a_lo * inv, s_hi = a_hi * inv;
      uint16_t* dst = p.out + ((size_t)(qtok + tok) * p.Hq + qhead + (r % p.hpr)) * kHD + cb;
#pragma unroll 1
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t o1[32], o2[32];
        tmem_ld32x2_sync(t_lo + cb + c0, t_hi + cb + c0, o1, o2);
        if (valid) {
          // the row's 32 columns as bf16: two 32-byte stores (16-byte ones
          // when the output is only 16-byte aligned)
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(
                __uint_as_float(o1[2 * i]) * s_lo + __uint_as_float(o2[2 * i]) * s_hi,
                __uint_as_float(o1[2 * i + 1]) * s_lo + __uint_as_float(o2[2 * i + 1]) * s_hi);
          if (p.out_align32) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint32_t v8[8] = {w[8 * k], w[8 * k + 1], w[8 * k + 2], w[8 * k + 3],
                                      w[8 * k + 4], w[8 * k + 5], w[8 * k + 6], w[8 * k + 7]};
              st_global_v8(dst + c0 + 16 * k, v8);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              *reinterpret_cast<uint4*>(dst + c0 + 8 * k) =
                  make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
          }
        }
      }
    } else {
      // split-KV partial: (M, L) and the unnormalised merged O of this chunk
      const int R = m * kRowsPerMTile + r;
#pragma unroll 1
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t o1[32], o2[32];
        tmem_ld32x2_sync(t_lo + cb + c0, t_hi + cb + c0, o1, o2);
        if (valid) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float4 v;
            v.x = __uint_as_float(o1[4 * k + 0]) * a_lo + __uint_as_float(o2[4 * k + 0]) * a_hi;
            v.y = __uint_as_float(o1[4 * k + 1]) * a_lo + __uint_as_float(o2[4 * k + 1]) * a_hi;
            v.z = __uint_as_float(o1[4 * k + 2]) * a_lo + __uint_as_float(o2[4 * k + 2]) * a_hi;
            v.w = __uint_as_float(o1[4 * k + 3]) * a_lo + __uint_as_float(o2[4 * k + 3]) * a_hi;
            const size_t idx = (((size_t)split * (kHD / 4) + ((cb + c0) / 4 + k)) * 256 + R) * 4;
            *reinterpret_cast<float4*>(p.part_o + idx) = v;
          }
        }
      }
      if (valid && h == 0)
        *reinterpret_cast<float2*>(p.part_ml + ((size_t)split * 256 + R) * 2) = make_float2(M, L);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_first(c, c.bar.o_empty, o_empty0);
  }
}

// ============================================================================
// the kernel
// ============================================================================
template <bool kBand>
__global__ void __launch_bounds__(kThreads, 1)
    attention_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_kp,
                          const __grid_constant__ CUtensorMap tm_vp,
                          const __grid_constant__ CUtensorMap tm_kd,
                          const __grid_constant__ CUtensorMap tm_vd,
                          const __grid_constant__ AttnParams p) {
  using C = PCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  PCtx c;
  c.smem = smem;
  c.rank = cluster_ctarank();
  c.ring = reinterpret_cast<Rec*>(smem + C::kOffRec);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  c.bar.rec_full = bars;
  c.bar.rec_empty = bars + kNumRec;
  c.bar.tile_full = bars + 2 * kNumRec;
  c.bar.kv_empty = c.bar.tile_full + C::kTileSlots;
  c.bar.q_full = c.bar.kv_empty + C::kStages;
  c.bar.q_empty = c.bar.q_full + 1;
  c.bar.s_full = c.bar.q_empty + 1;
  c.bar.p_full = c.bar.s_full + 2;
  c.bar.o_full = c.bar.p_full + 2;
  c.bar.o_empty = c.bar.o_full + 1;
  c.bar.drain = c.bar.o_empty + 1;
  c.bar.mail_full = c.bar.drain + 1;
  c.bar.mail_empty = c.bar.mail_full + kMailSlots;
  static_assert(2 * kNumRec + C::kTileSlots + C::kStages + 9 + 2 * kMailSlots == C::kNumBars,
                "barriers");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  c.abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  c.mail = reinterpret_cast<int*>(smem + C::kOffMisc + 16);
  c.ml = reinterpret_cast<float2*>(smem + C::kOffMl);

  if (threadIdx.x == 0) {
    // the ring's consumers: 2 loaders + 8 softmax warps, and in the first
    // CTA the MMA warp (whose tile records the planner releases)
    const uint32_t consumers = c.rank == 0 ? 11u : 10u;
    for (int i = 0; i < kNumRec; ++i) {
      mbar_init(&c.bar.rec_full[i], 1);
      mbar_init(&c.bar.rec_empty[i], consumers);
    }
    for (int i = 0; i < C::kTileSlots; ++i) mbar_init(&c.bar.tile_full[i], 1);
    for (int i = 0; i < C::kStages; ++i) mbar_init(&c.bar.kv_empty[i], 1);
    mbar_init(c.bar.q_full, 1);
    mbar_init(c.bar.q_empty, 1);
    for (int b = 0; b < 2; ++b) mbar_init(&c.bar.s_full[b], 1);
    // one per S buffer: a softmax warp may run one tile ahead of the others
    // (S of the next tile is ready early), and its arrival must not complete
    // the phase of the tile the others are still on
    for (int b = 0; b < 2; ++b) mbar_init(&c.bar.p_full[b], 16);  // 8 warps of each CTA
    mbar_init(c.bar.o_full, 1);
    mbar_init(c.bar.o_empty, 16);      // 8 warps of each CTA
    mbar_init(c.bar.drain, 1);
    for (int i = 0; i < kMailSlots; ++i) {
      mbar_init(&c.bar.mail_full[i], 1);
      mbar_init(&c.bar.mail_empty[i], 1);
    }
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
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised before any remote arrival or copy
  cluster_sync();
  tc_fence_after();
  c.tmem = *tmem_slot;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // register split as in the single-CTA kernel (see attention.cu)
  if (warp < 4) {
    regs_dealloc<kRegsControl>();
    named_barrier_sync(1, kThreads);
    if (warp == 3) {
      Planner<PCtx, true> pl(p, c, lane);
      pl.run();
    } else if (warp == 0 || warp == 2) {
      run_loader(c, p, &tm_q, &tm_kp, &tm_vp, &tm_kd, &tm_vd, warp >> 1, lane);
    } else if (warp == 1 && c.rank == 0) {
      run_mma(c, p, lane);
    }
    __syncwarp();
    regs_alloc<kRegsLaunch>();
  } else {
    regs_alloc<kRegsSoftmax>();
    named_barrier_sync(1, kThreads);
    run_softmax<kBand>(c, p, (warp - 4) >> 2, warp & 3, lane);
    __syncwarp();
    regs_dealloc<kRegsLaunch>();
  }

  tc_fence_before();
  __syncthreads();
  // the first CTA has drained the pair's MMAs and copies; no thread of
  // either CTA touches the other's shared memory after this point
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(c.tmem, C::kTmemCols);
  }
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

}  // namespace

namespace {
template <bool kBand>
cudaError_t launch_pair(const AttnParams& p, const AttnMaps& maps, int n_pairs,
                        cudaStream_t stream) {
  using C = PCfg;
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (!cached || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attention_pair_kernel<kBand>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits for registers released by setmaxnreg.dec; the
    // split must fit what the block is launched with
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attention_pair_kernel<kBand>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
    if (cached) configured[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n_pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attention_pair_kernel<kBand>, maps.q, maps.kp, maps.vp, maps.kd,
                            maps.vd, p);
}
}  // namespace

cudaError_t launch_attention_pair(const AttnParams& p, const AttnMaps& maps, int n_pairs,
                                  cudaStream_t stream) {
  const bool band = p.mode == kModeMulticanvas && p.window > 0;
  return band ? launch_pair<true>(p, maps, n_pairs, stream)
              : launch_pair<false>(p, maps, n_pairs, stream);
}

int attention_pair_max_pairs(int n_sms) {
  using C = PCfg;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(attention_pair_kernel<false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (n_sms / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attention_pair_kernel<false>, &cfg) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace bca
