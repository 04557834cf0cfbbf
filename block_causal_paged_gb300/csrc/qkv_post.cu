// QKV-post: the step between the fused QKV projection and attention, in one
// pass over the projection's output.
//
// "Inference: Fewer, smaller forwards", "Advancement 16" lists an optional
// fused QKV-post (RoPE, norms, arena write), and "Advancement 10" bakes RoPE
// into the keys at each token's true absolute position, so that the cache
// can be stored out of order.  Per token (rows of qkv [Hq + 2 Hkv, d]:
// query heads, then key heads, then value heads):
//   norms: each query / key head vector x becomes x * w / sqrt(mean(x^2) + eps)
//          (w of length d shared by the heads; skipped where w is null);
//   RoPE:  the pair (x_i, x_{i+d/2}), i < d/2, is rotated by the angle
//          pos * theta^(-2i/d) (skipped for theta = 0);
//   values pass through;
// and the finished key / value rows are optionally written into the paged
// cache at write_pos (page page_table[b][p / S], slot p % S), with the
// token's position stored in kv_pos (arena mode).
//
// A warp per group of 4 heads of a token, a half-warp per head: each lane
// holds d/32 consecutive elements and their rotation partners d/2 further, so
// a rotation needs no shuffle and every load of a head pair is contiguous.
// The group's loads are issued one token ahead of the processing (software
// pipeline), and the grid is what stays resident.  Arithmetic in fp32, one
// rounding to bf16 at the end.  The angle needs no floating point on a large argument:
// the host gives each pair's frequency in turns per position as a 64-bit
// fixed-point fraction F, and pos * F modulo 2^64 (integer arithmetic, exact
// for any int32 position) is the angle's fraction of a turn; its top 32 bits,
// read as a signed number, map to [-pi, pi) for the single-precision sine and
// cosine (a phase accumulator).  Its error is that of F, about 2^-22 turns
// at the largest positions.
#include <atomic>
#include <cstdint>
#include <type_traits>

#include "bca_internal.h"

namespace bca {
namespace {

constexpr int kErrPageOob = -16;
constexpr int kErrBadLength = -17;
constexpr int kThreadsQP = 256;
constexpr int kUnroll = 4;  // heads of one work unit, loaded together

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Warp w of W = n_grp * W_t warps takes head group g = w % n_grp (heads
// 4g .. 4g+3) of tokens w / n_grp, + W_t, ...: the group, its heads' kinds and
// output offsets are fixed for the warp's life.  Each half-warp takes one head
// of a pair (heads 4g + 2p + s for half s): lane j of the half holds elements
// kV*j .. kV*j+kV-1 and their rotation partners d/2 further (kV = d/32), so a
// head's sum of squares takes four shuffle rounds shared by the pair.
template <int HD>
__global__ void __launch_bounds__(kThreadsQP) qkv_post_kernel(const __grid_constant__ QkvPostParams c,
                                                              int n_grp, int W) {
  constexpr int kHalf = HD / 2;
  constexpr int kV = HD / 32;          // elements per lane in each half
  constexpr int kPairs = kUnroll / 2;  // head pairs per group
  using Vec = typename std::conditional<kV == 4, uint2, uint32_t>::type;
  const int lane = threadIdx.x & 31, sub = lane >> 4, jl = lane & 15;
  const int w = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (w >= W) return;
  const int g = w % n_grp, W_t = W / n_grp;
  const int T = c.B * c.n;
  const int Htot = c.Hq + 2 * c.Hkv;
  const int h0 = g * kUnroll;
  const bool any_qk = h0 < c.Hq + c.Hkv;
  const bool any_kv = h0 + kUnroll > c.Hq && h0 < Htot;
  const bool first_kv = h0 <= c.Hq && c.Hq < h0 + kUnroll;  // reports errors, stores kv_pos
  const bool has_qw = c.q_norm_w != nullptr, has_kw = c.k_norm_w != nullptr;
  // this lane's heads: kind (0 q, 1 k, 2 v), index within its kind, validity
  int kd[kPairs], gh[kPairs];
  bool live[kPairs];
#pragma unroll
  for (int p = 0; p < kPairs; ++p) {
    const int h = h0 + 2 * p + sub;
    live[p] = h < Htot;
    kd[p] = h < c.Hq ? 0 : (h < c.Hq + c.Hkv ? 1 : 2);
    gh[p] = kd[p] == 0 ? h : (kd[p] == 1 ? h - c.Hq : h - c.Hq - c.Hkv);
  }
  // this lane's elements i = kV*jl + e and i + d/2: the norm weight of each
  // of its heads (fixed for the warp's life) and the RoPE turns
  float wsel[kPairs][2 * kV];
  bool normed[kPairs];
  unsigned long long turns[kV];
#pragma unroll
  for (int p = 0; p < kPairs; ++p) {
    const uint16_t* wv = kd[p] == 0 ? c.q_norm_w : (kd[p] == 1 ? c.k_norm_w : nullptr);
    normed[p] = wv != nullptr;
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      const int i = kV * jl + e;
      wsel[p][e] = wv ? bf2f(__ldg(wv + i)) : 1.f;
      wsel[p][kV + e] = wv ? bf2f(__ldg(wv + i + kHalf)) : 1.f;
    }
  }
#pragma unroll
  for (int e = 0; e < kV; ++e) turns[e] = c.rope_turns[kV * jl + e];
  // a group of value heads only is a copy
  const bool all_v = h0 >= c.Hq + c.Hkv;
  const float kTurnToRad = 6.28318530717958647692f / 4294967296.0f;  // 2 pi / 2^32
  auto load_tok = [&](int tkn, Vec (&raw)[kPairs][2], int& pos, int& wp) {
    const uint16_t* src = c.qkv + ((size_t)tkn * Htot + h0 + sub) * HD + kV * jl;
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      if (live[p]) {
        raw[p][0] = __ldg(reinterpret_cast<const Vec*>(src + 2 * p * HD));
        raw[p][1] = __ldg(reinterpret_cast<const Vec*>(src + 2 * p * HD + kHalf));
      }
    }
    pos = (c.positions && (any_qk || c.kv_pos)) ? __ldg(c.positions + tkn) : 0;
    wp = (c.write_pos && any_kv) ? __ldg(c.write_pos + tkn) : -1;
  };
  auto unpack = [](const Vec& v, float* f) {
    if constexpr (kV == 4) {
      f[0] = __uint_as_float(v.x << 16);
      f[1] = __uint_as_float(v.x & 0xffff0000u);
      f[2] = __uint_as_float(v.y << 16);
      f[3] = __uint_as_float(v.y & 0xffff0000u);
    } else {
      f[0] = __uint_as_float(v << 16);
      f[1] = __uint_as_float(v & 0xffff0000u);
    }
  };
  // software pipeline: the next token's rows are loaded before this one is processed
  Vec raw[kPairs][2];
  int pos = 0, wp = -1;
  int tkn = w / n_grp;
  if (tkn < T) load_tok(tkn, raw, pos, wp);
  for (; tkn < T; tkn += W_t) {
    Vec nraw[kPairs][2];
    int npos = 0, nwp = -1;
    if (tkn + W_t < T) load_tok(tkn + W_t, nraw, npos, nwp);
    // cache destination of this token's key / value rows
    int page = -1, slot = 0;
    if (wp >= 0) {
      const int b = tkn / c.n;
      if ((long long)wp >= (long long)c.max_pages * c.S) {
        if (lane == 0 && first_kv) atomicCAS(&c.hdr->status, 0, kErrBadLength);
      } else {
        const int pg = __ldg(c.page_table + (size_t)b * c.max_pages + wp / c.S);
        if (pg < 0 || pg >= c.num_pages) {
          if (lane == 0 && first_kv) atomicCAS(&c.hdr->status, 0, kErrPageOob);
        } else {
          page = pg;
          slot = wp % c.S;
          if (c.kv_pos && lane == 0 && first_kv) c.kv_pos[(size_t)page * c.S + slot] = pos;
        }
      }
    }
    float cs[kV], sn[kV];
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      cs[e] = 1.f;
      sn[e] = 0.f;
      if (c.rope_theta > 0.f && any_qk) {
        const unsigned long long ph = (unsigned long long)(long long)pos * turns[e];
        const float red = (float)(int)(unsigned)(ph >> 32) * kTurnToRad;  // in [-pi, pi)
        __sincosf(red, &sn[e], &cs[e]);  // |red| <= pi: the fast form is accurate here
      }
    }
    // the heads in branch-free phases: unpack, norms, rotation, stores
    float y[kPairs][2 * kV];
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      unpack(raw[p][0], &y[p][0]);
      unpack(raw[p][1], &y[p][kV]);
    }
    if (!all_v && (has_qw || has_kw)) {
      float ss[kPairs];
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        ss[p] = 0.f;
#pragma unroll
        for (int e = 0; e < 2 * kV; ++e) ss[p] = fmaf(y[p][e], y[p][e], ss[p]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {  // within each half-warp
#pragma unroll
        for (int p = 0; p < kPairs; ++p) ss[p] += __shfl_xor_sync(0xffffffffu, ss[p], o);
      }
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        const float r = normed[p] ? rsqrtf(ss[p] * (1.0f / HD) + c.eps) : 1.f;
#pragma unroll
        for (int e = 0; e < 2 * kV; ++e) y[p][e] *= r * wsel[p][e];
      }
    }
    if (!all_v && c.rope_theta > 0.f) {
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
#pragma unroll
        for (int e = 0; e < kV; ++e) {
          const float a = y[p][e], bb = y[p][kV + e];
          y[p][e] = a * cs[e] - bb * sn[e];
          y[p][kV + e] = bb * cs[e] + a * sn[e];
        }
      }
    }
    uint16_t* const qb = c.q_out + (size_t)tkn * c.Hq * HD + kV * jl;
    uint16_t* const kb = c.k_out + (size_t)tkn * c.Hkv * HD + kV * jl;
    uint16_t* const vb = c.v_out + (size_t)tkn * c.Hkv * HD + kV * jl;
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      if (!live[p]) continue;
      Vec o0 = raw[p][0], o1 = raw[p][1];  // values pass through as bits
      if (kd[p] != 2) {
        if constexpr (kV == 4) {
          o0 = make_uint2(pack_bf16x2(y[p][0], y[p][1]), pack_bf16x2(y[p][2], y[p][3]));
          o1 = make_uint2(pack_bf16x2(y[p][4], y[p][5]), pack_bf16x2(y[p][6], y[p][7]));
        } else {
          o0 = pack_bf16x2(y[p][0], y[p][1]);
          o1 = pack_bf16x2(y[p][2], y[p][3]);
        }
      }
      uint16_t* dst = (kd[p] == 0 ? qb : (kd[p] == 1 ? kb : vb)) + gh[p] * HD;
      *reinterpret_cast<Vec*>(dst) = o0;
      *reinterpret_cast<Vec*>(dst + kHalf) = o1;
      if (kd[p] != 0 && page >= 0) {
        uint16_t* cache = (kd[p] == 1 ? c.k_pool : c.v_pool) +
                          (((size_t)page * c.Hkv + gh[p]) * c.S + slot) * HD + kV * jl;
        *reinterpret_cast<Vec*>(cache) = o0;
        *reinterpret_cast<Vec*>(cache + kHalf) = o1;
      }
    }
#pragma unroll
    for (int p = 0; p < kPairs; ++p) {
      raw[p][0] = nraw[p][0];
      raw[p][1] = nraw[p][1];
    }
    pos = npos;
    wp = nwp;
  }
}

}  // namespace

cudaError_t launch_qkv_post(const QkvPostParams& c, int head_dim, int n_sms, cudaStream_t stream) {
  const long long T = (long long)c.B * c.n;
  const int n_grp = (c.Hq + 2 * c.Hkv + kUnroll - 1) / kUnroll;
  // warps: a whole number of groups, at most what is resident at once (each
  // warp loops over tokens), at most one per unit
  // blocks per SM, per head dim: a fixed property of the kernel, queried once
  // (host threads that race here store the same value)
  static std::atomic<int> resident[2] = {{0}, {0}};
  const int hi = head_dim == 128 ? 1 : 0;
  int per_sm = resident[hi].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    int nb = 0;
    const cudaError_t e = head_dim == 128
        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, qkv_post_kernel<128>, kThreadsQP, 0)
        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, qkv_post_kernel<64>, kThreadsQP, 0);
    if (e != cudaSuccess) return e;
    per_sm = nb > 0 ? nb : 1;
    resident[hi].store(per_sm, std::memory_order_relaxed);
  }
  long long W = (long long)(n_sms > 0 ? n_sms : 1) * per_sm * (kThreadsQP / 32);
  if (W > T * n_grp) W = T * n_grp;
  W = W / n_grp * n_grp;
  if (W < n_grp) W = n_grp;
  const long long blocks = (W + kThreadsQP / 32 - 1) / (kThreadsQP / 32);
  if (head_dim == 128)
    qkv_post_kernel<128><<<(unsigned)blocks, kThreadsQP, 0, stream>>>(c, n_grp, (int)W);
  else
    qkv_post_kernel<64><<<(unsigned)blocks, kThreadsQP, 0, stream>>>(c, n_grp, (int)W);
  return cudaGetLastError();
}

}  // namespace bca
