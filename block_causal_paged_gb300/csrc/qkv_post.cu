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
// Lane layout: a head is spread over L = d/16 lanes, lane j of its group
// holding elements 8j .. 8j + 7 of the head's first half and their rotation
// partners d/2 further (two 16-byte accesses), so a rotation needs no
// shuffle and a head's sum of squares takes log2(L) shuffle rounds; a warp
// pass covers 32/L heads.  Work unit: 8 consecutive heads of a token's row
// (one or two warp passes).  The units of all tokens, in memory order, are
// cut into equal contiguous ranges, one per resident warp (so any batch
// spreads over the whole GPU).  A warp loads unit i + 1 while it processes
// unit i; in a unit the heads' sums of squares and their shuffle rounds are
// interleaved.  The norm weights sit in shared memory in word-major order,
// so that the lanes of a head read consecutive 16-byte entries.
// A token's sines and cosines are computed once per warp that touches it,
// and the token metadata (position, cache page and slot) is loaded 32 tokens
// at a time, a lane per token.  Arithmetic in fp32 on (x_i, x_(i+1)) pairs,
// the halves of a bf16x2 word, with paired f32x2 instructions; one rounding
// to bf16 at the end.  The angle needs no floating point on a large argument:
// the host gives each pair's frequency in turns per position as a 64-bit
// fixed-point fraction F, and pos * F modulo 2^64 (integer arithmetic, exact
// for any int32 position) is the angle's fraction of a turn; its top 32 bits,
// read as a signed number, map to [-pi, pi) for the single-precision sine and
// cosine (a phase accumulator).  Its error is that of F, about 2^-22 turns
// at the largest positions.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <type_traits>

#include "bca_internal.h"
#include "ptx_sm103.cuh"

namespace bca {
namespace {

constexpr int kErrPageOob = -16;
constexpr int kErrBadLength = -17;
constexpr int kThreadsQP = 256;
constexpr int kUnitHeads = 8;  // heads per work unit (of one token)

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  return ffma2(a, b, make_float2(0.f, 0.f));
}
// a bf16x2 word as the float pair (low element, high element)
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
__device__ __forceinline__ uint32_t word4(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

template <int HD>
__global__ void __launch_bounds__(kThreadsQP, 2) qkv_post_kernel(const __grid_constant__ QkvPostParams c,
                                                                 int per_warp) {
  constexpr int kHalf = HD / 2;
  constexpr int kL = HD / 16;              // lanes per head
  constexpr int kHpp = 32 / kL;            // heads per warp pass
  constexpr int kPasses = kUnitHeads / kHpp;
  constexpr int kWords = 4;                // bf16x2 words per lane in each half of a head
  static_assert(kPasses * kHpp == kUnitHeads, "unit shape");
  const int lane = threadIdx.x & 31, hs = lane / kL, jl = lane % kL;
  // norm weights of the element pairs of lane jl: word k of a head's first
  // half holds elements i, i + 1 (i = 8 jl + 2 k), of its second half
  // i + d/2, i + d/2 + 1; s_w[q|k][k * L + jl] = {w_i, w_(i+1), w_(i+d/2), w_(i+d/2+1)}
  __shared__ float4 s_w[2][kHalf / 2];
  const bool has_qw = c.q_norm_w != nullptr, has_kw = c.k_norm_w != nullptr;
  for (int j = threadIdx.x; j < kHalf; j += blockDim.x) {
    const int which = j / (kHalf / 2), e = j % (kHalf / 2);  // e = k * L + jl
    const int i = 8 * (e % kL) + 2 * (e / kL);
    const uint16_t* wv = which == 0 ? c.q_norm_w : c.k_norm_w;
    s_w[which][e] =
        wv ? make_float4(bf2f(__ldg(wv + i)), bf2f(__ldg(wv + i + 1)), bf2f(__ldg(wv + i + kHalf)),
                         bf2f(__ldg(wv + i + kHalf + 1)))
           : make_float4(1.f, 1.f, 1.f, 1.f);
  }
  __syncthreads();

  const long long w = (long long)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int T = c.B * c.n;
  const int Htot = c.Hq + 2 * c.Hkv;
  const int NC = (Htot + kUnitHeads - 1) / kUnitHeads;  // units per token
  const long long U = (long long)T * NC;
  const long long u0 = w * per_warp;
  if (u0 >= U) return;
  const int n_units = (int)(U - u0 < per_warp ? U - u0 : (long long)per_warp);
  const int t_first = (int)(u0 / NC), c_first = (int)(u0 % NC);
  const int t_last = (int)((u0 + n_units - 1) / NC);
  const bool rope = c.rope_theta > 0.f;
  const float kTurnToRad = 6.28318530717958647692f / 4294967296.0f;  // 2 pi / 2^32

  // token metadata, lane j holding token t_base + j: position, cache page
  // (-1: no cache write) and slot.  Side effects (error status, kv_pos) are
  // taken by the warp holding the token's first unit.
  int t_base = t_first, m_pos = 0, m_page = -1, m_slot = 0;
  auto load_meta = [&]() {
    const int tt = t_base + lane;
    m_pos = 0;
    m_page = -1;
    m_slot = 0;
    if (tt > t_last) return;
    const bool owner = (long long)tt * NC >= u0;
    if (c.positions && (rope || c.kv_pos)) m_pos = __ldg(c.positions + tt);
    const int wp = c.write_pos ? __ldg(c.write_pos + tt) : -1;
    if (wp < 0) return;
    if ((long long)wp >= (long long)c.max_pages * c.S) {
      if (owner) atomicCAS(&c.hdr->status, 0, kErrBadLength);
      return;
    }
    const int pg = __ldg(c.page_table + (size_t)(tt / c.n) * c.max_pages + wp / c.S);
    if (pg < 0 || pg >= c.num_pages) {
      if (owner) atomicCAS(&c.hdr->status, 0, kErrPageOob);
      return;
    }
    m_page = pg;
    m_slot = wp % c.S;
    if (c.kv_pos && owner) c.kv_pos[(size_t)pg * c.S + m_slot] = m_pos;
  };
  load_meta();

  // state of the token being processed
  int cur_t = -1, page = -1, slot = 0;
  // cosines, sines and negated sines of this lane's pairs i, i + 1 (word k)
  float2 cs[kWords], sn[kWords], nsn[kWords];
  auto enter_token = [&](int t) {
    if (t - t_base >= 32) {
      t_base = t;
      load_meta();
    }
    const int pos = __shfl_sync(0xffffffffu, m_pos, t - t_base);
    page = __shfl_sync(0xffffffffu, m_page, t - t_base);
    slot = __shfl_sync(0xffffffffu, m_slot, t - t_base);
    cur_t = t;
#pragma unroll
    for (int kk = 0; kk < kWords; ++kk) {
      float c2[2] = {1.f, 1.f}, s2[2] = {0.f, 0.f};
      if (rope) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const unsigned long long ph =
              (unsigned long long)(long long)pos * c.rope_turns[8 * jl + 2 * kk + e];
          const float red = (float)(int)(unsigned)(ph >> 32) * kTurnToRad;  // in [-pi, pi)
          __sincosf(red, &s2[e], &c2[e]);  // |red| <= pi: the fast form is accurate here
        }
      }
      cs[kk] = make_float2(c2[0], c2[1]);
      sn[kk] = make_float2(s2[0], s2[1]);
      nsn[kk] = make_float2(-s2[0], -s2[1]);
    }
  };

  // load iterator (lt, lc) and process iterator (t, ci) over the warp's units
  int lt = t_first, lc = c_first, t = t_first, ci = c_first;
  const uint16_t* const src = c.qkv + 8 * jl;
  auto load_unit = [&](uint4 (&r)[kPasses][2]) {
#pragma unroll
    for (int g = 0; g < kPasses; ++g) {
      const int h = kUnitHeads * lc + g * kHpp + hs;
      if (h < Htot) {
        const uint16_t* a = src + ((size_t)lt * Htot + h) * HD;
        r[g][0] = __ldg(reinterpret_cast<const uint4*>(a));
        r[g][1] = __ldg(reinterpret_cast<const uint4*>(a + kHalf));
      }
    }
    if (++lc == NC) {
      lc = 0;
      ++lt;
    }
  };
  auto process_unit = [&](const uint4 (&r)[kPasses][2]) {
    if (t != cur_t) enter_token(t);
    // the heads' sums of squares, their reductions over each head's lanes
    // interleaved (every lane takes part in the shuffles; values heads and
    // heads past the row ignore the result)
    float ss[kPasses];
#pragma unroll
    for (int g = 0; g < kPasses; ++g) {
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int kk = 0; kk < kWords; ++kk) {
        const float2 x0 = unpack2(word4(r[g][0], kk)), x1 = unpack2(word4(r[g][1], kk));
        s2 = ffma2(x0, x0, s2);
        s2 = ffma2(x1, x1, s2);
      }
      ss[g] = s2.x + s2.y;
    }
#pragma unroll
    for (int o = kL / 2; o > 0; o >>= 1)
#pragma unroll
      for (int g = 0; g < kPasses; ++g) ss[g] += __shfl_xor_sync(0xffffffffu, ss[g], o);
#pragma unroll
    for (int g = 0; g < kPasses; ++g) {
      const int h = kUnitHeads * ci + g * kHpp + hs;
      if (kUnitHeads * ci + g * kHpp >= Htot) break;  // warp-uniform
      const int kd = h < c.Hq ? 0 : (h < c.Hq + c.Hkv ? 1 : 2);  // q, k, v
      const bool normed = kd == 0 ? has_qw : (kd == 1 && has_kw);
      uint4 o0 = r[g][0], o1 = r[g][1];  // values pass through as bits
      if (kd != 2) {
        // x[hf][k]: elements (i, i + 1) of half hf, word k
        float2 x[2][kWords];
#pragma unroll
        for (int kk = 0; kk < kWords; ++kk) {
          x[0][kk] = unpack2(word4(r[g][0], kk));
          x[1][kk] = unpack2(word4(r[g][1], kk));
        }
        if (normed) {
          const float rs = rsqrtf(ss[g] * (1.0f / HD) + c.eps);
          const float2 r2 = make_float2(rs, rs);
          const float4* wl = &s_w[kd][jl];
#pragma unroll
          for (int kk = 0; kk < kWords; ++kk) {
            const float4 wv = wl[kk * kL];
            x[0][kk] = fmul2(fmul2(x[0][kk], r2), make_float2(wv.x, wv.y));
            x[1][kk] = fmul2(fmul2(x[1][kk], r2), make_float2(wv.z, wv.w));
          }
        }
        if (rope) {
#pragma unroll
          for (int kk = 0; kk < kWords; ++kk) {
            // (a, b) -> (a cos - b sin, b cos + a sin), a in the first half
            const float2 a0 = x[0][kk], b0 = x[1][kk];
            x[0][kk] = ffma2(b0, nsn[kk], fmul2(a0, cs[kk]));
            x[1][kk] = ffma2(a0, sn[kk], fmul2(b0, cs[kk]));
          }
        }
        o0 = make_uint4(pack_bf16(x[0][0].x, x[0][0].y), pack_bf16(x[0][1].x, x[0][1].y),
                        pack_bf16(x[0][2].x, x[0][2].y), pack_bf16(x[0][3].x, x[0][3].y));
        o1 = make_uint4(pack_bf16(x[1][0].x, x[1][0].y), pack_bf16(x[1][1].x, x[1][1].y),
                        pack_bf16(x[1][2].x, x[1][2].y), pack_bf16(x[1][3].x, x[1][3].y));
      }
      if (h < Htot) {
        uint16_t* dst;
        int gh;
        if (kd == 0) {
          gh = h;
          dst = c.q_out + ((size_t)t * c.Hq + gh) * HD;
        } else {
          gh = kd == 1 ? h - c.Hq : h - c.Hq - c.Hkv;
          dst = (kd == 1 ? c.k_out : c.v_out) + ((size_t)t * c.Hkv + gh) * HD;
        }
        dst += 8 * jl;
        *reinterpret_cast<uint4*>(dst) = o0;
        *reinterpret_cast<uint4*>(dst + kHalf) = o1;
        if (kd != 0 && page >= 0) {
          uint16_t* cache = (kd == 1 ? c.k_pool : c.v_pool) +
                            (((size_t)page * c.Hkv + gh) * c.S + slot) * HD + 8 * jl;
          *reinterpret_cast<uint4*>(cache) = o0;
          *reinterpret_cast<uint4*>(cache + kHalf) = o1;
        }
      }
    }
    if (++ci == NC) {
      ci = 0;
      ++t;
    }
  };
  // two units in flight: unit i + 1 is loaded while unit i is processed
  uint4 ra[kPasses][2], rb[kPasses][2];
  load_unit(ra);
  for (int i = 0; i < n_units; i += 2) {
    if (i + 1 < n_units) load_unit(rb);
    process_unit(ra);
    if (i + 1 >= n_units) break;
    if (i + 2 < n_units) load_unit(ra);
    process_unit(rb);
  }
}

}  // namespace

cudaError_t launch_qkv_post(const QkvPostParams& c, int head_dim, int n_sms, cudaStream_t stream) {
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
  // units of kUnitHeads heads of a token, cut into equal ranges over the
  // resident warps
  const long long units = (long long)c.B * c.n * ((c.Hq + 2 * c.Hkv + kUnitHeads - 1) / kUnitHeads);
  const long long resident_warps = (long long)(n_sms > 0 ? n_sms : 1) * per_sm * (kThreadsQP / 32);
  const long long per_warp = (units + resident_warps - 1) / resident_warps;
  if (per_warp > (1ll << 30)) return cudaErrorInvalidValue;
  const long long warps = (units + per_warp - 1) / per_warp;
  const long long blocks = (warps + kThreadsQP / 32 - 1) / (kThreadsQP / 32);
  if (head_dim == 128)
    qkv_post_kernel<128><<<(unsigned)blocks, kThreadsQP, 0, stream>>>(c, (int)per_warp);
  else
    qkv_post_kernel<64><<<(unsigned)blocks, kThreadsQP, 0, stream>>>(c, (int)per_warp);
  return cudaGetLastError();
}

}  // namespace bca
