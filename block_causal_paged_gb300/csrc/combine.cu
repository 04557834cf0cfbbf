// Decode epilogue kernel: the KV commit of the step's blocks and the split-KV
// combine.
//
// Commit: the blocks' rows P .. P+D-1 are bit-copied from the dense block K/V
// into their pages ("Inference for Interpretable Text-Diffusion Models", "KV
// Cache": a final pass commits the block; "Paged Attention": position p lives
// in page page_table[b][p / S], slot p % S); a warp copies two token rows at
// a time with 16-byte accesses.  It runs after the attention kernel, which
// reads only rows below P, and before anything later in the stream reads the
// pages.
//
// A long prefix is split into chunks that different CTAs attend to (each
// chunk is an online softmax over its keys), so every row
// of a split group has, per chunk c, a running maximum m_c (log2 units), a sum
// l_c and an unnormalised output O_c.  Merging them is the same rescaling the
// online softmax does between tiles:
//     M = max_c m_c,  O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
//
// Work unit: one split group (its first slot in the slot table) x 32 head-dim
// columns; 256 threads, one per row (two M-tiles of 128), so every load of a
// partial is 512 contiguous bytes per warp.  The (max, sum) pairs and partial
// outputs of kBatch chunks are loaded together and merged online (running
// maximum, rescaled accumulator), so a unit costs about one memory round trip
// per kBatch chunks.  Two CTAs per SM; the combine CTAs read the slot table
// in coalesced chunks and keep only the first slot of each group.  Launched
// with programmatic dependent launch: the grid may start while the attention
// kernel drains, and waits for it to finish.
#include <cstdint>

#include "bca_internal.h"

namespace bca {
namespace {

constexpr int kCombineThreads = 256;  // rows of a split group
constexpr int kCols = 32;             // head-dim columns per work unit
constexpr int kBatch = 2;             // chunks whose loads are in flight together

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Commit of the blocks' K/V by CTAs first_cta .. gridDim.x-1: their warp w
// copies token rows w, w + W, ... two at a time.  Both rows' K/V pieces are
// loaded first (they do not depend on the destination), then both prefix
// lengths, then both page-table entries, so that a pair of rows costs about
// one memory round trip instead of three per row.
template <int HD>
__device__ __forceinline__ void commit_rows(const AttnParams& p, int first_cta) {
  constexpr int kPerHead = HD / 8;  // 16-byte pieces per head row
  constexpr int kLane = 4;          // pieces per lane and row held in registers
  const int lane = threadIdx.x & 31;
  const int per_row = p.Hkv * kPerHead;
  const long long rows = (long long)p.B * p.Dblk;
  const long long warp = ((long long)(blockIdx.x - first_cta) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = ((long long)(gridDim.x - first_cta) * blockDim.x) >> 5;
  const uint4* ks = reinterpret_cast<const uint4*>(p.k_dense);
  const uint4* vs = reinterpret_cast<const uint4*>(p.v_dense);
  uint4* kd = reinterpret_cast<uint4*>(p.commit_k);
  uint4* vd = reinterpret_cast<uint4*>(p.commit_v);
  // destination piece of piece i (head i / kPerHead) of a row at (page, slot)
  auto dst_of = [&](int page, int slot, int i) {
    return (((size_t)page * p.Hkv + i / kPerHead) * p.S + slot) * kPerHead + i % kPerHead;
  };
  for (long long row0 = warp; row0 < rows; row0 += 2 * n_warps) {
    const long long rr[2] = {row0, row0 + n_warps};
    uint4 kv[2][kLane], vv[2][kLane];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int u = 0; u < kLane; ++u) {
        const int i = 32 * u + lane;
        if (rr[j] < rows && i < per_row) {
          kv[j][u] = __ldg(ks + rr[j] * per_row + i);
          vv[j][u] = __ldg(vs + rr[j] * per_row + i);
        }
      }
    int pos[2], page[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      pos[j] = -1;
      if (rr[j] < rows) {
        const int b = (int)(rr[j] / p.Dblk), t = (int)(rr[j] % p.Dblk);
        const int P = __ldg(p.lens + b);
        // a bad prefix length is reported by the plan kernel
        if (P >= 0 && (p.causal || P % p.Dblk == 0) &&
            (long long)P + p.Dblk <= (long long)p.max_pages * p.S)
          pos[j] = P + t;
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      page[j] = -1;
      if (pos[j] >= 0) {
        const int b = (int)(rr[j] / p.Dblk);
        page[j] = __ldg(p.page_table + (size_t)b * p.max_pages + pos[j] / p.S);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (pos[j] < 0) continue;
      if (page[j] < 0 || page[j] >= p.num_pages) {
        if (lane == 0) atomicCAS(&p.hdr->status, 0, -16);  // page id outside the pool
        continue;
      }
      const int slot = pos[j] % p.S;
#pragma unroll
      for (int u = 0; u < kLane; ++u) {
        const int i = 32 * u + lane;
        if (i < per_row) {
          const size_t dst = dst_of(page[j], slot, i);
          kd[dst] = kv[j][u];
          vd[dst] = vv[j][u];
        }
      }
      // rows wider than the registers' share (more than 8 KV heads at d = 128)
      for (int i = 32 * kLane + lane; i < per_row; i += 32) {
        const size_t dst = dst_of(page[j], slot, i);
        kd[dst] = __ldg(ks + rr[j] * per_row + i);
        vd[dst] = __ldg(vs + rr[j] * per_row + i);
      }
    }
  }
}

template <int HD>
__global__ void __launch_bounds__(kCombineThreads, 2) combine_kernel(const __grid_constant__ AttnParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kQ = HD / kCols;
  const int n_slots = *reinterpret_cast<volatile int*>(&p.hdr->n_split_slots);
  // the two jobs are latency-bound: when both exist, half the CTAs do each
  const bool commit = p.commit_k != nullptr, combine = n_slots > 0;
  const int n_comb = combine ? (commit ? (int)gridDim.x / 2 : (int)gridDim.x) : 0;
  if (commit && (int)blockIdx.x >= n_comb) {
    commit_rows<HD>(p, n_comb);
    return;
  }
  __shared__ int s_first[kCombineThreads];  // group starts of the current table chunk
  __shared__ int s_wcnt[kCombineThreads / 32];
  const int R = threadIdx.x, lane = R & 31, warp = R >> 5;
  const int m = R / kRowsPerMTile, r = R % kRowsPerMTile;
  // The slot table, 256 entries at a time: every combine CTA reads the chunk
  // (one coalesced load), keeps the group starts, and takes its share of the
  // (group, column slice) units.
  for (int s0 = 0; s0 < n_slots; s0 += kCombineThreads) {
    const int my_s = s0 + R;
    const bool first = my_s < n_slots && p.slot_info[my_s].z == my_s;
    const unsigned bal = __ballot_sync(0xffffffffu, first);
    __syncthreads();  // the previous chunk's list is no longer read
    if (lane == 0) s_wcnt[warp] = __popc(bal);
    __syncthreads();
    int before = 0, n_groups = 0;
    for (int w = 0; w < kCombineThreads / 32; ++w) {
      before += w < warp ? s_wcnt[w] : 0;
      n_groups += s_wcnt[w];
    }
    if (first) s_first[before + __popc(bal & ((1u << lane) - 1))] = my_s;
    __syncthreads();
    for (int u = blockIdx.x; u < n_groups * kQ; u += n_comb) {
      const int s = s_first[u / kQ], q = u % kQ;
      const int4 info = p.slot_info[s];
      const int b = info.x, g = info.y >> 16, rb = info.y & 0xffff, nch = info.w;
      const int tok = rb * 2 * p.tpm + m * p.tpm + r / p.hpr;
      if (r >= p.hpr * p.tpm || tok >= p.Dblk) continue;
      const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
      const float4* po = reinterpret_cast<const float4*>(p.part_o);
      // online merge, kBatch chunks per round with all their loads in flight
      float M = -INFINITY, den = 0.f;
      float acc[kCols];
  #pragma unroll
      for (int k = 0; k < kCols; ++k) acc[k] = 0.f;
      for (int c0 = 0; c0 < nch; c0 += kBatch) {
        float2 mlv[kBatch];
        float4 v[kBatch][kCols / 4];
  #pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (c0 + k < nch) {
            const size_t slot = (size_t)(s + c0 + k);
            mlv[k] = ml[slot * 256 + R];
            const float4* src = po + (slot * (HD / 4) + q * (kCols / 4)) * 256 + R;
  #pragma unroll
            for (int k4 = 0; k4 < kCols / 4; ++k4) v[k][k4] = src[(size_t)k4 * 256];
          } else {
            mlv[k] = make_float2(-INFINITY, 0.f);
          }
        }
        float Mn = M;
  #pragma unroll
        for (int k = 0; k < kBatch; ++k) Mn = fmaxf(Mn, mlv[k].x);
        if (Mn == -INFINITY) continue;  // no key seen yet
        const float a = M == -INFINITY ? 0.f : ex2f(M - Mn);
        den *= a;
  #pragma unroll
        for (int k = 0; k < kCols; ++k) acc[k] *= a;
  #pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (c0 + k >= nch) break;
          const float w = mlv[k].x == -INFINITY ? 0.f : ex2f(mlv[k].x - Mn);
          den += w * mlv[k].y;
  #pragma unroll
          for (int k4 = 0; k4 < kCols / 4; ++k4) {
            acc[4 * k4 + 0] += w * v[k][k4].x;
            acc[4 * k4 + 1] += w * v[k][k4].y;
            acc[4 * k4 + 2] += w * v[k][k4].z;
            acc[4 * k4 + 3] += w * v[k][k4].w;
          }
        }
        M = Mn;
      }
      const float inv = den > 0.f ? 1.0f / den : 0.f;
      uint16_t* dst = p.out +
                      ((size_t)(b * p.Dblk + tok) * p.Hq + g * p.G + (r % p.hpr)) * HD + q * kCols;
  #pragma unroll
      for (int k = 0; k < kCols; k += 8) {
        uint4 o;
        o.x = pack2(acc[k + 0] * inv, acc[k + 1] * inv);
        o.y = pack2(acc[k + 2] * inv, acc[k + 3] * inv);
        o.z = pack2(acc[k + 4] * inv, acc[k + 5] * inv);
        o.w = pack2(acc[k + 6] * inv, acc[k + 7] * inv);
        *reinterpret_cast<uint4*>(dst + k) = o;
      }
    }
  }
}

}  // namespace

cudaError_t launch_decode_combine(const AttnParams& p, int head_dim, int n_sms,
                                  cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (n_sms > 0 ? n_sms : 1));  // two CTAs per SM
  cfg.blockDim = dim3(kCombineThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, combine_kernel<128>, p);
  return cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
}

}  // namespace bca
