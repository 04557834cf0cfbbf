// Page writes of K/V: the commit of a finished block (and the cache fill of a
// prefill), and the arena promotion of a multicanvas step.  Pure bit copies
// with 16-byte vector accesses; one warp moves one token row (all KV heads).
//
// "Inference for Interpretable Text-Diffusion Models", "KV Cache" step 3 (a
// final pass commits the block) and "Paged Attention" (position p lives in
// page page_table[b][p / S], slot p % S).  "Inference: Fewer, smaller
// forwards", "Advancement 11" (promotion appends at the arena end and the
// entry keeps its absolute position).
#include <cstdint>

#include "bca_internal.h"

namespace bca {
namespace {

constexpr int kErrPageOob = -16;
constexpr int kErrBadLength = -17;

__device__ __forceinline__ void record(WsHeader* hdr, int code) {
  if (hdr) atomicCAS(&hdr->status, 0, code);
}

// Copy one token row [Hkv, d] from src_row to (page, slot) of both pools.
__device__ __forceinline__ void copy_row(const uint16_t* k_src, const uint16_t* v_src,
                                         size_t src_row, uint16_t* k_pool, uint16_t* v_pool,
                                         int page, int slot, int Hkv, int d, int S, int lane) {
  const int per_head = d / 8;  // 16-byte pieces per head row
  const uint4* ks = reinterpret_cast<const uint4*>(k_src + src_row * Hkv * d);
  const uint4* vs = reinterpret_cast<const uint4*>(v_src + src_row * Hkv * d);
  uint4* kd = reinterpret_cast<uint4*>(k_pool);
  uint4* vd = reinterpret_cast<uint4*>(v_pool);
  for (int i = lane; i < Hkv * per_head; i += 32) {
    const int h = i / per_head, cc = i % per_head;
    const size_t dst = (((size_t)page * Hkv + h) * S + slot) * per_head + cc;
    const uint4 kv = __ldg(ks + i);
    const uint4 vv = __ldg(vs + i);
    kd[dst] = kv;
    vd[dst] = vv;
  }
}

__global__ void __launch_bounds__(256) commit_kernel(const __grid_constant__ CommitParams c) {
  const int lane = threadIdx.x & 31;
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long rows = (long long)c.B * c.max_rows;
  for (long long row = warp_id; row < rows; row += n_warps) {
    const int b = (int)(row / c.max_rows), t = (int)(row % c.max_rows);
    long long first, count, start;
    if (c.cu) {
      first = __ldg(c.cu + b);
      count = (long long)__ldg(c.cu + b + 1) - first;
      start = 0;
    } else {
      first = (long long)b * c.rows_per_seq;
      count = c.num_tokens;
      start = __ldg(c.start_pos + b);
    }
    if (t >= count) continue;
    const long long pos = start + t;
    if (pos < 0 || pos / c.S >= c.max_pages || first < 0) {
      if (lane == 0) record(c.hdr, kErrBadLength);
      continue;
    }
    const int page = __ldg(c.page_table + (size_t)b * c.max_pages + pos / c.S);
    if (page < 0 || page >= c.num_pages) {
      if (lane == 0) record(c.hdr, kErrPageOob);
      continue;
    }
    copy_row(c.k_src, c.v_src, (size_t)(first + t), c.k_pool, c.v_pool, page, (int)(pos % c.S),
             c.Hkv, c.d, c.S, lane);
  }
}

// One CTA per sequence: append commit rows at the arena end, record their
// positions, then advance arena_len (read by every thread before the update).
__global__ void __launch_bounds__(256) promote_kernel(const __grid_constant__ PromoteParams c) {
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  __shared__ int s_ok;
  const int A = c.arena_len[b];
  const int nc = __ldg(c.commit_count + b);
  const int n_live = c.live_count ? __ldg(c.live_count + b) : c.max_live;
  if (threadIdx.x == 0) {
    s_ok = (A >= 0 && nc >= 0 && nc <= c.max_commit &&
            (long long)A + nc <= (long long)c.max_pages * c.S && n_live >= 0 &&
            n_live <= c.max_live);
    if (!s_ok) record(c.hdr, kErrBadLength);
  }
  __syncthreads();
  if (!s_ok) return;
  for (int i = warp; i < nc; i += n_warps) {
    const int r = __ldg(c.commit_rows + (size_t)b * c.max_commit + i);
    const int e = A + i;
    const int page = __ldg(c.page_table + (size_t)b * c.max_pages + e / c.S);
    if (r < 0 || r >= n_live) {
      if (lane == 0) record(c.hdr, kErrBadLength);
      continue;
    }
    if (page < 0 || page >= c.num_pages) {
      if (lane == 0) record(c.hdr, kErrPageOob);
      continue;
    }
    copy_row(c.k_live, c.v_live, (size_t)b * c.max_live + r, c.k_pool, c.v_pool, page, e % c.S,
             c.Hkv, c.d, c.S, lane);
    if (lane == 0) {
      c.kv_pos[(size_t)page * c.S + e % c.S] =
          c.live_pos ? __ldg(c.live_pos + (size_t)b * c.max_live + r) : c.prompt_len + r;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) c.arena_len[b] = A + nc;
}

}  // namespace

cudaError_t launch_commit(const CommitParams& c, cudaStream_t stream) {
  const long long rows = (long long)c.B * c.max_rows;
  if (rows <= 0) return cudaSuccess;
  long long blocks = (rows + 7) / 8;  // 8 warps per block
  if (blocks > 4096) blocks = 4096;
  commit_kernel<<<(unsigned)blocks, 256, 0, stream>>>(c);
  return cudaGetLastError();
}

cudaError_t launch_promote(const PromoteParams& c, cudaStream_t stream) {
  if (c.B <= 0) return cudaSuccess;
  promote_kernel<<<c.B, 256, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace bca
