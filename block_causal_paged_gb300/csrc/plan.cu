// Plan kernel, one CTA, launched before every attention kernel.
//
// It resets the work counter the attention CTAs take items from.  For a
// decode step it also does the split-KV planning from the prefix lengths
// (device data, so the host never synchronizes):
//   - chooses the chunk size CH (KV tiles per work item) so that there are
//     about `waves` items per CTA, never fewer than ch_min tiles per chunk,
//     and the split-KV partials and the item list fit the workspace;
//   - orders the sequences longest first (bitonic sort in shared memory) so
//     that the dynamic schedule hands out the largest items first;
//   - writes the item list {b, g, rb, split slot}{t0, t1, P, -} and, for each
//     sequence, the first split-KV slot of its chunks (read by the combine).
#include <cstdint>

#include "bca_internal.h"

namespace bca {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanSortMax = 2048;  // larger batches keep their natural order
constexpr int kErrBadLength = -17;
constexpr int kErrWorkspace = -4;

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int plan_prefix(const AttnParams& p, int b, int* bad) {
  const int P = __ldg(p.lens + b);
  if (P < 0 || P % p.Dblk != 0 || (long long)P + p.Dblk > (long long)p.max_pages * p.S) {
    *bad = 1;
    return 0;  // treated as an empty prefix, reported in the status word
  }
  return P;
}

__device__ __forceinline__ int plan_tiles(const AttnParams& p, int P) {
  return cdiv(P, kTileKeys) + cdiv(p.Dblk, kTileKeys);
}

// Sum over the block (every thread gets the result).
__device__ long long block_sum(long long v, long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  long long t = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  __syncthreads();
  return t;
}

// Exclusive prefix sum over the block in thread order; *total gets the sum.
__device__ long long block_excl_scan(long long v, long long* red, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) red[warp] = x;
  __syncthreads();
  long long before = 0, all = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) before += red[w];
    all += red[w];
  }
  __syncthreads();
  *total = all;
  return before + x - v;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ AttnParams p,
                                                            int attn_grid) {
  __shared__ int s_nt[kPlanSortMax];
  __shared__ int s_ord[kPlanSortMax];
  __shared__ int s_base[kPlanSortMax + 1];
  __shared__ long long s_red[32];
  const int tid = threadIdx.x;
  const int nth = blockDim.x;
  if (tid == 0) p.hdr->work_next = 0;
  if (p.mode != kModeDecode) return;

  const int B = p.B;
  const int per_seq = p.Hkv * p.n_rb;
  const bool sorted = B <= kPlanSortMax;

  // tiles per sequence and in total
  int bad = 0;
  long long tot = 0;
  for (int b = tid; b < B; b += nth) {
    const int nt = plan_tiles(p, plan_prefix(p, b, &bad));
    if (sorted) s_nt[b] = nt;
    tot += nt;
  }
  tot = block_sum(tot, s_red) * per_seq;
  if (__syncthreads_or(bad) && tid == 0) atomicCAS(&p.hdr->status, 0, kErrBadLength);

  auto tiles_of = [&](int b) {
    if (sorted) return s_nt[b];
    int dummy = 0;
    return plan_tiles(p, plan_prefix(p, b, &dummy));
  };

  // chunk size: ~waves items per CTA, at least ch_min tiles, fits the workspace
  const long long target = (long long)attn_grid * (p.waves > 0 ? p.waves : 1);
  long long ch = (tot + target - 1) / target;
  if (ch < p.ch_min) ch = p.ch_min;
  if (ch < 1) ch = 1;
  for (int guard = 0; guard < 40; ++guard) {
    long long ns = 0, ni = 0;
    for (int b = tid; b < B; b += nth) {
      const long long nch = (tiles_of(b) + ch - 1) / ch;
      ni += nch;
      if (nch > 1) ns += nch;
    }
    ns = block_sum(ns, s_red) * per_seq;
    ni = block_sum(ni, s_red) * per_seq;
    if (ns <= p.split_cap && ni <= p.items_cap) break;
    ch *= 2;
  }
  const int CH = (int)(ch < (1ll << 30) ? ch : (1ll << 30));

  // longest sequences first (ties by index)
  if (sorted) {
    int n2 = 1;
    while (n2 < B) n2 <<= 1;
    for (int i = tid; i < n2; i += nth) s_ord[i] = i;
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < n2; i += nth) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const int a = s_ord[i], c = s_ord[ixj];
            const int ka = a < B ? s_nt[a] : -1, kc = c < B ? s_nt[c] : -1;
            const bool a_first = ka > kc || (ka == kc && a < c);
            const bool up = (i & k) == 0;
            if (up ? !a_first : a_first) {
              s_ord[i] = c;
              s_ord[ixj] = a;
            }
          }
        }
        __syncthreads();
      }
    }
  }
  auto seq_at = [&](int i) { return sorted ? s_ord[i] : i; };

  // split-KV slots: in natural sequence order, per-thread contiguous segments
  const int seg = (B + nth - 1) / nth;
  const int lo = min(B, tid * seg), hi = min(B, lo + seg);
  long long local = 0, total = 0;
  for (int b = lo; b < hi; ++b) {
    const int nch = cdiv(tiles_of(b), CH);
    if (nch > 1) local += (long long)nch * per_seq;
  }
  long long off = block_excl_scan(local, s_red, &total);
  for (int b = lo; b < hi; ++b) {
    p.split_base[b] = (int)off;
    const int nch = cdiv(tiles_of(b), CH);
    if (nch > 1) off += (long long)nch * per_seq;
  }
  if (total > p.split_cap && tid == 0) atomicCAS(&p.hdr->status, 0, kErrWorkspace);

  // item bases in schedule order
  local = 0;
  for (int i = lo; i < hi; ++i) local += (long long)cdiv(tiles_of(seq_at(i)), CH) * per_seq;
  off = block_excl_scan(local, s_red, &total);
  const int n_items = (int)(total < p.items_cap ? total : p.items_cap);
  if (sorted) {
    for (int i = lo; i < hi; ++i) {
      s_base[i] = (int)off;
      off += (long long)cdiv(tiles_of(seq_at(i)), CH) * per_seq;
    }
    if (tid == 0) s_base[B] = (int)total;
  }
  __syncthreads();  // split_base (global) and s_base visible to the block

  auto write_item = [&](int idx, int b, int l) {
    const int nt = tiles_of(b);
    const int nch = cdiv(nt, CH);
    const int c = l / per_seq, rest = l % per_seq;
    const int g = rest / p.n_rb, rb = rest % p.n_rb;
    const int t0 = c * CH, t1 = min(nt, t0 + CH);
    const int split = nch > 1 ? p.split_base[b] + (g * p.n_rb + rb) * nch + c : -1;
    int dummy = 0;
    const int P = plan_prefix(p, b, &dummy);
    p.items[2 * idx] = make_int4(b, g, rb, split);
    p.items[2 * idx + 1] = make_int4(t0, t1, P, 0);
  };
  if (sorted) {
    // one thread per item: find its sequence by binary search over the bases
    for (int idx = tid; idx < n_items; idx += nth) {
      int a = 0, z = B - 1;
      while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (s_base[mid] <= idx) a = mid;
        else z = mid - 1;
      }
      write_item(idx, seq_at(a), idx - s_base[a]);
    }
  } else {
    long long idx = off;  // this thread's first item (natural order)
    for (int i = lo; i < hi; ++i) {
      const int b = seq_at(i);
      const int n = cdiv(tiles_of(b), CH) * per_seq;
      for (int l = 0; l < n && idx < n_items; ++l, ++idx) write_item((int)idx, b, l);
    }
  }
  if (tid == 0) {
    p.hdr->chunk_tiles = CH;
    p.hdr->n_items = n_items;
    if (total > p.items_cap) atomicCAS(&p.hdr->status, 0, kErrWorkspace);
  }
}

}  // namespace

cudaError_t launch_plan(const AttnParams& p, int attn_grid, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(p, attn_grid);
  return cudaGetLastError();
}

}  // namespace bca
