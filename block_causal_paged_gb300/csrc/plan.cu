// Plan kernel, one CTA, launched before every attention kernel.
//
// It resets the work counter the attention CTAs take items from.  For a
// decode step it also does the split-KV planning from the prefix lengths
// (device data, so the host never synchronizes):
//   - chooses the chunk size CH (KV tiles per work item) so that there are
//     about `waves` items per CTA, never fewer than ch_min tiles per chunk,
//     and the split-KV partials and the item list fit the workspace;
//   - orders the sequences longest first (a rank sort in shared memory: each
//     thread counts the sequences that go before its own) so that the dynamic
//     schedule hands out the largest items first;
//   - writes the item list {b, g, rb, split slot}{t0, t1, P, chunks}, for each
//     sequence the first split-KV slot of its chunks, and for each split slot
//     {b, g << 16 | rb, first slot of its group, chunks} (read by the combine).
// The block is sized to the batch (a multiple of 32 threads, at most 1024),
// so small batches pay for few warps at every barrier.
//
// For a multicanvas step the plan is a summary of the arena instead: every
// work item of a sequence (one per row block and KV head) classifies the
// same arena tiles against its own rows, so the smallest and largest key
// position of each tile are found once here rather than once per item.
#include <algorithm>
#include <climits>
#include <cstdint>

#include "bca_internal.h"

namespace bca {
namespace {

constexpr int kPlanThreads = 1024;  // upper bound; the launch uses fewer for small batches
constexpr int kPlanSortMax = 2048;  // larger batches keep their natural order
constexpr int kErrBadLength = -17;
constexpr int kErrWorkspace = -4;
constexpr int kErrPageOob = -16;
constexpr int kSummaryThreads = 256;

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int plan_prefix(const AttnParams& p, int b, int* bad) {
  const int P = __ldg(p.lens + b);
  if (P < 0 || (!p.causal && P % p.Dblk != 0) ||
      (long long)P + p.Dblk > (long long)p.max_pages * p.S) {
    *bad = 1;
    return 0;  // treated as an empty prefix, reported in the status word
  }
  return P;
}

__device__ __forceinline__ int plan_tiles(const AttnParams& p, int P) {
  return cdiv(P, kTileKeys) + cdiv(p.Dblk, kTileKeys);
}

// Sums of two values over the block (every thread gets both).
__device__ longlong2 block_sum2(long long a, long long b, longlong2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  __syncthreads();
  if (lane == 0) red[warp] = make_longlong2(a, b);
  __syncthreads();
  longlong2 t = make_longlong2(0, 0);
  for (int w = 0; w < nw; ++w) {
    t.x += red[w].x;
    t.y += red[w].y;
  }
  return t;
}

// Exclusive prefix sums of two values in thread order; *total gets the sums.
__device__ longlong2 block_scan2(long long a, long long b, longlong2* red, longlong2* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long x = a, y = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long xo = __shfl_up_sync(0xffffffffu, x, o);
    const long long yo = __shfl_up_sync(0xffffffffu, y, o);
    if (lane >= o) {
      x += xo;
      y += yo;
    }
  }
  __syncthreads();
  if (lane == 31) red[warp] = make_longlong2(x, y);
  __syncthreads();
  longlong2 before = make_longlong2(0, 0), all = make_longlong2(0, 0);
  for (int w = 0; w < nw; ++w) {
    if (w < warp) {
      before.x += red[w].x;
      before.y += red[w].y;
    }
    all.x += red[w].x;
    all.y += red[w].y;
  }
  *total = all;
  return make_longlong2(before.x + x - a, before.y + y - b);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ AttnParams p,
                                                            int attn_grid) {
  __shared__ int s_nt[kPlanSortMax];     // KV tiles per sequence
  __shared__ int s_P[kPlanSortMax];      // prefix length per sequence
  __shared__ int s_ord[kPlanSortMax];    // schedule position -> sequence
  __shared__ int s_split[kPlanSortMax];  // first split slot per sequence
  __shared__ int s_base[kPlanSortMax];   // first item of each schedule position
  __shared__ longlong2 s_red[32];
  const int tid = threadIdx.x;
  const int nth = blockDim.x;
  // Programmatic dependent launch: the attention kernel may start its
  // prologue now; everything it reads from here is behind its own wait for
  // this grid.  This grid in turn waits for the work before it in the stream
  // (which may still be reading the workspace) before touching anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    p.hdr->work_next = 0;
    p.hdr->exit_count = 0;
  }
  if (p.mode != kModeDecode) return;

  const int B = p.B;
  const int per_seq = p.Hkv * p.n_rb;
  const bool small = B <= kPlanSortMax;  // tables fit in shared memory; sort

  // 1. prefix lengths and tiles per sequence
  long long tot = 0, bad = 0;
  for (int b = tid; b < B; b += nth) {
    int bb = 0;
    const int P = plan_prefix(p, b, &bb);
    const int nt = plan_tiles(p, P);
    if (small) {
      s_nt[b] = nt;
      s_P[b] = P;
    }
    tot += nt;
    bad |= bb;
  }
  const longlong2 t1 = block_sum2(tot, bad, s_red);
  tot = t1.x * per_seq;
  if (t1.y && tid == 0) atomicCAS(&p.hdr->status, 0, kErrBadLength);
  auto tiles_of = [&](int b) {
    if (small) return s_nt[b];
    int dummy = 0;
    return plan_tiles(p, plan_prefix(p, b, &dummy));
  };
  auto prefix_of = [&](int b) {
    if (small) return s_P[b];
    int dummy = 0;
    return plan_prefix(p, b, &dummy);
  };

  // 2. chunk size: ~waves items per CTA, at least ch_min tiles, fits the workspace
  const long long target = (long long)attn_grid * (p.waves > 0 ? p.waves : 1);
  long long ch = (tot + target - 1) / target;
  if (ch < p.ch_min) ch = p.ch_min;
  if (ch < 1) ch = 1;
  for (int guard = 0; guard < 40; ++guard) {
    long long ns = 0, ni = 0;
    const int ch32 = (int)(ch < (1ll << 30) ? ch : (1ll << 30));  // tiles per sequence < 2^30
    for (int b = tid; b < B; b += nth) {
      const int nch = cdiv(tiles_of(b), ch32);
      ni += nch;
      if (nch > 1) ns += nch;
    }
    const longlong2 t2 = block_sum2(ns, ni, s_red);
    if (t2.x * per_seq <= p.split_cap && t2.y * per_seq <= p.items_cap) break;
    ch *= 2;
  }
  const int CH = (int)(ch < (1ll << 30) ? ch : (1ll << 30));

  // 3. schedule order, longest first (ties by index): rank of each sequence
  if (small) {
    for (int i = tid; i < B; i += nth) {
      const int ki = s_nt[i];
      int rank = 0;
      for (int j = 0; j < B; ++j) {
        const int kj = s_nt[j];
        rank += (kj > ki) | ((kj == ki) & (j < i));
      }
      s_ord[rank] = i;
    }
    __syncthreads();
  }
  auto seq_at = [&](int i) { return small ? s_ord[i] : i; };

  // 4. split slots (sequence order) and item bases (schedule order), one scan
  //    over per-thread contiguous segments of positions
  const int seg = (B + nth - 1) / nth;
  const int lo = min(B, tid * seg), hi = min(B, lo + seg);
  long long ls = 0, li = 0;
  for (int i = lo; i < hi; ++i) {
    const int nch = cdiv(tiles_of(i), CH);
    if (nch > 1) ls += (long long)nch * per_seq;
    li += (long long)cdiv(tiles_of(seq_at(i)), CH) * per_seq;
  }
  longlong2 all;
  const longlong2 off = block_scan2(ls, li, s_red, &all);
  long long so = off.x, ib = off.y;
  for (int b = lo; b < hi; ++b) {
    if (small) {
      s_split[b] = (int)so;
      s_base[b] = (int)ib;  // position b of the schedule
    }
    p.split_base[b] = (int)so;
    const int nch = cdiv(tiles_of(b), CH);
    if (nch > 1) so += (long long)nch * per_seq;
    ib += (long long)cdiv(tiles_of(seq_at(b)), CH) * per_seq;
  }
  const int n_items = (int)(all.y < p.items_cap ? all.y : p.items_cap);
  __syncthreads();  // split bases visible to the block

  // 5. items
  auto write_item = [&](int io, int b, int l) {
    const int nt = tiles_of(b), P = prefix_of(b);
    const int nch = cdiv(nt, CH);
    const int c = l / per_seq, rest = l % per_seq;
    const int g = rest / p.n_rb, rb = rest % p.n_rb;
    const int t0 = c * CH, t1e = min(nt, t0 + CH);
    const int split =
        nch > 1 ? (small ? s_split[b] : p.split_base[b]) + (g * p.n_rb + rb) * nch + c : -1;
    p.items[2 * io] = make_int4(b, g, rb, split);
    p.items[2 * io + 1] = make_int4(t0, t1e, P, nch);
    if (split >= 0 && split < p.split_cap)
      p.slot_info[split] = make_int4(b, (g << 16) | rb, split - c, nch);
  };
  if (small) {
    // one item per thread: its schedule position by binary search over the bases
    for (int io = tid; io < n_items; io += nth) {
      int a = 0, z = B - 1;
      while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (s_base[mid] <= io) a = mid;
        else z = mid - 1;
      }
      write_item(io, s_ord[a], io - s_base[a]);
    }
  } else {
    // each thread writes the items of the sequences at its positions
    long long io = off.y;
    for (int i = lo; i < hi; ++i) {
      const int b = seq_at(i);
      const int n = cdiv(tiles_of(b), CH) * per_seq;
      for (int l = 0; l < n && io < n_items; ++l, ++io) write_item((int)io, b, l);
    }
  }
  if (tid == 0) {
    p.hdr->chunk_tiles = CH;
    p.hdr->n_items = n_items;
    p.hdr->n_split_slots = (int)(all.x < p.split_cap ? all.x : p.split_cap);
    if (all.x > p.split_cap || all.y > p.items_cap) atomicCAS(&p.hdr->status, 0, kErrWorkspace);
  }
}

// Multicanvas: tile_kv[b * n_at_max + a] = {min, max} of the key positions
// kv_pos[page][slot] of arena entries 128a .. 128a+127 of sequence b (entry
// e lives in page page_table[b][e / S], slot e % S).  Entries at or past
// arena_len[b] do not count; nor do entries whose page id lies outside the
// pool, which are reported (kErrPageOob) as the attention kernel would.  A
// tile with no counted entry gets {INT_MAX, INT_MIN}, which every row skips.
// One warp per tile, four entries per lane.
__global__ void __launch_bounds__(kSummaryThreads) arena_summary_kernel(
    const __grid_constant__ AttnParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.hdr->work_next = 0;
    p.hdr->exit_count = 0;
  }
  const int lane = threadIdx.x & 31;
  const long long n = (long long)p.B * p.n_at_max;
  const long long stride = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < n; w += stride) {
    const int b = (int)(w / p.n_at_max), a = (int)(w % p.n_at_max);
    int A = __ldg(p.arena_len + b);
    if (A < 0 || (long long)A > (long long)p.max_pages * p.S) A = 0;  // reported by the attention kernel
    int kmin = INT_MAX, kmax = INT_MIN, bad = 0;
#pragma unroll
    for (int h = 0; h < kTileKeys / 32; ++h) {
      const int e = a * kTileKeys + 32 * h + lane;
      if (e < A) {
        const int page = __ldg(p.page_table + (size_t)b * p.max_pages + e / p.S);
        if (page >= 0 && page < p.num_pages) {
          const int pos = __ldg(p.kv_pos + (size_t)page * p.S + e % p.S);
          kmin = min(kmin, pos);
          kmax = max(kmax, pos);
        } else {
          bad = 1;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(&p.hdr->status, 0, kErrPageOob);
    if (lane == 0) p.tile_kv[w] = make_int2(kmin, kmax);
  }
}

}  // namespace

cudaError_t launch_plan(const AttnParams& p, int attn_grid, cudaStream_t stream) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if (p.mode == kModeMulticanvas) {
    constexpr int kWarps = kSummaryThreads / 32;
    const long long tiles = (long long)p.B * p.n_at_max;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<long long>(std::max<long long>(1, (tiles + kWarps - 1) / kWarps), 4096));
    cfg.blockDim = dim3(kSummaryThreads);
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, arena_summary_kernel, p);
  }
  int threads = p.mode == kModeDecode ? ((p.B + 31) / 32) * 32 : 32;
  threads = threads < 256 ? 256 : (threads > kPlanThreads ? kPlanThreads : threads);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, p, attn_grid);
}

}  // namespace bca
