// Host-side input checks run before a launch when the environment sets
// BCA_DEBUG=1 ("Paged Attention": the page table used with stricter error
// checking).  Each entry point copies the lengths and page-table entries its
// kernels will use to the host (ordered on the call's stream, then waited
// for) and checks them, so that a bad request is refused with an error code
// instead of being detected, and its access skipped, on the device:
//   - lengths and positions: in range for their operation, within the
//     capacity of a sequence's page list (BCA_ERR_INVALID_ARG,
//     BCA_ERR_CAPACITY);
//   - every page-table entry the call reads or writes lies in
//     [0, num_pages) (BCA_ERR_PAGE_RANGE);
//   - a page the call writes is used by no other sequence, and no page
//     appears twice among one sequence's used entries (BCA_ERR_PAGE_SHARED).
//     Pages that several sequences only read (a shared prefix) are allowed.
// Not on any timed path: the copies synchronise the stream.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "bca.h"
#include "bca_internal.h"

namespace bca {

bool debug_enabled() {
  const char* v = std::getenv("BCA_DEBUG");
  return v && v[0] == '1' && v[1] == '\0';
}

namespace {

// n int32 values from src (device, managed or host memory), copied on the
// stream and waited for.  In a process without a usable CUDA device src must
// be host memory, and is read directly.
int fetch(const int32_t* src, size_t n, cudaStream_t s, std::vector<int32_t>& out) {
  out.assign(n, 0);
  if (n == 0) return BCA_OK;
  cudaPointerAttributes a;
  const cudaError_t e = cudaPointerGetAttributes(&a, src);
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) {
    cudaGetLastError();
    std::memcpy(out.data(), src, n * sizeof(int32_t));
    return BCA_OK;
  }
  if (e != cudaSuccess) return BCA_ERR_CUDA;
  if (a.type == cudaMemoryTypeUnregistered || a.type == cudaMemoryTypeHost) {
    std::memcpy(out.data(), src, n * sizeof(int32_t));
    return BCA_OK;
  }
  if (cudaMemcpyAsync(out.data(), src, n * sizeof(int32_t), cudaMemcpyDefault, s) != cudaSuccess)
    return BCA_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

// Page-table entries sequence b uses: [0, n_read) read, [w0, w1) written.
struct Use {
  int n_read, w0, w1;
};

int ceil_div(long long a, int b) { return (int)((a + b - 1) / b); }

// Range of every used entry; a written page must not be used by another
// sequence; no page twice among one sequence's used entries.
int check_pages(const bca_dims* d, const int32_t* page_table, const std::vector<Use>& use,
                cudaStream_t s) {
  int n_max = 0;
  for (const Use& u : use) n_max = std::max(n_max, std::max(u.n_read, u.w1));
  if (n_max == 0) return BCA_OK;
  if (!page_table) return BCA_ERR_NULL;
  std::vector<int32_t> pt;
  int rc = fetch(page_table, (size_t)d->batch * d->max_pages_per_seq, s, pt);
  if (rc) return rc;
  std::vector<int32_t> writer((size_t)d->num_pages, -1), seen((size_t)d->num_pages, -1);
  for (int b = 0; b < d->batch; ++b) {
    const Use& u = use[(size_t)b];
    const int n = std::max(u.n_read, u.w1);
    for (int i = 0; i < n; ++i) {
      const bool used = i < u.n_read || (i >= u.w0 && i < u.w1);
      if (!used) continue;
      const int32_t page = pt[(size_t)b * d->max_pages_per_seq + i];
      if (page < 0 || page >= d->num_pages) return BCA_ERR_PAGE_RANGE;
      if (seen[(size_t)page] == b) return BCA_ERR_PAGE_SHARED;  // twice in one sequence
      seen[(size_t)page] = b;
      if (i >= u.w0 && i < u.w1) {
        if (writer[(size_t)page] >= 0 && writer[(size_t)page] != b) return BCA_ERR_PAGE_SHARED;
        writer[(size_t)page] = b;
      }
    }
  }
  // a page read by one sequence and written by another
  for (int b = 0; b < d->batch; ++b) {
    const Use& u = use[(size_t)b];
    for (int i = 0; i < u.n_read; ++i) {
      const int32_t page = pt[(size_t)b * d->max_pages_per_seq + i];
      if (writer[(size_t)page] >= 0 && writer[(size_t)page] != b) return BCA_ERR_PAGE_SHARED;
    }
  }
  return BCA_OK;
}

long long capacity(const bca_dims* d) { return (long long)d->max_pages_per_seq * d->page_size; }

}  // namespace

int debug_check_decode(const bca_dims* d, const int32_t* page_table, const int32_t* prefix_len,
                       int commit, int causal, cudaStream_t s) {
  std::vector<int32_t> P;
  int rc = fetch(prefix_len, (size_t)d->batch, s, P);
  if (rc) return rc;
  std::vector<Use> use((size_t)d->batch);
  const int D = d->block_size, S = d->page_size;
  for (int b = 0; b < d->batch; ++b) {
    const long long p = P[(size_t)b];
    if (p < 0 || (!causal && p % D != 0)) return BCA_ERR_INVALID_ARG;
    if (p + D > capacity(d)) return BCA_ERR_CAPACITY;
    use[(size_t)b] = {ceil_div(p, S), commit ? (int)(p / S) : 0, commit ? ceil_div(p + D, S) : 0};
  }
  return check_pages(d, page_table, use, s);
}

int debug_check_prefill(const bca_dims* d, const int32_t* cu_seqlens, int32_t total_tokens,
                        int32_t max_seqlen, const int32_t* page_table, cudaStream_t s) {
  std::vector<int32_t> cu;
  int rc = fetch(cu_seqlens, (size_t)d->batch + 1, s, cu);
  if (rc) return rc;
  if (cu[0] != 0 || cu[(size_t)d->batch] != total_tokens) return BCA_ERR_INVALID_ARG;
  std::vector<Use> use((size_t)d->batch, Use{0, 0, 0});
  for (int b = 0; b < d->batch; ++b) {
    const long long len = (long long)cu[(size_t)b + 1] - cu[(size_t)b];
    if (len < 0 || len > max_seqlen) return BCA_ERR_INVALID_ARG;
    if (page_table) {
      if (len > capacity(d)) return BCA_ERR_CAPACITY;
      use[(size_t)b] = {0, 0, ceil_div(len, d->page_size)};
    }
  }
  return page_table ? check_pages(d, page_table, use, s) : BCA_OK;
}

int debug_check_commit(const bca_dims* d, const int32_t* page_table, const int32_t* start_pos,
                       int32_t num_tokens, cudaStream_t s) {
  std::vector<int32_t> st;
  int rc = fetch(start_pos, (size_t)d->batch, s, st);
  if (rc) return rc;
  std::vector<Use> use((size_t)d->batch);
  for (int b = 0; b < d->batch; ++b) {
    const long long p = st[(size_t)b];
    if (p < 0) return BCA_ERR_INVALID_ARG;
    if (p + num_tokens > capacity(d)) return BCA_ERR_CAPACITY;
    use[(size_t)b] = {0, (int)(p / d->page_size), ceil_div(p + num_tokens, d->page_size)};
  }
  return check_pages(d, page_table, use, s);
}

int debug_check_qkv_post(const bca_dims* d, const int32_t* write_pos, const int32_t* page_table,
                         cudaStream_t s) {
  if (!write_pos) return BCA_OK;
  const int n = d->block_size, S = d->page_size;
  std::vector<int32_t> wp;
  int rc = fetch(write_pos, (size_t)d->batch * n, s, wp);
  if (rc) return rc;
  if (!page_table) return BCA_ERR_NULL;
  std::vector<int32_t> pt;
  if ((rc = fetch(page_table, (size_t)d->batch * d->max_pages_per_seq, s, pt))) return rc;
  // every written slot once; a page written by one sequence only
  std::vector<int32_t> writer((size_t)d->num_pages, -1);
  std::vector<uint8_t> slot_used((size_t)d->num_pages * S, 0);
  for (int b = 0; b < d->batch; ++b) {
    for (int t = 0; t < n; ++t) {
      const long long p = wp[(size_t)b * n + t];
      if (p < 0) continue;  // not written
      if (p >= capacity(d)) return BCA_ERR_CAPACITY;
      const int32_t page = pt[(size_t)b * d->max_pages_per_seq + p / S];
      if (page < 0 || page >= d->num_pages) return BCA_ERR_PAGE_RANGE;
      if (writer[(size_t)page] >= 0 && writer[(size_t)page] != b) return BCA_ERR_PAGE_SHARED;
      writer[(size_t)page] = b;
      uint8_t& u = slot_used[(size_t)page * S + p % S];
      if (u) return BCA_ERR_INVALID_ARG;  // two tokens write one slot
      u = 1;
    }
  }
  return BCA_OK;
}

int debug_check_multicanvas(const bca_dims* d, const int32_t* live_count, int32_t max_live,
                            const int32_t* page_table, const int32_t* arena_len,
                            const int32_t* commit_rows, const int32_t* commit_count,
                            int32_t max_commit, cudaStream_t s) {
  const int B = d->batch, S = d->page_size;
  std::vector<int32_t> nl, A, cc, cr;
  int rc;
  if (live_count && (rc = fetch(live_count, (size_t)B, s, nl))) return rc;
  if ((rc = fetch(arena_len, (size_t)B, s, A))) return rc;
  if (commit_rows) {
    if ((rc = fetch(commit_count, (size_t)B, s, cc))) return rc;
    if ((rc = fetch(commit_rows, (size_t)B * max_commit, s, cr))) return rc;
  }
  std::vector<Use> use((size_t)B);
  for (int b = 0; b < B; ++b) {
    const int n_live = live_count ? nl[(size_t)b] : max_live;
    if (n_live < 0 || n_live > max_live) return BCA_ERR_INVALID_ARG;
    const long long a = A[(size_t)b];
    if (a < 0) return BCA_ERR_INVALID_ARG;
    if (a > capacity(d)) return BCA_ERR_CAPACITY;
    int w0 = 0, w1 = 0;
    if (commit_rows) {
      const int c = cc[(size_t)b];
      if (c < 0 || c > max_commit || c > n_live) return BCA_ERR_INVALID_ARG;
      if (a + c > capacity(d)) return BCA_ERR_CAPACITY;
      std::vector<uint8_t> taken((size_t)n_live, 0);
      for (int i = 0; i < c; ++i) {  // indices into the live rows, each at most once
        const int row = cr[(size_t)b * max_commit + i];
        if (row < 0 || row >= n_live || taken[(size_t)row]) return BCA_ERR_INVALID_ARG;
        taken[(size_t)row] = 1;
      }
      if (c > 0) {
        w0 = (int)(a / S);
        w1 = ceil_div(a + c, S);
      }
    }
    use[(size_t)b] = {ceil_div(a, S), w0, w1};
  }
  return check_pages(d, page_table, use, s);
}

}  // namespace bca
