// C ABI of the library: argument checks, workspace layout, TMA descriptor
// encoding (with a small cache) and kernel launches.  Declarations and the
// contract of every entry point are in include/bca.h.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "bca.h"
#include "bca_internal.h"

namespace bca {
namespace {

constexpr int kChMin = 8;   // decode: never split a prefix into chunks shorter than 1024 keys
constexpr int kWaves = 1;   // decode: aim for about one chunk per CTA (fewest split partials)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int validate_dims(const bca_dims* d) {
  if (!d) return BCA_ERR_NULL;
  if (d->version != BCA_ABI_VERSION) return BCA_ERR_INVALID_ARG;
  if (d->batch < 0 || d->block_size < 1) return BCA_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return BCA_ERR_INVALID_ARG;
  if (d->num_kv_heads < 1 || d->num_q_heads < 1) return BCA_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return BCA_ERR_INVALID_ARG;
  if (d->num_q_heads / d->num_kv_heads > 128) return BCA_ERR_INVALID_ARG;
  if (d->page_size < 16 || d->page_size > 256 || d->page_size % 16 != 0) return BCA_ERR_INVALID_ARG;
  if (d->num_pages < 1 || d->max_pages_per_seq < 1) return BCA_ERR_INVALID_ARG;
  if (!(d->softmax_scale >= 0.0f) || !std::isfinite(d->softmax_scale)) return BCA_ERR_INVALID_ARG;
  const long long rows = (long long)d->num_pages * d->num_kv_heads * d->page_size;
  if (rows >= (1ll << 31)) return BCA_ERR_INVALID_ARG;
  return BCA_OK;
}

float scale_log2(const bca_dims* d) {
  const double s = d->softmax_scale > 0.0f ? (double)d->softmax_scale
                                           : 1.0 / std::sqrt((double)d->head_dim);
  return (float)(s * 1.4426950408889634);  // log2(e)
}

// The CTA-pair attention kernel is used wherever it applies, unless the
// environment sets BCA_PAIR_KERNEL=0 (read at each call; the single-CTA
// kernel then runs every shape, with results equal within rounding).
bool pair_kernel_enabled() {
  const char* v = std::getenv("BCA_PAIR_KERNEL");
  return !(v && v[0] == '0' && v[1] == '\0');
}

// Resident pairs of the pair kernel on the current device (cached per device).
int pair_capacity(int sms) {
  static std::atomic<int> cap[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= kMaxDevices) return attention_pair_max_pairs(sms);
  int n = cap[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    n = attention_pair_max_pairs(sms);
    if (n <= 0) return 0;
    cap[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

int device_info(DeviceInfo* di) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BCA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&di->sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&di->major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&di->minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return BCA_ERR_CUDA;
  // the kernels are built for sm_103a only
  if (di->major != 10 || di->minor != 3) return BCA_ERR_UNSUPPORTED;
  return BCA_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

using MapKey = std::tuple<uintptr_t, int, uint64_t, uint64_t, uint64_t, uint64_t, uint64_t,
                          uint32_t, uint32_t, uint32_t>;
std::mutex g_map_mu;
std::map<MapKey, CUtensorMap> g_map_cache;

// bf16 tensor map, 128-byte swizzle, zero fill out of range.  dims/strides
// innermost first; strides in bytes for dims 1..rank-1.
int encode_map(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box) {
  MapKey key{reinterpret_cast<uintptr_t>(base), rank, dims[0], dims[1], rank > 2 ? dims[2] : 0,
             strides[0], rank > 2 ? strides[1] : 0, box[0], box[1], rank > 2 ? box[2] : 0};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *out = it->second;
      return BCA_OK;
    }
  }
  EncodeFn fn = encode_fn();
  if (!fn) return BCA_ERR_CUDA;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                  gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return BCA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_map_cache.size() > 1024) g_map_cache.clear();
    g_map_cache[key] = m;
  }
  *out = m;
  return BCA_OK;
}

// [tokens, heads, d] bf16 viewed as (d, heads, tokens); box (64, box_h, box_t).
int encode_tokens_map(CUtensorMap* out, const void* base, int d, int heads, long long tokens,
                      int box_h, int box_t) {
  const uint64_t dims[3] = {(uint64_t)d, (uint64_t)heads, (uint64_t)(tokens > 0 ? tokens : 1)};
  const uint64_t strides[2] = {(uint64_t)d * 2, (uint64_t)heads * d * 2};
  const uint32_t box[3] = {64u, (uint32_t)box_h, (uint32_t)box_t};
  return encode_map(out, base, 3, dims, strides, box);
}

// [num_pages, Hkv, S, d] bf16 viewed as (d, num_pages*Hkv*S); box (64, 16).
int encode_pool_map(CUtensorMap* out, const void* base, int d, long long rows) {
  const uint64_t dims[2] = {(uint64_t)d, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)d * 2};
  const uint32_t box[2] = {64u, (uint32_t)kChunkKeys};
  return encode_map(out, base, 2, dims, strides, box);
}

int ceil_div_i(long long a, long long b) { return (int)((a + b - 1) / b); }

AttnParams base_params(const bca_dims* d) {
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = d->batch;
  p.Hq = d->num_q_heads;
  p.Hkv = d->num_kv_heads;
  p.G = d->num_q_heads / d->num_kv_heads;
  p.S = d->page_size;
  p.num_pages = d->num_pages;
  p.max_pages = d->max_pages_per_seq;
  p.Dblk = d->block_size;
  p.scale_log2 = scale_log2(d);
  p.ch_min = kChMin;
  p.waves = kWaves;
  p.pool_rows = d->num_pages * d->num_kv_heads * d->page_size;
  return p;
}

// ---------------------------------------------------------------------------
// optional kernel timing (bca_profile_start / bca_profile_stop)
// ---------------------------------------------------------------------------
struct Profile {
  std::mutex mu;
  bool active = false;
  std::vector<cudaEvent_t> ev;     // 2 per slot
  std::vector<int> kind;           // per used slot
  int used = 0;
};
Profile g_prof;

// Returns a slot index (or -1) and records its start event on `s`.
int prof_begin(int k, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.active || g_prof.used * 2 >= (int)g_prof.ev.size()) return -1;
  const int i = g_prof.used++;
  g_prof.kind[i] = k;
  cudaEventRecord(g_prof.ev[2 * i], s);
  return i;
}

void prof_end(int i, cudaStream_t s) {
  if (i < 0) return;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  cudaEventRecord(g_prof.ev[2 * i + 1], s);
}

// Launch helper: times the launch when a profile is active.
template <typename F>
cudaError_t timed(int k, cudaStream_t s, F&& launch) {
  const int i = prof_begin(k, s);
  const cudaError_t e = launch();
  prof_end(i, s);
  return e;
}

}  // namespace

DecodeWsLayout decode_ws_layout(int B, int Hkv, int n_rb, int head_dim, int n_sms,
                                size_t ws_bytes) {
  DecodeWsLayout l;
  l.split_base_off = kWsHeaderBytes;
  l.items_off = l.split_base_off + round_up((size_t)(B > 0 ? B : 1) * 4, 256);
  l.items_cap = n_sms * kWaves + B * Hkv * n_rb;
  l.slot_off = l.items_off + round_up((size_t)l.items_cap * 32, 256);
  // per split slot: its table entry, (max, sum) for 256 rows, O for 256 rows
  l.bytes_per_slot = 16 + 256 * 2 * 4 + (size_t)256 * head_dim * 4;
  l.cap = 0;
  if (ws_bytes > l.slot_off + 512)
    l.cap = (int)std::min<size_t>((ws_bytes - l.slot_off - 512) / l.bytes_per_slot, 1 << 30);
  l.ml_off = l.slot_off + round_up((size_t)l.cap * 16, 256);
  l.o_off = l.ml_off + round_up((size_t)l.cap * 256 * 2 * 4, 256);
  return l;
}

size_t multicanvas_ws_bytes(int B, int max_pages, int S) {
  const size_t n_at = ((size_t)max_pages * S + kTileKeys - 1) / kTileKeys;
  return kWsHeaderBytes + round_up((size_t)(B > 0 ? B : 1) * n_at * sizeof(int2), 256);
}

size_t decode_ws_minimum(int B, int Hkv, int n_rb, int head_dim, int n_sms) {
  return decode_ws_layout(B, Hkv, n_rb, head_dim, n_sms, 0).slot_off;
}

size_t decode_ws_recommended(int B, int Hkv, int n_rb, int head_dim, int n_sms) {
  DecodeWsLayout l = decode_ws_layout(B, Hkv, n_rb, head_dim, n_sms, 0);
  // split slots never exceed the work items
  return l.slot_off + (size_t)l.items_cap * l.bytes_per_slot + 512;
}

}  // namespace bca

using namespace bca;

extern "C" {

int bca_version(void) { return BCA_ABI_VERSION; }

const char* bca_status_string(int s) {
  switch (s) {
    case BCA_OK: return "ok";
    case BCA_ERR_INVALID_ARG: return "invalid argument";
    case BCA_ERR_NULL: return "null pointer";
    case BCA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case BCA_ERR_WORKSPACE: return "workspace missing or too small";
    case BCA_ERR_CAPACITY: return "request exceeds the page table capacity";
    case BCA_ERR_CUDA: return "CUDA call failed";
    case BCA_ERR_UNSUPPORTED: return "device is not sm_103 (GB300)";
    case BCA_ERR_PAGE_SHARED: return "a page is used twice";
    case BCA_ERR_PAGE_RANGE: return "a page id is outside the pool";
    case BCA_ERR_DEVICE_PAGE_OOB: return "device: page id outside the pool";
    case BCA_ERR_DEVICE_BAD_LENGTH: return "device: length or position out of range";
    case BCA_ERR_DEVICE_TIMEOUT: return "device: internal wait timed out";
    default: return "unknown status";
  }
}

size_t bca_workspace_size(const bca_dims* d, int op) {
  if (validate_dims(d) != BCA_OK) return 0;
  if (op == BCA_OP_DECODE || op == BCA_OP_DECODE_MIN) {
    DeviceInfo di;
    int sms = 160;
    if (device_info(&di) == BCA_OK) sms = di.sms;
    const int G = d->num_q_heads / d->num_kv_heads;
    const int tpm = 128 / G;
    const int n_rb = ceil_div_i(d->block_size, 2 * tpm);
    return op == BCA_OP_DECODE
               ? decode_ws_recommended(d->batch, d->num_kv_heads, n_rb, d->head_dim, sms)
               : decode_ws_minimum(d->batch, d->num_kv_heads, n_rb, d->head_dim, sms);
  }
  if (op == BCA_OP_MULTICANVAS)
    return multicanvas_ws_bytes(d->batch, d->max_pages_per_seq, d->page_size);
  if (op == BCA_OP_PREFILL || op == BCA_OP_COMMIT) return kWsHeaderBytes;
  return 0;
}

int bca_workspace_init(void* ws, size_t bytes, bca_stream_t stream) {
  if (!ws) return BCA_ERR_NULL;
  if (bytes < kWsHeaderBytes) return BCA_ERR_WORKSPACE;
  if (cudaMemsetAsync(ws, 0, kWsHeaderBytes, (cudaStream_t)stream) != cudaSuccess)
    return BCA_ERR_CUDA;
  return BCA_OK;
}

int bca_read_device_status(void* ws, bca_stream_t stream) {
  if (!ws) return BCA_ERR_NULL;
  int32_t st = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&st, ws, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(st), s) != cudaSuccess) return BCA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BCA_ERR_CUDA;
  return st;
}

int bca_read_tile_counters(void* ws, int64_t counters[3], bca_stream_t stream) {
  if (!ws || !counters) return BCA_ERR_NULL;
  WsHeader h;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BCA_ERR_CUDA;
  counters[0] = (int64_t)h.tiles_full;
  counters[1] = (int64_t)h.tiles_partial;
  counters[2] = (int64_t)h.tiles_skipped;
  return BCA_OK;
}

int bca_qkv_post(const bca_dims* d, const void* qkv, const int32_t* positions,
                 const void* q_norm_w, const void* k_norm_w, float eps, float rope_theta,
                 void* q_out, void* k_out, void* v_out, const int32_t* write_pos,
                 void* k_pool, void* v_pool, const int32_t* page_table, int32_t* kv_pos,
                 void* ws, size_t ws_bytes, bca_stream_t stream) {
  int rc = validate_dims(d);
  if (rc) return rc;
  if (!(eps >= 0.f) || !std::isfinite(eps) || !(rope_theta >= 0.f) || !std::isfinite(rope_theta))
    return BCA_ERR_INVALID_ARG;
  if (d->batch == 0) return BCA_OK;
  if (!qkv || !q_out || !k_out || !v_out || !ws) return BCA_ERR_NULL;
  if ((rope_theta > 0.f || kv_pos) && !positions) return BCA_ERR_NULL;
  if (write_pos && (!k_pool || !v_pool || !page_table)) return BCA_ERR_NULL;
  if (kv_pos && !write_pos) return BCA_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(v_out) ||
      (write_pos && (!aligned16(k_pool) || !aligned16(v_pool))) || !aligned16(ws))
    return BCA_ERR_ALIGN;
  if (ws_bytes < kWsHeaderBytes) return BCA_ERR_WORKSPACE;
  if (debug_enabled() &&
      (rc = debug_check_qkv_post(d, write_pos, page_table, (cudaStream_t)stream)))
    return rc;
  DeviceInfo di;
  if ((rc = device_info(&di))) return rc;
  QkvPostParams c;
  std::memset(&c, 0, sizeof(c));
  c.qkv = (const uint16_t*)qkv;
  c.positions = positions;
  c.q_norm_w = (const uint16_t*)q_norm_w;
  c.k_norm_w = (const uint16_t*)k_norm_w;
  c.eps = eps;
  c.rope_theta = rope_theta;
  if (rope_theta > 0.f) {
    const int half = d->head_dim / 2;
    for (int i = 0; i < half; ++i) {
      const double f = std::pow((double)rope_theta, -2.0 * i / d->head_dim);  // radians per position
      const double t = f / 6.283185307179586476925286766559;                 // turns per position
      c.rope_turns[i] = (unsigned long long)(t * 18446744073709551616.0);     // * 2^64, < 2^62
    }
  }
  c.q_out = (uint16_t*)q_out;
  c.k_out = (uint16_t*)k_out;
  c.v_out = (uint16_t*)v_out;
  c.write_pos = write_pos;
  c.k_pool = (uint16_t*)k_pool;
  c.v_pool = (uint16_t*)v_pool;
  c.page_table = page_table;
  c.kv_pos = kv_pos;
  c.B = d->batch;
  c.n = d->block_size;
  c.Hq = d->num_q_heads;
  c.Hkv = d->num_kv_heads;
  c.S = d->page_size;
  c.num_pages = d->num_pages;
  c.max_pages = d->max_pages_per_seq;
  c.hdr = (WsHeader*)ws;
  cudaStream_t s = (cudaStream_t)stream;
  return timed(BCA_KERNEL_QKV_POST, s, [&] { return launch_qkv_post(c, d->head_dim, di.sms, s); }) ==
                 cudaSuccess
             ? BCA_OK
             : BCA_ERR_CUDA;
}

int bca_confidence(int64_t rows, int64_t vocab, int64_t ld, int dtype, const void* logits,
                   int32_t* argmax, float* conf, bca_stream_t stream) {
  if (rows < 0 || vocab < 1 || vocab >= (1ll << 31) || ld < vocab) return BCA_ERR_INVALID_ARG;
  if (dtype != BCA_DTYPE_BF16 && dtype != BCA_DTYPE_F32) return BCA_ERR_INVALID_ARG;
  if (rows == 0) return BCA_OK;
  if (rows >= (1ll << 31)) return BCA_ERR_INVALID_ARG;  // one CTA per row
  if (!logits || !argmax || !conf) return BCA_ERR_NULL;
  const int esize = dtype == BCA_DTYPE_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % esize != 0 ||
      reinterpret_cast<uintptr_t>(argmax) % 4 != 0 || reinterpret_cast<uintptr_t>(conf) % 4 != 0)
    return BCA_ERR_ALIGN;
  DeviceInfo di;
  int rc = device_info(&di);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  return timed(BCA_KERNEL_CONFIDENCE, s, [&] {
           return launch_confidence(rows, (int)vocab, ld, dtype, logits, argmax, conf, s);
         }) == cudaSuccess
             ? BCA_OK
             : BCA_ERR_CUDA;
}

int bca_commit_kv(const bca_dims* d, const void* k_blk, const void* v_blk, void* k_pool,
                  void* v_pool, const int32_t* page_table, const int32_t* start_pos,
                  int32_t num_tokens, void* ws, size_t ws_bytes, bca_stream_t stream) {
  int rc = validate_dims(d);
  if (rc) return rc;
  if (num_tokens < 0 || num_tokens > d->block_size) return BCA_ERR_INVALID_ARG;
  if (d->batch == 0 || num_tokens == 0) return BCA_OK;
  if (!k_blk || !v_blk || !k_pool || !v_pool || !page_table || !start_pos || !ws)
    return BCA_ERR_NULL;
  if (!aligned16(k_blk) || !aligned16(v_blk) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(ws))
    return BCA_ERR_ALIGN;
  if (ws_bytes < kWsHeaderBytes) return BCA_ERR_WORKSPACE;
  if (debug_enabled() &&
      (rc = debug_check_commit(d, page_table, start_pos, num_tokens, (cudaStream_t)stream)))
    return rc;
  CommitParams c;
  std::memset(&c, 0, sizeof(c));
  c.k_src = (const uint16_t*)k_blk;
  c.v_src = (const uint16_t*)v_blk;
  c.k_pool = (uint16_t*)k_pool;
  c.v_pool = (uint16_t*)v_pool;
  c.page_table = page_table;
  c.start_pos = start_pos;
  c.rows_per_seq = d->block_size;
  c.num_tokens = num_tokens;
  c.max_rows = num_tokens;
  c.B = d->batch;
  c.Hkv = d->num_kv_heads;
  c.d = d->head_dim;
  c.S = d->page_size;
  c.num_pages = d->num_pages;
  c.max_pages = d->max_pages_per_seq;
  c.hdr = (WsHeader*)ws;
  return timed(BCA_KERNEL_COMMIT, (cudaStream_t)stream, [&] { return launch_commit(c, (cudaStream_t)stream); }) == cudaSuccess
             ? BCA_OK
             : BCA_ERR_CUDA;
}

namespace {
// Decode step (causal = 0) or short causal extend (causal = 1): the same
// kernels, the extend with one-token mask blocks and no prefix alignment.
int decode_impl(const bca_dims* d, const void* q, const void* k_blk, const void* v_blk,
                void* k_pool, void* v_pool, const int32_t* page_table,
                const int32_t* prefix_len, void* out, int commit, int causal, void* ws,
                size_t ws_bytes, bca_stream_t stream) {
  int rc = validate_dims(d);
  if (rc) return rc;
  if (commit != 0 && commit != 1) return BCA_ERR_INVALID_ARG;
  if (d->batch == 0) return BCA_OK;
  if (!q || !k_blk || !v_blk || !k_pool || !v_pool || !page_table || !prefix_len || !out || !ws)
    return BCA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(k_pool) ||
      !aligned16(v_pool) || !aligned16(out) || !aligned16(ws))
    return BCA_ERR_ALIGN;
  const long long cap_tokens = (long long)d->max_pages_per_seq * d->page_size;
  if (d->block_size > cap_tokens) return BCA_ERR_CAPACITY;
  const long long q_tokens = (long long)d->batch * d->block_size;
  if (q_tokens * d->num_q_heads >= (1ll << 31)) return BCA_ERR_INVALID_ARG;
  if (ws_bytes < kWsHeaderBytes + round_up((size_t)d->batch * 4, 256)) return BCA_ERR_WORKSPACE;
  if (debug_enabled() &&
      (rc = debug_check_decode(d, page_table, prefix_len, commit, causal, (cudaStream_t)stream)))
    return rc;
  DeviceInfo di;
  if ((rc = device_info(&di))) return rc;
  const int G0 = d->num_q_heads / d->num_kv_heads;
  const int n_rb0 = ceil_div_i(d->block_size, 2 * (128 / G0));
  const DecodeWsLayout lay =
      decode_ws_layout(d->batch, d->num_kv_heads, n_rb0, d->head_dim, di.sms, ws_bytes);
  if (ws_bytes < lay.slot_off) return BCA_ERR_WORKSPACE;

  AttnParams p = base_params(d);
  p.mode = kModeDecode;
  p.causal = causal;
  p.hpr = p.G;
  p.tpm = 128 / p.G;
  p.n_hp = 1;
  p.n_rb = ceil_div_i(d->block_size, 2 * p.tpm);
  p.page_table = page_table;
  p.lens = prefix_len;
  p.k_pool = (const uint16_t*)k_pool;
  p.v_pool = (const uint16_t*)v_pool;
  p.k_dense = (const uint16_t*)k_blk;
  p.v_dense = (const uint16_t*)v_blk;
  p.dense_tokens = (int)q_tokens;
  p.out = (uint16_t*)out;
  p.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p.hdr = (WsHeader*)ws;
  p.split_base = (int32_t*)((char*)ws + lay.split_base_off);
  p.items = (int4*)((char*)ws + lay.items_off);
  p.items_cap = lay.items_cap;
  p.slot_info = (int4*)((char*)ws + lay.slot_off);
  p.part_ml = (float*)((char*)ws + lay.ml_off);
  p.part_o = (float*)((char*)ws + lay.o_off);
  p.split_cap = lay.cap;
  // the commit of the block runs in the epilogue kernel, after the attention
  p.commit_k = commit ? (uint16_t*)k_pool : nullptr;
  p.commit_v = commit ? (uint16_t*)v_pool : nullptr;

  AttnMaps maps;
  const int HD = d->head_dim;
  if ((rc = encode_tokens_map(&maps.q, q, HD, d->num_q_heads, q_tokens, p.hpr, p.tpm))) return rc;
  if ((rc = encode_pool_map(&maps.kp, k_pool, HD, p.pool_rows))) return rc;
  if ((rc = encode_pool_map(&maps.vp, v_pool, HD, p.pool_rows))) return rc;
  if ((rc = encode_tokens_map(&maps.kd, k_blk, HD, d->num_kv_heads, q_tokens, 1, kChunkKeys)))
    return rc;
  if ((rc = encode_tokens_map(&maps.vd, v_blk, HD, d->num_kv_heads, q_tokens, 1, kChunkKeys)))
    return rc;

  const long long max_tiles = ceil_div_i(cap_tokens, kTileKeys) + ceil_div_i(d->block_size, kTileKeys);
  const long long max_items =
      (long long)d->batch * d->num_kv_heads * p.n_rb * ceil_div_i(max_tiles, kChMin);
  int grid = (int)std::min<long long>(di.sms, std::max<long long>(1, max_items));
  // CTA pairs: blocks whose first row block fills both M-tiles, head_dim 128
  int n_pairs = 0;
  if (pair_kernel_enabled() && HD == 128 && d->block_size > p.tpm) {
    n_pairs = (int)std::min<long long>(pair_capacity(di.sms), std::max<long long>(1, max_items));
    p.pair = n_pairs > 0 ? 1 : 0;
  }
  const int units = p.pair ? n_pairs : grid;
  cudaStream_t s = (cudaStream_t)stream;
  // small batches are planned inside the attention kernel (no plan launch)
  p.fused_plan = d->batch <= kFusedPlanMax ? 1 : 0;
  if (!p.fused_plan &&
      timed(BCA_KERNEL_PLAN, s, [&] { return launch_plan(p, units, s); }) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (timed(BCA_KERNEL_ATTENTION, s, [&] {
        return p.pair ? launch_attention_pair(p, maps, n_pairs, s)
                      : launch_attention(p, maps, HD, grid, s);
      }) != cudaSuccess)
    return BCA_ERR_CUDA;
  // epilogue: the commit (if asked) and the split-KV combine (if any prefix can split)
  if (commit || max_tiles > kChMin) {
    if (timed(BCA_KERNEL_COMBINE, s, [&] { return launch_decode_combine(p, HD, di.sms, s); }) != cudaSuccess)
      return BCA_ERR_CUDA;
  }
  return BCA_OK;
}
}  // namespace

int bca_decode(const bca_dims* d, const void* q, const void* k_blk, const void* v_blk,
               void* k_pool, void* v_pool, const int32_t* page_table, const int32_t* prefix_len,
               void* out, int commit, void* ws, size_t ws_bytes, bca_stream_t stream) {
  return decode_impl(d, q, k_blk, v_blk, k_pool, v_pool, page_table, prefix_len, out, commit, 0,
                     ws, ws_bytes, stream);
}

int bca_extend(const bca_dims* d, const void* q, const void* k_new, const void* v_new,
               void* k_pool, void* v_pool, const int32_t* page_table, const int32_t* prefix_len,
               void* out, int commit, void* ws, size_t ws_bytes, bca_stream_t stream) {
  return decode_impl(d, q, k_new, v_new, k_pool, v_pool, page_table, prefix_len, out, commit, 1,
                     ws, ws_bytes, stream);
}

int bca_prefill(const bca_dims* d, const void* q, const void* k, const void* v,
                const int32_t* cu_seqlens, int32_t total_tokens, int32_t max_seqlen,
                void* k_pool, void* v_pool, const int32_t* page_table, void* out, void* ws,
                size_t ws_bytes, bca_stream_t stream) {
  int rc = validate_dims(d);
  if (rc) return rc;
  if (total_tokens < 0 || max_seqlen < 0) return BCA_ERR_INVALID_ARG;
  if (d->batch == 0 || total_tokens == 0 || max_seqlen == 0) return BCA_OK;
  if (!q || !k || !v || !cu_seqlens || !out || !ws) return BCA_ERR_NULL;
  if ((k_pool == nullptr) != (v_pool == nullptr)) return BCA_ERR_NULL;
  if (k_pool && !page_table) return BCA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws) ||
      (k_pool && (!aligned16(k_pool) || !aligned16(v_pool))))
    return BCA_ERR_ALIGN;
  if ((long long)total_tokens * d->num_q_heads >= (1ll << 31)) return BCA_ERR_INVALID_ARG;
  if (k_pool && (long long)max_seqlen > (long long)d->max_pages_per_seq * d->page_size)
    return BCA_ERR_CAPACITY;
  if (ws_bytes < kWsHeaderBytes) return BCA_ERR_WORKSPACE;
  if (debug_enabled() &&
      (rc = debug_check_prefill(d, cu_seqlens, total_tokens, max_seqlen,
                                k_pool ? page_table : nullptr, (cudaStream_t)stream)))
    return rc;
  DeviceInfo di;
  if ((rc = device_info(&di))) return rc;

  AttnParams p = base_params(d);
  p.mode = kModePrefill;
  p.hpr = 1;
  p.tpm = 128;
  p.n_hp = (p.G + 1) / 2;
  p.n_rb = 1;
  p.n_qt_max = ceil_div_i(max_seqlen, 128);
  p.page_table = page_table;
  p.lens = cu_seqlens;
  p.k_dense = (const uint16_t*)k;
  p.v_dense = (const uint16_t*)v;
  p.dense_tokens = total_tokens;
  p.out = (uint16_t*)out;
  p.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p.hdr = (WsHeader*)ws;

  AttnMaps maps;
  const int HD = d->head_dim;
  if ((rc = encode_tokens_map(&maps.q, q, HD, d->num_q_heads, total_tokens, 1, 128))) return rc;
  if ((rc = encode_tokens_map(&maps.kd, k, HD, d->num_kv_heads, total_tokens, 1, kChunkKeys)))
    return rc;
  if ((rc = encode_tokens_map(&maps.vd, v, HD, d->num_kv_heads, total_tokens, 1, kChunkKeys)))
    return rc;
  maps.kp = maps.kd;  // no paged source in prefill
  maps.vp = maps.vd;
  const long long max_items = (long long)d->batch * ceil_div_i(max_seqlen, 128) *
                              d->num_kv_heads * p.n_hp;
  const int grid = (int)std::min<long long>(di.sms, std::max<long long>(1, max_items));
  // CTA pairs: two query heads per item (G >= 2), head_dim 128
  int n_pairs = 0;
  if (pair_kernel_enabled() && HD == 128 && p.G >= 2) {
    n_pairs = (int)std::min<long long>(pair_capacity(di.sms), std::max<long long>(1, max_items));
    p.pair = n_pairs > 0 ? 1 : 0;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (timed(BCA_KERNEL_PLAN, s, [&] { return launch_plan(p, p.pair ? n_pairs : grid, s); }) !=
      cudaSuccess)
    return BCA_ERR_CUDA;
  if (timed(BCA_KERNEL_ATTENTION, s, [&] {
        return p.pair ? launch_attention_pair(p, maps, n_pairs, s)
                      : launch_attention(p, maps, HD, grid, s);
      }) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (k_pool) {
    CommitParams c;
    std::memset(&c, 0, sizeof(c));
    c.k_src = (const uint16_t*)k;
    c.v_src = (const uint16_t*)v;
    c.k_pool = (uint16_t*)k_pool;
    c.v_pool = (uint16_t*)v_pool;
    c.page_table = page_table;
    c.cu = cu_seqlens;
    c.max_rows = max_seqlen;
    c.B = d->batch;
    c.Hkv = d->num_kv_heads;
    c.d = HD;
    c.S = d->page_size;
    c.num_pages = d->num_pages;
    c.max_pages = d->max_pages_per_seq;
    c.hdr = p.hdr;
    if (timed(BCA_KERNEL_COMMIT, s, [&] { return launch_commit(c, s); }) != cudaSuccess) return BCA_ERR_CUDA;
  }
  return BCA_OK;
}

namespace {
int multicanvas_impl(const bca_dims* d, const void* q_live, const void* k_live,
                     const void* v_live, const int32_t* live_pos, const int32_t* live_count,
                     int32_t max_live, int32_t prompt_len, int32_t n_canvas, void* k_pool,
                     void* v_pool, const int32_t* page_table, int32_t* kv_pos,
                     int32_t* arena_len, const int32_t* commit_rows,
                     const int32_t* commit_count, int32_t max_commit, int32_t window, void* out,
                     void* ws, size_t ws_bytes, bca_stream_t stream) {
  int rc = validate_dims(d);
  if (rc) return rc;
  if (max_live < 0 || prompt_len < 0 || n_canvas < 1 || max_commit < 0 || window < 0)
    return BCA_ERR_INVALID_ARG;
  if ((long long)prompt_len + (long long)n_canvas * d->block_size >= (1ll << 31))
    return BCA_ERR_INVALID_ARG;
  if (d->batch == 0 || max_live == 0) return BCA_OK;
  if (!q_live || !k_live || !v_live || !k_pool || !v_pool || !page_table || !kv_pos ||
      !arena_len || !out || !ws)
    return BCA_ERR_NULL;
  if (commit_rows && !commit_count) return BCA_ERR_NULL;
  if (!aligned16(q_live) || !aligned16(k_live) || !aligned16(v_live) || !aligned16(k_pool) ||
      !aligned16(v_pool) || !aligned16(out) || !aligned16(ws))
    return BCA_ERR_ALIGN;
  const long long q_tokens = (long long)d->batch * max_live;
  if (q_tokens * d->num_q_heads >= (1ll << 31)) return BCA_ERR_INVALID_ARG;
  if (ws_bytes < multicanvas_ws_bytes(d->batch, d->max_pages_per_seq, d->page_size))
    return BCA_ERR_WORKSPACE;
  if (debug_enabled() &&
      (rc = debug_check_multicanvas(d, live_count, max_live, page_table, arena_len, commit_rows,
                                    commit_count, max_commit, (cudaStream_t)stream)))
    return rc;
  DeviceInfo di;
  if ((rc = device_info(&di))) return rc;

  AttnParams p = base_params(d);
  p.mode = kModeMulticanvas;
  p.hpr = p.G;
  p.tpm = 128 / p.G;
  p.n_hp = 1;
  p.n_rb = 1;
  p.n_rb_max = ceil_div_i(max_live, 2 * p.tpm);
  p.page_table = page_table;
  p.lens = live_count;
  p.live_pos = live_pos;
  p.kv_pos = kv_pos;
  p.arena_len = arena_len;
  p.max_live = max_live;
  p.prompt_len = prompt_len;
  p.window = window;
  p.k_pool = (const uint16_t*)k_pool;
  p.v_pool = (const uint16_t*)v_pool;
  p.k_dense = (const uint16_t*)k_live;
  p.v_dense = (const uint16_t*)v_live;
  p.dense_tokens = (int)q_tokens;
  p.out = (uint16_t*)out;
  p.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p.hdr = (WsHeader*)ws;
  p.tile_kv = (int2*)((char*)ws + kWsHeaderBytes);
  p.n_at_max = ceil_div_i((long long)d->max_pages_per_seq * d->page_size, kTileKeys);

  AttnMaps maps;
  const int HD = d->head_dim;
  if ((rc = encode_tokens_map(&maps.q, q_live, HD, d->num_q_heads, q_tokens, p.hpr, p.tpm)))
    return rc;
  if ((rc = encode_pool_map(&maps.kp, k_pool, HD, p.pool_rows))) return rc;
  if ((rc = encode_pool_map(&maps.vp, v_pool, HD, p.pool_rows))) return rc;
  if ((rc = encode_tokens_map(&maps.kd, k_live, HD, d->num_kv_heads, q_tokens, 1, kChunkKeys)))
    return rc;
  if ((rc = encode_tokens_map(&maps.vd, v_live, HD, d->num_kv_heads, q_tokens, 1, kChunkKeys)))
    return rc;
  const long long max_items =
      (long long)d->batch * d->num_kv_heads * ceil_div_i(max_live, 2 * p.tpm);
  const int grid = (int)std::min<long long>(di.sms, std::max<long long>(1, max_items));
  // CTA pairs for head_dim 128 (items are two M-tiles of live rows)
  int n_pairs = 0;
  if (pair_kernel_enabled() && HD == 128) {
    n_pairs = (int)std::min<long long>(pair_capacity(di.sms), std::max<long long>(1, max_items));
    p.pair = n_pairs > 0 ? 1 : 0;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (timed(BCA_KERNEL_PLAN, s, [&] { return launch_plan(p, p.pair ? n_pairs : grid, s); }) !=
      cudaSuccess)
    return BCA_ERR_CUDA;
  if (timed(BCA_KERNEL_ATTENTION, s, [&] {
        return p.pair ? launch_attention_pair(p, maps, n_pairs, s)
                      : launch_attention(p, maps, HD, grid, s);
      }) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (commit_rows && max_commit > 0) {
    PromoteParams c;
    std::memset(&c, 0, sizeof(c));
    c.k_live = (const uint16_t*)k_live;
    c.v_live = (const uint16_t*)v_live;
    c.k_pool = (uint16_t*)k_pool;
    c.v_pool = (uint16_t*)v_pool;
    c.page_table = page_table;
    c.live_pos = live_pos;
    c.live_count = live_count;
    c.kv_pos = kv_pos;
    c.arena_len = arena_len;
    c.commit_rows = commit_rows;
    c.commit_count = commit_count;
    c.B = d->batch;
    c.Hkv = d->num_kv_heads;
    c.d = HD;
    c.S = d->page_size;
    c.num_pages = d->num_pages;
    c.max_pages = d->max_pages_per_seq;
    c.max_live = max_live;
    c.max_commit = max_commit;
    c.prompt_len = prompt_len;
    c.hdr = p.hdr;
    if (timed(BCA_KERNEL_PROMOTE, s, [&] { return launch_promote(c, s); }) != cudaSuccess) return BCA_ERR_CUDA;
  }
  return BCA_OK;
}
}  // namespace

int bca_multicanvas(const bca_dims* d, const void* q_live, const void* k_live,
                    const void* v_live, const int32_t* live_pos, const int32_t* live_count,
                    int32_t max_live, int32_t prompt_len, int32_t n_canvas, void* k_pool,
                    void* v_pool, const int32_t* page_table, int32_t* kv_pos,
                    int32_t* arena_len, const int32_t* commit_rows,
                    const int32_t* commit_count, int32_t max_commit, void* out, void* ws,
                    size_t ws_bytes, bca_stream_t stream) {
  return multicanvas_impl(d, q_live, k_live, v_live, live_pos, live_count, max_live, prompt_len,
                          n_canvas, k_pool, v_pool, page_table, kv_pos, arena_len, commit_rows,
                          commit_count, max_commit, 0, out, ws, ws_bytes, stream);
}

int bca_multicanvas_window(const bca_dims* d, const void* q_live, const void* k_live,
                           const void* v_live, const int32_t* live_pos,
                           const int32_t* live_count, int32_t max_live, int32_t prompt_len,
                           int32_t n_canvas, int32_t window, void* k_pool, void* v_pool,
                           const int32_t* page_table, int32_t* kv_pos, int32_t* arena_len,
                           const int32_t* commit_rows, const int32_t* commit_count,
                           int32_t max_commit, void* out, void* ws, size_t ws_bytes,
                           bca_stream_t stream) {
  return multicanvas_impl(d, q_live, k_live, v_live, live_pos, live_count, max_live, prompt_len,
                          n_canvas, k_pool, v_pool, page_table, kv_pos, arena_len, commit_rows,
                          commit_count, max_commit, window, out, ws, ws_bytes, stream);
}

int bca_validate_page_table(const bca_dims* d, const int32_t* pt, const int32_t* used,
                            int32_t* bad_seq, int32_t* bad_entry) {
  int rc = validate_dims(d);
  if (rc) return rc;
  if (!pt || !used) return BCA_ERR_NULL;
  std::vector<int32_t> owner((size_t)d->num_pages, -1);
  for (int b = 0; b < d->batch; ++b) {
    if (used[b] < 0 || (long long)used[b] > (long long)d->max_pages_per_seq * d->page_size) {
      if (bad_seq) *bad_seq = b;
      if (bad_entry) *bad_entry = -1;
      return BCA_ERR_CAPACITY;
    }
    const int n = (used[b] + d->page_size - 1) / d->page_size;
    for (int i = 0; i < n; ++i) {
      const int32_t page = pt[(size_t)b * d->max_pages_per_seq + i];
      if (page < 0 || page >= d->num_pages) {
        if (bad_seq) *bad_seq = b;
        if (bad_entry) *bad_entry = i;
        return BCA_ERR_PAGE_RANGE;
      }
      if (owner[page] >= 0) {
        if (bad_seq) *bad_seq = b;
        if (bad_entry) *bad_entry = i;
        return BCA_ERR_PAGE_SHARED;
      }
      owner[page] = b;
    }
  }
  return BCA_OK;
}

int bca_profile_start(int32_t max_launches) {
  if (max_launches < 1 || max_launches > (1 << 20)) return BCA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.active) return BCA_ERR_INVALID_ARG;
  g_prof.ev.assign((size_t)max_launches * 2, nullptr);
  for (auto& e : g_prof.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (auto& x : g_prof.ev)
        if (x) cudaEventDestroy(x);
      g_prof.ev.clear();
      return BCA_ERR_CUDA;
    }
  }
  g_prof.kind.assign((size_t)max_launches, -1);
  g_prof.used = 0;
  g_prof.active = true;
  return BCA_OK;
}

int bca_profile_stop(bca_kernel_times* out) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.active) return BCA_ERR_INVALID_ARG;
  bca_kernel_times t;
  std::memset(&t, 0, sizeof(t));
  int rc = BCA_OK;
  for (int i = 0; i < g_prof.used; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) {
      rc = BCA_ERR_CUDA;
      continue;
    }
    const int k = g_prof.kind[i];
    if (k >= 0 && k < BCA_KERNEL_KINDS) {
      t.launches[k] += 1;
      t.total_ms[k] += ms;
    }
  }
  for (auto& e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  g_prof.kind.clear();
  g_prof.used = 0;
  g_prof.active = false;
  if (out) *out = t;
  return rc;
}

}  // extern "C"
