// bca_decode_static_scratch: the decode step with its scratch memory in a
// fixed device array owned by this library, so that the caller never has to
// allocate anything.
//
// Who needs it: code that must not call cudaMalloc (or any allocator) on the
// decode path -- a plugin hosted by an engine that owns all device memory and
// hands it no allocator, a serving loop that treats an allocation (which may
// synchronize the device or fail under fragmentation) as a fault, or a
// runtime without access to the CUDA allocator at all.  Such a caller still
// passes its own inputs and outputs; only the scratch (status header,
// per-sequence table, work list and split-KV partials) comes from here.
//
// Limits and sharing:
//  - the array holds kStaticScratchBytes (16 MiB) on every GPU that loads
//    the library, for the life of the process;
//  - a request whose minimum decode scratch does not fit is rejected with
//    BCA_ERR_WORKSPACE before anything is launched; requests that fit but
//    whose split-KV partials would not are planned with fewer splits;
//  - every call (on every stream and host thread) uses the same array, which
//    keeps the last call's contents: the header is cleared at the start of each
//    call, and calls that overlap on the GPU race on the array.
#include <mutex>

#include <cuda_runtime.h>

#include "bca.h"
#include "bca_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the name
// g_static_scratch is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BCA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return BCA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return BCA_OK;
}

}  // namespace

extern "C" int bca_decode_static_scratch(const bca_dims* d, const void* q, const void* k_blk,
                                         const void* v_blk, void* k_pool, void* v_pool,
                                         const int32_t* page_table, const int32_t* prefix_len,
                                         void* out, int commit, int32_t* device_status,
                                         bca_stream_t stream) {
  // size check from the dims alone (no workspace pointer needed for it)
  if (!d) return BCA_ERR_NULL;
  const size_t need = bca_workspace_size(d, BCA_OP_DECODE_MIN);
  if (need == 0) return BCA_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return BCA_ERR_WORKSPACE;
  void* ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc != BCA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word and counters start at zero for every call
  if (cudaMemsetAsync(ws, 0, bca::kWsHeaderBytes, s) != cudaSuccess) return BCA_ERR_CUDA;
  rc = bca_decode(d, q, k_blk, v_blk, k_pool, v_pool, page_table, prefix_len, out, commit, ws,
                  kStaticScratchBytes, stream);
  if (rc != BCA_OK) return rc;
  if (device_status) {
    // first device-detected error of this call (0 if none), stream-ordered
    if (cudaMemcpyAsync(device_status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return BCA_ERR_CUDA;
  }
  return BCA_OK;
}
