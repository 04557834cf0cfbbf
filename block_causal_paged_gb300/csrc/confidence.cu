// Softmax-plus-argmax over the vocabulary: the top prediction of each
// position and its probability ("Inference: Fewer, smaller forwards",
// "Advancement 2: tau_conf"; "Advancement 16": one fused pass).
//
// One CTA per row streams the row once with 16-byte loads (four in flight
// per thread; the elements before the row's first 16-byte boundary and after
// its last one are read singly) and keeps, per thread, an online (running maximum m in log2
// units, sum of 2^(x - m), first index of the maximum); the block merges the
// 256 triples (ties go to the lower index) and conf = 1 / sum.  The pass is
// bound by HBM: per row vocab x element size bytes read, 8 bytes written.
#include <cstdint>

#include "bca_internal.h"

namespace bca {
namespace {

constexpr int kConfThreads = 256;
constexpr int kUnroll = 4;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Running state of one thread.  The maximum is kept as the raw logit, so
// that the argmax is decided by exact comparisons of the input values (two
// logits that differ never tie after a rounding), and scaled by log2(e) for
// the exponents.
struct Acc {
  float m;   // running maximum logit (-inf: nothing seen)
  float mb;  // m * log2(e)
  float s;   // sum of exp(x - m) = 2^(x log2 e - mb)
  int i;     // first index holding the maximum
};

__device__ __forceinline__ Acc merge(Acc a, Acc b) {
  Acc r;
  if (a.m == -INFINITY && b.m == -INFINITY) {
    r = a;
    r.i = min(a.i, b.i);
    return r;
  }
  const bool take_a = a.m > b.m || (a.m == b.m && a.i < b.i);
  r.m = take_a ? a.m : b.m;
  r.mb = take_a ? a.mb : b.mb;
  r.i = take_a ? a.i : b.i;
  r.s = (a.m == -INFINITY ? 0.f : a.s * ex2f(a.mb - r.mb)) +
        (b.m == -INFINITY ? 0.f : b.s * ex2f(b.mb - r.mb));
  return r;
}

template <typename T>
struct Vec;
template <>
struct Vec<uint16_t> {  // 8 bf16
  static constexpr int kN = 8;
  static __device__ __forceinline__ void unpack(const uint4& v, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ float scalar(const uint16_t* p) {
    return __uint_as_float((uint32_t)*p << 16);
  }
};
template <>
struct Vec<float> {  // 4 fp32
  static constexpr int kN = 4;
  static __device__ __forceinline__ void unpack(const uint4& v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ float scalar(const float* p) { return *p; }
};

// Add raw logits x[0..N) starting at vocabulary index `first` (increasing
// indices across calls of one thread, so a later equal maximum never wins).
template <int N>
__device__ __forceinline__ void add(Acc& a, const float (&x)[N], int first) {
  float cm = x[0];
#pragma unroll
  for (int k = 1; k < N; ++k) cm = fmaxf(cm, x[k]);
  if (cm > a.m) {
    int ci = 0;
#pragma unroll
    for (int k = N - 1; k >= 0; --k) ci = x[k] == cm ? k : ci;  // first index of the chunk maximum
    const float cmb = cm * kLog2e;
    a.s = a.m == -INFINITY ? 0.f : a.s * ex2f(a.mb - cmb);
    a.m = cm;
    a.mb = cmb;
    a.i = first + ci;
  }
  if (a.m != -INFINITY) {
    float t0 = 0.f, t1 = 0.f;
#pragma unroll
    for (int k = 0; k < N; k += 2) {
      t0 += ex2f(fmaf(x[k], kLog2e, -a.mb));
      t1 += ex2f(fmaf(x[k + 1], kLog2e, -a.mb));
    }
    a.s += t0 + t1;
  }
}

template <typename T>
__global__ void __launch_bounds__(kConfThreads) confidence_kernel(int64_t rows, int vocab,
                                                                  int64_t ld, const T* logits,
                                                                  int32_t* argmax, float* conf) {
  constexpr int N = Vec<T>::kN;
  __shared__ Acc s_acc[kConfThreads / 32];
  const int64_t r = blockIdx.x;
  if (r >= rows) return;
  const T* row = logits + r * ld;
  // elements before the first 16-byte boundary, then whole vectors, then the rest
  const int mis = (int)((reinterpret_cast<uintptr_t>(row) & 15) / sizeof(T));
  const int head = min(vocab, mis ? N - mis : 0);
  const uint4* rv = reinterpret_cast<const uint4*>(row + head);
  const int nvec = (vocab - head) / N;
  Acc a{-INFINITY, -INFINITY, 0.f, INT32_MAX};
  auto add1 = [&](int e) {
    const float x = Vec<T>::scalar(row + e);
    if (x > a.m) {
      const float xb = x * kLog2e;
      a.s = a.m == -INFINITY ? 0.f : a.s * ex2f(a.mb - xb);
      a.m = x;
      a.mb = xb;
      a.i = e;
    }
    if (a.m != -INFINITY) a.s += ex2f(fmaf(x, kLog2e, -a.mb));
  };
  if ((int)threadIdx.x < head) add1(threadIdx.x);
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kConfThreads * kUnroll) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * kConfThreads;
      if (v < nvec) buf[u] = __ldcs(rv + v);  // streamed once: do not keep in L1/L2
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * kConfThreads;
      if (v < nvec) {
        float x[N];
        Vec<T>::unpack(buf[u], x);
        add<N>(a, x, head + v * N);
      }
    }
  }
  // ragged end of the row: one element per thread
  for (int e = head + nvec * N + threadIdx.x; e < vocab; e += kConfThreads) add1(e);
  // block merge
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Acc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.mb = __shfl_xor_sync(0xffffffffu, a.mb, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    a = merge(a, b);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_acc[warp] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    Acc t = s_acc[0];
    for (int w = 1; w < kConfThreads / 32; ++w) t = merge(t, s_acc[w]);
    if (t.m == -INFINITY) {
      argmax[r] = 0;
      conf[r] = 0.f;
    } else {
      argmax[r] = t.i;
      conf[r] = 1.0f / t.s;
    }
  }
}

}  // namespace

cudaError_t launch_confidence(int64_t rows, int vocab, int64_t ld, int dtype, const void* logits,
                              int32_t* argmax, float* conf, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((unsigned)rows);
  if (dtype == 0)
    confidence_kernel<uint16_t><<<grid, kConfThreads, 0, stream>>>(
        rows, vocab, ld, static_cast<const uint16_t*>(logits), argmax, conf);
  else
    confidence_kernel<float><<<grid, kConfThreads, 0, stream>>>(
        rows, vocab, ld, static_cast<const float*>(logits), argmax, conf);
  return cudaGetLastError();
}

}  // namespace bca
