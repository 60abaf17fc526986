// Shared device helpers for libvt (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/vt.h"

#define VT_LOG2E 1.4426950408889634f

// Host-side: turn the last launch error into a status code.
#define VT_RETURN_IF_LAUNCH_FAILED()                 \
  do {                                               \
    cudaError_t e_ = cudaGetLastError();             \
    if (e_ != cudaSuccess) return VT_ERR_CUDA;       \
  } while (0)

#define VT_RETURN_IF_CUDA(call)                      \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return VT_ERR_CUDA;       \
  } while (0)

namespace vt {

// Most negative finite float: the "empty" running maximum of an online
// softmax.  Using a finite value keeps exp2(x - m) well defined when a
// segment holds only -inf logits.
constexpr float kNegBig = -3.402823466e38f;

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// A word that another thread block publishes by setting bit 31: re-read `p`
// (whose last value read is v) until bit 31 is set or `limit` reads have
// passed; returns the last value (bit 31 clear: the wait gave up).
__device__ __forceinline__ unsigned poll_published(const unsigned* p, unsigned v, uint32_t limit) {
  for (uint32_t it = 0; (v >> 31) == 0u && it < limit; ++it) v = ld_relaxed_u32(p);
  return v;
}

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// (m, s) pairs of an online softmax in base 2: s = sum 2^(x - m).
struct MS {
  float m;
  float s;
};

__device__ __forceinline__ MS ms_combine(MS a, MS b) {
  float m = fmaxf(a.m, b.m);
  float s = a.s * exp2_approx(a.m - m) + b.s * exp2_approx(b.m - m);
  return MS{m, s};
}

__device__ __forceinline__ MS warp_ms_reduce(MS v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS w;
    w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
    w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    v = ms_combine(v, w);
  }
  return v;
}

// Block-wide (m, s) reduction; result valid in every thread.
template <int NT>
__device__ __forceinline__ MS block_ms_reduce(MS v, MS* smem /* >= NT/32 */) {
  v = warp_ms_reduce(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) smem[warp] = v;
  __syncthreads();
  MS r = smem[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = ms_combine(r, smem[w]);
  __syncthreads();
  return r;
}

// Block-wide inclusive scan of one float per thread, in thread order.
// The association order is fixed by NT, so two calls on the same values give
// bit-identical results.  `excl` receives the exclusive prefix; the return
// value is the inclusive prefix; `total` the block total.
template <int NT>
__device__ __forceinline__ float block_scan_incl(float v, float* smem /* >= NT/32 */,
                                                 float& excl, float& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem[warp] = x;
  __syncthreads();
  float wpre = 0.f;
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    float t = smem[w];
    if (w < warp) wpre += t;
    tot += t;
  }
  __syncthreads();
  float incl = wpre + x;
  float up = __shfl_up_sync(0xffffffffu, x, 1);
  excl = wpre + (lane == 0 ? 0.f : up);
  total = tot;
  return incl;
}

__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int NT>
__device__ __forceinline__ int block_max_int(int v, int* smem) {
  v = warp_max_int(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) smem[warp] = v;
  __syncthreads();
  int r = smem[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = max(r, smem[w]);
  __syncthreads();
  return r;
}

template <int NT>
__device__ __forceinline__ int block_min_int(int v, int* smem) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) smem[warp] = v;
  __syncthreads();
  int r = smem[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = min(r, smem[w]);
  __syncthreads();
  return r;
}

// Programmatic dependent launch: wait until the previous kernel in the stream
// has completed and its writes are visible / let the next kernel launch.
// Both are no-ops for kernels launched without the attribute.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

}  // namespace vt
