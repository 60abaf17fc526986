// Element access and online-softmax helpers shared by the verification
// kernels (vt_verify.cu, vt_verify_fused.cu).
#pragma once

#include "vt_common.cuh"

namespace vt {

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16-byte load
  __device__ static float load(const float* p) { return __ldg(p); }
  __device__ static void unpack16(uint4 v, float* x) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
  // eight consecutive elements at a 32-byte aligned index
  __device__ static void load8(const float* p, float* x) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    unpack16(__ldg(q), x);
    unpack16(__ldg(q + 1), x + 4);
  }
};
template <> struct Elem<uint16_t> {
  static constexpr int kVec = 8;
  __device__ static float load(const uint16_t* p) { return bf16_bits_to_float(__ldg(p)); }
  __device__ static void unpack16(uint4 v, float* x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  __device__ static void load8(const uint16_t* p, float* x) {
    unpack16(__ldg(reinterpret_cast<const uint4*>(p)), x);
  }
};

template <int N>
__device__ __forceinline__ void online_update(float& m, float& s, const float* x, float scale) {
  float t[N];
  float vmax = kNegBig;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    t[k] = x[k] * scale;
    vmax = fmaxf(vmax, t[k]);
  }
  if (vmax > m) {
    s *= exp2_approx(m - vmax);
    m = vmax;
  }
#pragma unroll
  for (int k = 0; k < N; ++k) s += exp2_approx(t[k] - m);
}

}  // namespace vt
