// Batched speculative verification (modified rejection sampling) on sm_103a.
//
// Operation (pages: "Speculative decoding" glossary, "Why a rejection needs a
// special draw" and "Propose a block, keep a prefix"; "A rejection rule keeps
// speculative decoding's output exact", "Extending the rule from one token to
// a drafted run"):
//   p_i = softmax(l[b,i,:] / T) for i = 0..gamma;  accept drafted x_i iff
//   u_acc < min(1, p_i(x_i)/q_i(x_i)), left to right, stop at the first
//   rejection n; draw t from norm(max(p_n - q_n, 0)) (or from p_gamma when
//   n = gamma) by a strict inverse CDF in ascending token-id order.
//
// Two kernels:
//  1. verify_stats  grid (B*(gamma+1) rows, C1 chunks): one HBM pass over the
//     logits, 128-bit loads, base-2 online softmax (max, sum 2^(x-max)) per
//     chunk.  This is the pass that moves almost all of the bytes.
//  2. verify_finish grid (B, C2 chunks): every CTA of sequence b merges the
//     chunk partials of its gamma+1 rows, replays the accept walk (a few
//     scalar loads), then computes the residual mass of its chunk of row n_b
//     (an L2 re-read of one row per sequence).  The last CTA of b to finish
//     (atomic ticket; no CTA ever waits on another) picks the chunk where the
//     running mass crosses u * Z and scans that chunk in id order.
// The chunk sums and the final scan run the same per-tile block scan, so the
// running sums the selection compares are bit-identical in both places.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kMaxGamma = 64;
constexpr int kMaxChunks1 = 64;
constexpr int kMaxChunks2 = 64;
constexpr int kNT1 = 256;
constexpr int kNT2 = 256;

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16-byte load
  __device__ static float load(const float* p) { return __ldg(p); }
  __device__ static void unpack16(uint4 v, float* x) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
  // four consecutive elements at an index that is a multiple of 4
  __device__ static void load4(const float* p, float* x) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
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
  __device__ static void load4(const uint16_t* p, float* x) {
    uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
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

// ---------------------------------------------------------------- kernel 1
template <typename T, int NT, int U>
__global__ void __launch_bounds__(NT)
verify_stats_kernel(const T* __restrict__ logits, int64_t V, int64_t chunk_len, int nchunk,
                    float scale, float2* __restrict__ part, int* __restrict__ counters, int B,
                    int* __restrict__ dev_status, int vec_ok) {
  __shared__ MS red[NT / 32];
  const int64_t row = blockIdx.x;
  const int c = blockIdx.y;
  if (row == 0 && c == 0) {
    // reset the per-sequence tickets of kernel 2 and the status word; kernel 2
    // starts only after this grid has completed (same stream)
    for (int i = threadIdx.x; i < B; i += NT) counters[i] = 0;
    if (threadIdx.x == 0) *dev_status = 0;
  }
  const T* rp = logits + row * V;
  const int64_t j0 = (int64_t)c * chunk_len;
  const int64_t j1 = min(V, j0 + chunk_len);
  float m = kNegBig, s = 0.f;
  int64_t jt = j0;  // start of the scalar tail
  if (vec_ok && j1 > j0) {
    constexpr int VEC = Elem<T>::kVec;
    const int64_t nv = (j1 - j0) / VEC;
    const uint4* vp = reinterpret_cast<const uint4*>(rp + j0);
    for (int64_t v = threadIdx.x; v < nv; v += (int64_t)NT * U) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t vi = v + (int64_t)u * NT;
        if (vi < nv) raw[u] = __ldg(vp + vi);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t vi = v + (int64_t)u * NT;
        if (vi < nv) {
          float x[VEC];
          Elem<T>::unpack16(raw[u], x);
          online_update<VEC>(m, s, x, scale);
        }
      }
    }
    jt = j0 + nv * VEC;
  }
  for (int64_t j = jt + threadIdx.x; j < j1; j += NT) {
    float x = Elem<T>::load(rp + j);
    online_update<1>(m, s, &x, scale);
  }
  MS r = block_ms_reduce<NT>(MS{m, s}, red);
  if (threadIdx.x == 0) part[row * nchunk + c] = make_float2(r.m, r.s);
}

// ---------------------------------------------------------------- kernel 2
struct FinishArgs {
  const void* logits;
  int64_t V;
  int B, gamma, K;
  const float* q;
  const int* inv_map;
  const int* draft;
  const float* u_acc;
  const float* u_res;
  float scale;  // log2(e) / T
  const float2* part;
  int nchunk1;
  float* zpart;
  int* lpart;
  int nchunk2;
  int64_t chunk2_len;
  int* counters;
  int* out_tokens;
  int* out_n;
  float* out_accept_prob;
  int* dev_status;
  int vec_ok;
};

// Residual weights r_j = max(p_j - q_j, 0) for j, j+1, j+2, j+3 (zero past j1).
// qrow == nullptr means q is identically zero (bonus draw: r = p).
template <typename T>
__device__ __forceinline__ void residual4(const T* __restrict__ rowp, const int* __restrict__ inv_map,
                                          const float* __restrict__ qrow, int K, int64_t j,
                                          int64_t j1, float scale, float m, float invS, bool vec,
                                          float* r) {
  float x[4];
  if (vec && j + 3 < j1) {
    Elem<T>::load4(rowp + j, x);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = (j + e < j1) ? Elem<T>::load(rowp + j + e) : 0.f;
  }
  int k[4] = {-1, -1, -1, -1};
  if (qrow != nullptr) {
    if (vec && j + 3 < j1) {
      int4 v = __ldg(reinterpret_cast<const int4*>(inv_map + j));
      k[0] = v.x; k[1] = v.y; k[2] = v.z; k[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) k[e] = (j + e < j1) ? __ldg(inv_map + j + e) : -1;
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float pj = exp2_approx(x[e] * scale - m) * invS;
    float qj = (k[e] >= 0 && k[e] < K) ? __ldg(qrow + k[e]) : 0.f;
    r[e] = (j + e < j1) ? fmaxf(pj - qj, 0.f) : 0.f;
  }
}

// Sum of r over [j0, j1) by tiles of NT*4, with the fixed association order
// shared by scan_select.  Also returns the last index with r > 0 (or -1).
template <typename T, int NT>
__device__ float scan_total(const T* rowp, const int* inv_map, const float* qrow, int K, int64_t j0,
                            int64_t j1, float scale, float m, float invS, bool vec, float* sred,
                            int* ired, int& lastpos) {
  float run = 0.f;
  int lp = -1;
  for (int64_t base = j0; base < j1; base += (int64_t)NT * 4) {
    const int64_t j = base + 4 * (int64_t)threadIdx.x;
    float r[4];
    residual4<T>(rowp, inv_map, qrow, K, j, j1, scale, m, invS, vec, r);
    const float t4 = ((r[0] + r[1]) + r[2]) + r[3];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (r[e] > 0.f) lp = (int)(j + e);
    float excl, tot;
    block_scan_incl<NT>(t4, sred, excl, tot);
    run += tot;
  }
  lastpos = block_max_int<NT>(lp, ired);
  return run;
}

// Smallest j in [j0, j1) whose running residual sum (from j0) exceeds
// `target`; -1 if the running sum never does.  `lastpos` gets the last j with
// r_j > 0 in the range.
template <typename T, int NT>
__device__ int scan_select(const T* rowp, const int* inv_map, const float* qrow, int K, int64_t j0,
                           int64_t j1, float scale, float m, float invS, bool vec, float target,
                           float* sred, int* ired, int* s_pick, int& lastpos) {
  float run = 0.f;
  int lp = -1;
  if (threadIdx.x == 0) *s_pick = -1;
  __syncthreads();
  for (int64_t base = j0; base < j1; base += (int64_t)NT * 4) {
    const int64_t j = base + 4 * (int64_t)threadIdx.x;
    float r[4];
    residual4<T>(rowp, inv_map, qrow, K, j, j1, scale, m, invS, vec, r);
    const float t4 = ((r[0] + r[1]) + r[2]) + r[3];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (r[e] > 0.f) lp = (int)(j + e);
    float excl, tot;
    const float incl = block_scan_incl<NT>(t4, sred, excl, tot);
    const bool hit = (run + incl > target);
    const int first = block_min_int<NT>(hit ? (int)threadIdx.x : NT, ired);
    if (first < NT) {
      if ((int)threadIdx.x == first) {
        float acc = run + excl;
        int pick = -1, lastp = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (r[e] > 0.f) lastp = (int)(j + e);
          acc += r[e];
          if (pick < 0 && acc > target) pick = (int)(j + e);
        }
        *s_pick = (pick >= 0) ? pick : lastp;
      }
      __syncthreads();
      break;  // `first` is uniform across the block
    }
    run += tot;
  }
  lastpos = block_max_int<NT>(lp, ired);
  return *s_pick;
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT) verify_finish_kernel(FinishArgs a) {
  __shared__ float s_m[kMaxGamma + 1], s_S[kMaxGamma + 1];
  __shared__ float sred[NT / 32];
  __shared__ int ired[NT / 32];
  __shared__ int s_n, s_flags, s_last, s_pick, s_sel, s_cstar;
  __shared__ float s_target;

  const int b = blockIdx.x;
  const int c = blockIdx.y;
  const int R = a.gamma + 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* logits = static_cast<const T*>(a.logits);

  // 1. merge the chunk partials of this sequence's gamma+1 rows
  for (int i = warp; i < R; i += NT / 32) {
    MS v{kNegBig, 0.f};
    const float2* pp = a.part + ((int64_t)b * R + i) * a.nchunk1;
    for (int k = lane; k < a.nchunk1; k += 32) {
      float2 t = pp[k];
      v = ms_combine(v, MS{t.x, t.y});
    }
    v = warp_ms_reduce(v);
    if (lane == 0) {
      s_m[i] = v.m;
      s_S[i] = v.s;
    }
  }
  __syncthreads();

  // 2. the accept walk (identical in every CTA of this sequence)
  if (threadIdx.x == 0) {
    int flags = 0, n = 0, tested = 0;
    for (int i = 0; i < R; ++i)
      if (!(s_S[i] > 0.f && isfinite(s_S[i]) && isfinite(s_m[i]))) flags |= VT_DEV_NONFINITE;
    if (!flags) {
      for (int i = 0; i < a.gamma; ++i) {
        const int x = a.draft[(int64_t)b * a.gamma + i];
        if (x < 0 || x >= a.V) { flags |= VT_DEV_BAD_DRAFT; break; }
        const int k = a.inv_map[x];
        if (k < 0 || k >= a.K) { flags |= VT_DEV_BAD_DRAFT; break; }
        const float qx = a.q[((int64_t)b * a.gamma + i) * a.K + k];
        if (!(qx > 0.f) || !isfinite(qx)) { flags |= VT_DEV_BAD_DRAFT; break; }
        const float lx = Elem<T>::load(logits + ((int64_t)b * R + i) * a.V + x);
        const float px = exp2_approx(lx * a.scale - s_m[i]) / s_S[i];
        const float acc = fminf(1.f, px / qx);
        if (c == 0 && a.out_accept_prob) a.out_accept_prob[(int64_t)b * a.gamma + i] = acc;
        tested = i + 1;
        if (a.u_acc[(int64_t)b * a.gamma + i] < acc) {
          n = i + 1;
        } else {
          break;
        }
      }
    }
    if (c == 0 && a.out_accept_prob)
      for (int i = tested; i < a.gamma; ++i)
        a.out_accept_prob[(int64_t)b * a.gamma + i] = __int_as_float(0x7fc00000);
    s_n = n;
    s_flags = flags;
  }
  __syncthreads();
  const int n = s_n;
  const int flags = s_flags;
  if (flags & (VT_DEV_BAD_DRAFT | VT_DEV_NONFINITE)) {
    if (c == 0) {
      for (int i = threadIdx.x; i < R; i += NT) a.out_tokens[(int64_t)b * R + i] = -1;
      if (threadIdx.x == 0) {
        a.out_n[b] = 0;
        atomicOr(a.dev_status, flags);
      }
    }
    return;
  }

  // 3. residual (n < gamma) or bonus (n == gamma) mass of this chunk of row n
  const T* rowp = logits + ((int64_t)b * R + n) * a.V;
  const float m_n = s_m[n];
  const float invS = 1.f / s_S[n];
  const float* qrow = (n < a.gamma) ? a.q + ((int64_t)b * a.gamma + n) * a.K : nullptr;
  const bool vec = a.vec_ok != 0;
  {
    const int64_t j0 = (int64_t)c * a.chunk2_len;
    const int64_t j1 = min(a.V, j0 + a.chunk2_len);
    int lp;
    const float z = scan_total<T, NT>(rowp, a.inv_map, qrow, a.K, j0, j1, a.scale, m_n, invS, vec,
                                      sred, ired, lp);
    if (threadIdx.x == 0) {
      a.zpart[(int64_t)b * a.nchunk2 + c] = z;
      a.lpart[(int64_t)b * a.nchunk2 + c] = lp;
      __threadfence();
      s_last = (atomicAdd(a.counters + b, 1) == a.nchunk2 - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }

  // 4. last CTA of sequence b: pick the chunk, then the token
  if (threadIdx.x == 0) {
    const float* zp = a.zpart + (int64_t)b * a.nchunk2;
    float total = 0.f;
    for (int k = 0; k < a.nchunk2; ++k) total += __ldcg(zp + k);
    const float target = a.u_res[(int64_t)b * R + n] * total;
    float pre = 0.f;
    int cstar = -1;
    if (total > 0.f) {
      for (int k = 0; k < a.nchunk2; ++k) {
        const float zk = __ldcg(zp + k);
        if (pre + zk > target) { cstar = k; break; }
        pre += zk;
      }
    }
    s_cstar = cstar;
    s_target = target - pre;
    int glast = -1;
    for (int k = 0; k < a.nchunk2; ++k) glast = max(glast, __ldcg(a.lpart + (int64_t)b * a.nchunk2 + k));
    s_pick = (total > 0.f) ? glast : -2;  // -2: zero residual mass
  }
  __syncthreads();
  int token = s_pick;
  int extra_flags = 0;
  if (token == -2) {
    // residual mass is zero (only through rounding): draw from p_n instead
    extra_flags = VT_DEV_ZERO_RESIDUAL;
    int lp;
    const float tp = scan_total<T, NT>(rowp, a.inv_map, nullptr, a.K, 0, a.V, a.scale, m_n, invS, vec,
                                       sred, ired, lp);
    const float target = a.u_res[(int64_t)b * R + n] * tp;
    int lp2;
    const int t = scan_select<T, NT>(rowp, a.inv_map, nullptr, a.K, 0, a.V, a.scale, m_n, invS, vec,
                                     target, sred, ired, &s_sel, lp2);
    token = (t >= 0) ? t : lp;
  } else if (s_cstar >= 0) {
    const int64_t j0 = (int64_t)s_cstar * a.chunk2_len;
    const int64_t j1 = min(a.V, j0 + a.chunk2_len);
    const int glast = token;
    int lpc;
    const int t = scan_select<T, NT>(rowp, a.inv_map, qrow, a.K, j0, j1, a.scale, m_n, invS, vec,
                                     s_target, sred, ired, &s_sel, lpc);
    token = (t >= 0) ? t : (lpc >= 0 ? lpc : glast);
  }
  // (s_cstar < 0 with positive mass: u*Z rounded to the top; token = last
  //  index with positive residual, already in `token`)

  for (int i = threadIdx.x; i < R; i += NT) {
    int v = -1;
    if (i < n) v = a.draft[(int64_t)b * a.gamma + i];
    else if (i == n) v = token;
    a.out_tokens[(int64_t)b * R + i] = v;
  }
  if (threadIdx.x == 0) {
    a.out_n[b] = n;
    if (extra_flags) atomicOr(a.dev_status, extra_flags);
    a.counters[b] = 0;
  }
}

int num_sms_of_current_device() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

struct VerifyPlan {
  int nchunk1;
  int64_t chunk1;
  int nchunk2;
  int64_t chunk2;
};

VerifyPlan plan_verify(int64_t rows, int B, int64_t V, int vec, int num_sms) {
  VerifyPlan p;
  // kernel 1: about two waves of 8 resident 256-thread CTAs per SM, chunks of
  // at least 4096 elements, aligned to the 16-byte vector width
  const int64_t want = (int64_t)num_sms * 16;
  int64_t c1 = (want + rows - 1) / rows;
  c1 = std::max<int64_t>(1, std::min<int64_t>(c1, kMaxChunks1));
  c1 = std::min<int64_t>(c1, std::max<int64_t>(1, V / 4096));
  int64_t len1 = (V + c1 - 1) / c1;
  len1 = (len1 + vec - 1) / vec * vec;
  p.chunk1 = len1;
  p.nchunk1 = (int)((V + len1 - 1) / len1);
  // kernel 2: about four CTAs per SM in total, at least one 1024-element tile
  int64_t c2 = ((int64_t)num_sms * 4 + B - 1) / B;
  c2 = std::max<int64_t>(1, std::min<int64_t>(c2, kMaxChunks2));
  c2 = std::min<int64_t>(c2, std::max<int64_t>(1, V / 1024));
  int64_t len2 = (V + c2 - 1) / c2;
  len2 = (len2 + 3) / 4 * 4;
  p.chunk2 = len2;
  p.nchunk2 = (int)((V + len2 - 1) / len2);
  return p;
}

struct VerifyWs {
  float2* part;
  float* zpart;
  int* lpart;
  int* counters;
  size_t bytes;
};

VerifyWs carve_verify(void* base, int64_t rows, int B) {
  VerifyWs w;
  size_t off = 0;
  auto take = [&](size_t n) {
    size_t o = off;
    off = align_up(off + n, 256);
    return o;
  };
  size_t o_part = take((size_t)rows * kMaxChunks1 * sizeof(float2));
  size_t o_z = take((size_t)B * kMaxChunks2 * sizeof(float));
  size_t o_l = take((size_t)B * kMaxChunks2 * sizeof(int));
  size_t o_c = take((size_t)B * sizeof(int));
  char* p = static_cast<char*>(base);
  w.part = reinterpret_cast<float2*>(p + o_part);
  w.zpart = reinterpret_cast<float*>(p + o_z);
  w.lpart = reinterpret_cast<int*>(p + o_l);
  w.counters = reinterpret_cast<int*>(p + o_c);
  w.bytes = off;
  return w;
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_verify_workspace_bytes(int32_t B, int32_t gamma, int32_t V, int32_t K) {
  (void)V;
  (void)K;
  if (B < 1 || gamma < 1) return 0;
  return vt::carve_verify(nullptr, (int64_t)B * (gamma + 1), B).bytes;
}

extern "C" int vt_verify(const void* target_logits, int32_t logits_dtype, int32_t B, int32_t gamma,
                         int32_t V, const float* q, const int32_t* inv_map, int32_t K,
                         const int32_t* draft_tokens, const float* u_accept,
                         const float* u_resample, float temperature, int32_t* out_tokens,
                         int32_t* out_num_accepted, float* out_accept_prob, int32_t* dev_status,
                         void* workspace, size_t workspace_bytes, void* stream) {
  using namespace vt;
  if (!target_logits || !q || !inv_map || !draft_tokens || !u_accept || !u_resample ||
      !out_tokens || !out_num_accepted || !dev_status)
    return VT_ERR_INVALID_ARG;
  if (B < 1 || gamma < 1 || gamma > kMaxGamma || V < 1 || K < 1 || K > V) return VT_ERR_INVALID_ARG;
  if (logits_dtype != VT_F32 && logits_dtype != VT_BF16) return VT_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return VT_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)B * (gamma + 1);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  VerifyWs ws = carve_verify(workspace, rows, B);
  if (workspace_bytes < ws.bytes) return VT_ERR_WORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t esize = (logits_dtype == VT_F32) ? 4 : 2;
  const int vec_elems = (logits_dtype == VT_F32) ? 4 : 8;
  // 16-byte loads need every row to start on a 16-byte boundary; the residual
  // pass also loads inv_map four ids at a time
  const int vec_ok = ((reinterpret_cast<uintptr_t>(target_logits) & 15) == 0) &&
                     (((int64_t)V * esize) % 16 == 0) &&
                     ((reinterpret_cast<uintptr_t>(inv_map) & 15) == 0);
  VerifyPlan plan = plan_verify(rows, B, V, vec_elems, num_sms_of_current_device());
  const float scale = VT_LOG2E / temperature;

  dim3 g1((unsigned)rows, (unsigned)plan.nchunk1);
  if (logits_dtype == VT_F32) {
    verify_stats_kernel<float, kNT1, 4><<<g1, kNT1, 0, s>>>(
        static_cast<const float*>(target_logits), V, plan.chunk1, plan.nchunk1, scale, ws.part,
        ws.counters, B, dev_status, vec_ok);
  } else {
    verify_stats_kernel<uint16_t, kNT1, 4><<<g1, kNT1, 0, s>>>(
        static_cast<const uint16_t*>(target_logits), V, plan.chunk1, plan.nchunk1, scale, ws.part,
        ws.counters, B, dev_status, vec_ok);
  }
  VT_RETURN_IF_LAUNCH_FAILED();

  FinishArgs fa;
  fa.logits = target_logits;
  fa.V = V;
  fa.B = B;
  fa.gamma = gamma;
  fa.K = K;
  fa.q = q;
  fa.inv_map = inv_map;
  fa.draft = draft_tokens;
  fa.u_acc = u_accept;
  fa.u_res = u_resample;
  fa.scale = scale;
  fa.part = ws.part;
  fa.nchunk1 = plan.nchunk1;
  fa.zpart = ws.zpart;
  fa.lpart = ws.lpart;
  fa.nchunk2 = plan.nchunk2;
  fa.chunk2_len = plan.chunk2;
  fa.counters = ws.counters;
  fa.out_tokens = out_tokens;
  fa.out_n = out_num_accepted;
  fa.out_accept_prob = out_accept_prob;
  fa.dev_status = dev_status;
  fa.vec_ok = vec_ok;
  dim3 g2((unsigned)B, (unsigned)plan.nchunk2);
  if (logits_dtype == VT_F32) {
    verify_finish_kernel<float, kNT2><<<g2, kNT2, 0, s>>>(fa);
  } else {
    verify_finish_kernel<uint16_t, kNT2><<<g2, kNT2, 0, s>>>(fa);
  }
  VT_RETURN_IF_LAUNCH_FAILED();
  return VT_OK;
}

// ---------------------------------------------------------------------------
// vt_verify_noalloc: the same verification with its scratch in a static
// device array instead of a caller-provided workspace, for callers that have
// no device allocator to call (a plug-in inside a runtime that owns all
// device memory, allocator-free C code, a loop that must not risk
// cudaMalloc's device-wide synchronisation).  All calls on a device share the
// array; overlapping calls race on it.
namespace vt {
namespace {

constexpr int kNoallocMaxDevices = 64;

// 2 MiB of scratch per device, resident for the life of the process.
static __device__ __align__(256) unsigned char g_noalloc_scratch[VT_VERIFY_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  Host code only
// holds a stand-in for the symbol, so the address is looked up once per
// device (with that device current) and cached.
int noalloc_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kNoallocMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VT_ERR_CUDA;
  if (dev < 0 || dev >= kNoallocMaxDevices) return VT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return VT_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return VT_OK;
}

}  // namespace
}  // namespace vt

extern "C" int vt_verify_noalloc(const void* target_logits, int32_t logits_dtype, int32_t B,
                                 int32_t gamma, int32_t V, const float* q,
                                 const int32_t* inv_map, int32_t K, const int32_t* draft_tokens,
                                 const float* u_accept, const float* u_resample,
                                 float temperature, int32_t* out_tokens,
                                 int32_t* out_num_accepted, float* out_accept_prob,
                                 int32_t* dev_status, void* stream) {
  using namespace vt;
  if (B < 1 || gamma < 1 || gamma > kMaxGamma) return VT_ERR_INVALID_ARG;
  const size_t need = vt_verify_workspace_bytes(B, gamma, V, K);
  if (need > VT_VERIFY_NOALLOC_SCRATCH_BYTES) return VT_ERR_SCRATCH_LIMIT;
  if (!target_logits || !q || !inv_map || !draft_tokens || !u_accept || !u_resample ||
      !out_tokens || !out_num_accepted || !dev_status)
    return VT_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int st = noalloc_scratch_address(&scratch);
  if (st != VT_OK) return st;
  return vt_verify(target_logits, logits_dtype, B, gamma, V, q, inv_map, K, draft_tokens,
                   u_accept, u_resample, temperature, out_tokens, out_num_accepted,
                   out_accept_prob, dev_status, scratch, VT_VERIFY_NOALLOC_SCRATCH_BYTES, stream);
}
