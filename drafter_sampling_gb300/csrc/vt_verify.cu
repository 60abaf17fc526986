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
// Design (one GPU; the logits are read once from HBM):
//  * verify_stats, grid (B*(gamma+1) rows, C1 chunks of 32 KB): 16-byte loads,
//    eight in flight per thread, base-2 online softmax (max, sum 2^(x-max))
//    per chunk, written as a partial.  The first chunk of each drafted row
//    also gathers the drafted token's scaled logit and its draft probability
//    q(x), and block (0,0) clears the finish kernel's tickets.
//  * verify_finish, grid (B, runs of consecutive 2048-id tiles): merges the
//    row partials, replays the accept walk for all positions at once (first
//    failing position = n), sums max(p_n - q_n, 0) over each of its tiles
//    (an L2 re-read of one row per sequence) and publishes the tile sums.
//    The last CTA of a sequence to finish (atomic ticket; nothing waits)
//    finds the tile where the running sum passes u * Z and rescans it to
//    draw the token.
//  * Both kernels are launched with programmatic dependent launch: each one
//    waits (griddepcontrol.wait) before touching data an earlier kernel
//    wrote, and releases its successor near its end, so the successor's
//    launch and start-up overlap this kernel's tail.  The finish kernel
//    fetches its inv_map tile and uniforms before that wait.
// The tile sums and the final rescan use the same per-thread sums and the
// same block scan, so the running sums the selection compares are
// bit-identical in both places.
#include <algorithm>
#include <cmath>

#include "vt_common.cuh"
#include "vt_internal.h"
#include "vt_verify_common.cuh"

namespace vt {
namespace {

constexpr int kMaxGamma = 64;
constexpr int kNT = 256;              // threads per CTA (main kernel)
constexpr int kResPerThread = 8;      // residual ids per thread
constexpr int kResChunk = kNT * kResPerThread;
constexpr int kStatsBytes = 32768;    // bytes of logits per stats item
constexpr int kMaxChunks1 = 64;
constexpr int kMaxTpc = 64;           // residual tiles per finish CTA at most

struct VArgs {
  const void* logits;
  int64_t V;
  int B, gamma, R, K;
  const float* q;
  const int* inv_map;
  const int* draft;
  const float* u_acc;
  const float* u_res;
  float scale;   // log2(e) / T
  int C1;        // stats chunks per row
  int64_t len1;  // ids per stats chunk (multiple of the vector width)
  int C2;        // residual tiles per sequence (kResChunk ids each)
  int tpc;       // residual tiles per finish CTA (consecutive)
  int nfin;      // finish CTAs per sequence = ceil(C2 / tpc)
  float2* part;  // [B*R][C1]
  float2* pre;   // [B][gamma]: (scaled logit at x, q(x)); q(x) = -1 if invalid
  float* zpart;  // [B][C2]
  int* lpart;    // [B][C2]
  unsigned* rdone;  // [B]
  int* out_tokens;
  int* out_n;
  float* out_accept_prob;
  int* dev_status;
  int vec_ok;
};

// -------------------------------------------------------------- kernel 1
template <typename T>
__global__ void __launch_bounds__(kNT) verify_stats_kernel(VArgs a) {
  __shared__ MS mred[kNT / 32];
  constexpr int VEC = Elem<T>::kVec;
  constexpr int U = kStatsBytes / 16 / kNT;  // 16-byte loads per thread per pass
  griddep_wait();  // inputs written by earlier work are complete and visible
  const int64_t row = blockIdx.x;
  const int c = blockIdx.y;
  const int b = (int)(row / a.R), i = (int)(row - (int64_t)b * a.R);
  if (row == 0 && c == 0) {
    for (int k = threadIdx.x; k < a.B; k += kNT) a.rdone[k] = 0;
    if (threadIdx.x == 0) *a.dev_status = 0;
  }
  const T* rp = static_cast<const T*>(a.logits) + row * a.V;
  const int64_t j0 = (int64_t)c * a.len1;
  const int64_t j1 = min(a.V, j0 + a.len1);
  float m = kNegBig, s = 0.f;
  int64_t jt = j0;
  const bool gather = (c == 0 && i < a.gamma && threadIdx.x == 0);
  float2 pv = make_float2(0.f, -1.f);
  if (a.vec_ok) {
    const int64_t nv = (j1 - j0) / VEC;
    const uint4* vp = reinterpret_cast<const uint4*>(rp + j0);
    for (int64_t v = threadIdx.x; v < nv; v += (int64_t)kNT * U) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t vi = v + (int64_t)u * kNT;
        if (vi < nv) raw[u] = __ldg(vp + vi);
      }
      if (gather && v == threadIdx.x) {
        // drafted token of this row: its logit and q(x), while the loads fly
        const int x = a.draft[(int64_t)b * a.gamma + i];
        if (x >= 0 && x < a.V) {
          const int k = a.inv_map[x];
          if (k >= 0 && k < a.K) {
            const float qx = a.q[((int64_t)b * a.gamma + i) * a.K + k];
            if (qx > 0.f && isfinite(qx)) pv = make_float2(Elem<T>::load(rp + x) * a.scale, qx);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t vi = v + (int64_t)u * kNT;
        if (vi < nv) {
          float x[VEC];
          Elem<T>::unpack16(raw[u], x);
          online_update<VEC>(m, s, x, a.scale);
        }
      }
    }
    jt = j0 + nv * VEC;
  }
  for (int64_t j = jt + threadIdx.x; j < j1; j += kNT) {
    float x = Elem<T>::load(rp + j);
    online_update<1>(m, s, &x, a.scale);
  }
  if (gather && !a.vec_ok) {
    const int x = a.draft[(int64_t)b * a.gamma + i];
    if (x >= 0 && x < a.V) {
      const int k = a.inv_map[x];
      if (k >= 0 && k < a.K) {
        const float qx = a.q[((int64_t)b * a.gamma + i) * a.K + k];
        if (qx > 0.f && isfinite(qx)) pv = make_float2(Elem<T>::load(rp + x) * a.scale, qx);
      }
    }
  }
  griddep_launch_dependents();
  const MS r = block_ms_reduce<kNT>(MS{m, s}, mred);
  if (threadIdx.x == 0) a.part[row * a.C1 + c] = make_float2(r.m, r.s);
  if (gather) a.pre[(int64_t)b * a.gamma + i] = pv;
}

// -------------------------------------------------------- residual tiles
// the eight inv_map entries of thread tid's ids in the tile at j0
__device__ __forceinline__ void load_kmap(const VArgs& a, int64_t j, int* k) {
  if (a.vec_ok && j + 8 <= a.V) {
    const int4* ip = reinterpret_cast<const int4*>(a.inv_map + j);
    const int4 v0 = __ldg(ip), v1 = __ldg(ip + 1);
    k[0] = v0.x; k[1] = v0.y; k[2] = v0.z; k[3] = v0.w;
    k[4] = v1.x; k[5] = v1.y; k[6] = v1.z; k[7] = v1.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) k[e] = (j + e < a.V) ? __ldg(a.inv_map + j + e) : -1;
  }
}

// the logits at ids j..j+7 of one row (zero past V)
template <typename T>
__device__ __forceinline__ void load_logits8(const VArgs& a, const T* rowp, int64_t j, float* x) {
  if (a.vec_ok && j + 8 <= a.V) {
    Elem<T>::load8(rowp + j, x);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (j + e < a.V) ? Elem<T>::load(rowp + j + e) : 0.f;
  }
}

// q at the trimmed indices k[0..7] (zero where an id is not kept, or
// qrow == nullptr)
__device__ __forceinline__ void gather_q8(const VArgs& a, const float* qrow, const int* k,
                                          float* qv) {
#pragma unroll
  for (int e = 0; e < 8; ++e)
    qv[e] = (qrow != nullptr && k[e] >= 0 && k[e] < a.K) ? __ldg(qrow + k[e]) : 0.f;
}

// r_e = max(p - q, 0) at ids j..j+7 from their logits and q (zero past V)
__device__ __forceinline__ void residual_of(const VArgs& a, const float* x, const float* qv,
                                            int64_t j, float m, float invS, float* r) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float pj = exp2_approx(x[e] * a.scale - m) * invS;
    r[e] = (j + e < a.V) ? fmaxf(pj - qv[e], 0.f) : 0.f;
  }
}

// r_e = max(p - q, 0) at ids j..j+7 (zero past V); qrow == nullptr: q = 0
template <typename T>
__device__ __forceinline__ void residual8k(const VArgs& a, const T* rowp, const float* qrow,
                                           int64_t j, float m, float invS, const int* k, float* r) {
  float x[8], qv[8];
  load_logits8<T>(a, rowp, j, x);
  gather_q8(a, qrow, k, qv);
  residual_of(a, x, qv, j, m, invS, r);
}

__device__ __forceinline__ float sum8(const float* r) {
  float s = r[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) s += r[e];
  return s;
}

struct Smem {
  float m[kMaxGamma + 1];
  float S[kMaxGamma + 1];
  float sred[kNT / 32];
  int ired[kNT / 32];
  unsigned fail[2];
  int last;
  int n;
  int flags;
  int pick;
  int cstar;
  float target;
  float tsum[kMaxTpc][kNT / 32];  // warp totals of each of the CTA's tiles
  float zbuf[kResChunk];  // tile sums of one sequence (selection)
};

// Inclusive/exclusive prefix of this thread's eight residuals within the tile
// and the tile total (fixed association order).
template <typename T>
__device__ __forceinline__ float tile_scan(const VArgs& a, const T* rowp, const float* qrow,
                                           int64_t j0, float m, float invS, const int* k, Smem& sm,
                                           float* r, float& excl, float& tot, int& lastpos) {
  const int64_t j = j0 + (int64_t)kResPerThread * threadIdx.x;
  residual8k<T>(a, rowp, qrow, j, m, invS, k, r);
  lastpos = -1;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (r[e] > 0.f) lastpos = (int)(j + e);
  return block_scan_incl<kNT>(sum8(r), sm.sred, excl, tot);
}

// First id of the tile at j0 whose running residual sum (from j0) exceeds
// `target`, or -1.  Uniform across the block.
template <typename T>
__device__ int select_in_tile(const VArgs& a, const T* rowp, const float* qrow, int64_t j0,
                              float m, float invS, float target, Smem& sm, int& lastpos) {
  int k[8];
  load_kmap(a, j0 + (int64_t)kResPerThread * threadIdx.x, k);
  float r[8], excl, tot;
  int lp;
  const float incl = tile_scan<T>(a, rowp, qrow, j0, m, invS, k, sm, r, excl, tot, lp);
  lastpos = block_max_int<kNT>(lp, sm.ired);
  const int first = block_min_int<kNT>(incl > target ? (int)threadIdx.x : kNT, sm.ired);
  if (threadIdx.x == 0) sm.pick = -1;
  __syncthreads();
  if ((int)threadIdx.x == first) {
    const int64_t j = j0 + (int64_t)kResPerThread * threadIdx.x;
    float acc = excl;
    int pk = -1, lastp = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (r[e] > 0.f) lastp = (int)(j + e);
      acc += r[e];
      if (pk < 0 && acc > target) pk = (int)(j + e);
    }
    sm.pick = (pk >= 0) ? pk : lastp;
  }
  __syncthreads();
  return sm.pick;
}

// -------------------------------------------------------------- kernel 2
template <typename T>
__global__ void __launch_bounds__(kNT, 4) verify_finish_kernel(VArgs a) {
  __shared__ Smem sm;
  const int b = blockIdx.x, c = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R;
  // this CTA's residual tiles [c0, c1)
  const int c0 = c * a.tpc, c1 = min(a.C2, c0 + a.tpc);
  // inputs that no earlier kernel of this call writes: fetch before waiting
  int kmap[8];
  load_kmap(a, (int64_t)c0 * kResChunk + (int64_t)kResPerThread * tid, kmap);
  const float ua = (tid < a.gamma) ? a.u_acc[(int64_t)b * a.gamma + tid] : 0.f;
  griddep_wait();  // the stats kernel has completed
  // the drafted tokens' (logit, q) pairs, requested with the partials below
  float2 pr = make_float2(0.f, -1.f);
  if (tid < a.gamma) pr = a.pre[(int64_t)b * a.gamma + tid];

  // 1. merge the row partials of the gamma+1 rows
  for (int i = warp; i < R; i += kNT / 32) {
    MS v{kNegBig, 0.f};
    const float2* pp = a.part + ((int64_t)b * R + i) * a.C1;
    for (int k = lane; k < a.C1; k += 32) {
      const float2 t = pp[k];
      v = ms_combine(v, MS{t.x, t.y});
    }
    v = warp_ms_reduce(v);
    if (lane == 0) {
      sm.m[i] = v.m;
      sm.S[i] = v.s;
    }
  }
  __syncthreads();

  // 2. accept walk at every position at once; n = first failing position
  float acc_p = 0.f;
  bool bad = false;
  if (tid < 64) {
    bool fail = false;
    if (tid < a.gamma) {
      bad = !(pr.y > 0.f);
      const float px = exp2_approx(pr.x - sm.m[tid]) / sm.S[tid];
      acc_p = fminf(1.f, px / pr.y);
      fail = bad || !(ua < acc_p);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, fail);
    if (lane == 0) sm.fail[warp] = bal;
  }
  __syncthreads();
  if (tid == 0) {
    const uint64_t mask = (uint64_t)sm.fail[0] | ((uint64_t)sm.fail[1] << 32);
    int flags = 0;
    for (int i = 0; i < R; ++i)
      if (!(sm.S[i] > 0.f && isfinite(sm.S[i]) && isfinite(sm.m[i]))) flags |= VT_DEV_NONFINITE;
    sm.n = mask ? (__ffsll((long long)mask) - 1) : a.gamma;
    sm.flags = flags;
  }
  __syncthreads();
  const int n = sm.n;
  if (tid == n && tid < a.gamma && bad) atomicOr(&sm.flags, VT_DEV_BAD_DRAFT);
  __syncthreads();
  const int flags = sm.flags;
  if (c == 0 && a.out_accept_prob != nullptr && tid < a.gamma)
    a.out_accept_prob[(int64_t)b * a.gamma + tid] =
        (tid <= n && !(flags & VT_DEV_NONFINITE)) ? acc_p : __int_as_float(0x7fc00000);
  if (flags & (VT_DEV_BAD_DRAFT | VT_DEV_NONFINITE)) {
    griddep_launch_dependents();
    if (c == 0) {
      for (int i = tid; i < R; i += kNT) a.out_tokens[(int64_t)b * R + i] = -1;
      if (tid == 0) {
        a.out_n[b] = 0;
        atomicOr(a.dev_status, flags);
      }
    }
    return;
  }

  // 3. residual mass of this CTA's tiles of row n (p alone at the bonus
  // position)
  const T* rowp = static_cast<const T*>(a.logits) + ((int64_t)b * R + n) * a.V;
  const float m_n = sm.m[n];
  const float invS = 1.f / sm.S[n];
  const float* qrow = (n < a.gamma) ? a.q + ((int64_t)b * a.gamma + n) * a.K : nullptr;
  {
    // Software pipeline over the CTA's tiles: the next tile's id map and
    // logits are requested before this tile's residuals are reduced (a
    // pipeline two tiles deep measured 1-3% slower), and no barrier
    // separates the tiles: each warp keeps its per-tile totals in shared
    // memory and they are summed after the last tile.  A tile's total takes
    // the association order of block_scan_incl (warp inclusive scans, then
    // the warp totals in order), so it equals the total the chosen tile's
    // rescan computes.  Only the largest positive id over all tiles is
    // used, so one per CTA is kept.
    const int64_t jt = (int64_t)kResPerThread * tid;
    float x[8];
    load_logits8<T>(a, rowp, (int64_t)c0 * kResChunk + jt, x);
    int lpmax = -1;
    for (int ct = c0; ct < c1; ++ct) {
      const int64_t j = (int64_t)ct * kResChunk + jt;
      float qv[8];
      gather_q8(a, qrow, kmap, qv);
      const bool more = ct + 1 < c1;
      int kn[8];
      float xn[8];
      if (more) {
        load_kmap(a, j + kResChunk, kn);
        load_logits8<T>(a, rowp, j + kResChunk, xn);
      }
      float r[8];
      residual_of(a, x, qv, j, m_n, invS, r);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (r[e] > 0.f) lpmax = (int)(j + e);
      float v = sum8(r);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      // each warp moves on to the next tile at once: the warp totals are
      // summed once all tiles are done
      if (lane == 31) sm.tsum[ct - c0][warp] = v;
      if (more) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kmap[e] = kn[e];
          x[e] = xn[e];
        }
      }
    }
    __syncthreads();
    for (int k = tid; k < c1 - c0; k += kNT) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kNT / 32; ++w) tot += sm.tsum[k][w];
      a.zpart[(int64_t)b * a.C2 + c0 + k] = tot;
      __threadfence();  // published before the CTA's ticket below
    }
    lpmax = block_max_int<kNT>(lpmax, sm.ired);
    griddep_launch_dependents();
    if (tid == 0) {
      for (int ct = c0; ct < c1; ++ct) a.lpart[(int64_t)b * a.C2 + ct] = lpmax;
      __threadfence();
      sm.last = (atomicAdd(a.rdone + b, 1u) == (unsigned)(a.nfin - 1));
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
  }

  // 4. last tile of sequence b to finish: choose the tile, then the token.
  // Thread t sums the consecutive tiles [t * per, (t + 1) * per) in order;
  // one block scan of those sums gives every running sum the choice needs.
  int glast = -1;
  for (int k = tid; k < a.C2; k += kNT) {
    sm.zbuf[k] = __ldcg(a.zpart + (int64_t)b * a.C2 + k);
    glast = max(glast, __ldcg(a.lpart + (int64_t)b * a.C2 + k));
  }
  const float ures = a.u_res[(int64_t)b * R + n];
  glast = block_max_int<kNT>(glast, sm.ired);  // also publishes zbuf
  {
    const int per = (a.C2 + kNT - 1) / kNT;
    const int k0 = tid * per, k1 = min(a.C2, k0 + per);
    float mine = 0.f;
    for (int k = k0; k < k1; ++k) mine += sm.zbuf[k];
    float excl, total;
    const float incl = block_scan_incl<kNT>(mine, sm.sred, excl, total);
    const float target = ures * total;
    const int first = block_min_int<kNT>((total > 0.f && incl > target) ? tid : kNT, sm.ired);
    if (tid == 0) {
      sm.cstar = (total > 0.f) ? -1 : -2;  // -1: rounding put u * Z past every sum
      sm.target = 0.f;
    }
    __syncthreads();
    if (tid == first) {
      float pre = excl;
      for (int k = k0; k < k1; ++k) {
        if (pre + sm.zbuf[k] > target) {
          sm.cstar = k;
          sm.target = target - pre;
          break;
        }
        pre += sm.zbuf[k];
      }
    }
    __syncthreads();
  }
  int token = glast;
  int extra = 0;
  if (sm.cstar >= 0) {
    int lp;
    const int t = select_in_tile<T>(a, rowp, qrow, (int64_t)sm.cstar * kResChunk, m_n, invS,
                                    sm.target, sm, lp);
    token = (t >= 0) ? t : (lp >= 0 ? lp : glast);
  } else if (sm.cstar == -2) {
    // no residual mass (only through rounding): draw from p_n instead
    extra = VT_DEV_ZERO_RESIDUAL;
    float total = 0.f;
    for (int k = 0; k < a.C2; ++k) {
      int km[8];
      load_kmap(a, (int64_t)k * kResChunk + (int64_t)kResPerThread * tid, km);
      float r[8], excl, tot;
      int lp;
      tile_scan<T>(a, rowp, nullptr, (int64_t)k * kResChunk, m_n, invS, km, sm, r, excl, tot, lp);
      if (tid == 0) sm.zbuf[k] = tot;
      total += tot;
    }
    __syncthreads();
    const float target = ures * total;
    float pre = 0.f;
    int cstar = a.C2 - 1;
    for (int k = 0; k < a.C2; ++k) {
      if (pre + sm.zbuf[k] > target) { cstar = k; break; }
      pre += sm.zbuf[k];
    }
    int lp;
    const int t = select_in_tile<T>(a, rowp, nullptr, (int64_t)cstar * kResChunk, m_n, invS,
                                    target - pre, sm, lp);
    token = (t >= 0) ? t : lp;
  }
  for (int i = tid; i < R; i += kNT) {
    int v = -1;
    if (i < n) v = a.draft[(int64_t)b * a.gamma + i];
    else if (i == n) v = token;
    a.out_tokens[(int64_t)b * R + i] = v;
  }
  if (tid == 0) {
    a.out_n[b] = n;
    if (extra) atomicOr(a.dev_status, extra);
  }
}

struct VerifyLayout {
  size_t part, pre, zpart, lpart, rdone, bytes;
};

int chunks2(int64_t V) { return (int)((V + kResChunk - 1) / kResChunk); }

// residual tiles per finish CTA.  Every finish CTA merges its sequence's row
// partials and replays the accept walk whatever its share of the row, and
// walks its tiles one after another, so a row is split over few CTAs: the
// tiles of all rows are dealt out as if to about 608 CTAs (one wave of four
// 256-thread CTAs per SM).  Measured per verify call in graphs of calls
// against targets of 304, 1216 and 2432: B = 16 (2 tiles per CTA) 21.8
// against 23.0-23.9 us, B = 64 57.2 against 60.4-64.5 us, B = 256 (bf16,
// V = 152064; three CTAs per row, 768 in all) 193 against 196.5-224 us.
// Splitting rows so that the grid never exceeds one wave was slower at
// B = 256 (two CTAs per row: 197.7 us).
void set_finish_split(VArgs& a) {
  constexpr int64_t kWant = 608;
  const int64_t t = ((int64_t)a.C2 * a.B + kWant - 1) / kWant;
  a.tpc = (int)std::max<int64_t>(1, std::min<int64_t>({(int64_t)a.C2, t, (int64_t)kMaxTpc}));
  a.nfin = (a.C2 + a.tpc - 1) / a.tpc;
}

VerifyLayout verify_layout(int B, int gamma, int64_t V) {
  VerifyLayout L;
  size_t off = 0;
  auto take = [&](size_t n) {
    size_t o = off;
    off = align_up(off + n, 256);
    return o;
  };
  const int64_t rows = (int64_t)B * (gamma + 1);
  L.part = take((size_t)rows * kMaxChunks1 * sizeof(float2));
  L.pre = take((size_t)B * gamma * sizeof(float2));
  L.zpart = take((size_t)B * chunks2(V) * sizeof(float));
  L.lpart = take((size_t)B * chunks2(V) * sizeof(int));
  L.rdone = take((size_t)B * sizeof(unsigned));
  L.bytes = off;
  return L;
}

template <typename Kern>
cudaError_t launch_pdl(Kern kern, dim3 grid, cudaStream_t s, const VArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kNT);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T>
int launch_verify(const VArgs& a, cudaStream_t s) {
  VT_RETURN_IF_CUDA(launch_pdl(verify_stats_kernel<T>,
                               dim3((unsigned)((int64_t)a.B * a.R), (unsigned)a.C1), s, a));
  VT_RETURN_IF_CUDA(launch_pdl(verify_finish_kernel<T>, dim3((unsigned)a.B, (unsigned)a.nfin), s, a));
  return VT_OK;
}

// ------------------------------------------------- greedy (temperature 0)
// VocabTrim's greedy setting (section 4, Algorithm 2): position i keeps the
// drafted x_i iff it is the largest logit of row i (ties to the lower id);
// the first mismatch is replaced by that row's choice, and a fully accepted
// block appends the choice at position gamma.  The logits are compared as
// given (fp32, or bf16 widened exactly), so the choices are exact.

// (value, index) argmax, ties to the lower index; NaN (a non-finite logit)
// wins every comparison so it reaches the result
__device__ __forceinline__ bool gbetter(float v, int i, float w, int k) {
  if (v != v) return false;
  if (w != w) return true;
  return w > v || (w == v && k < i);
}

__device__ __forceinline__ void warp_gmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    const int k = __shfl_xor_sync(0xffffffffu, i, o);
    if (gbetter(v, i, w, k)) {
      v = w;
      i = k;
    }
  }
}

// grid (rows, C1 chunks): per chunk the largest logit and its lowest id
template <typename T>
__global__ void __launch_bounds__(kNT) verify_greedy_stats_kernel(VArgs a) {
  __shared__ float sv[kNT / 32];
  __shared__ int si[kNT / 32];
  constexpr int VEC = Elem<T>::kVec;
  constexpr int U = kStatsBytes / 16 / kNT;
  griddep_wait();
  const int64_t row = blockIdx.x;
  const int c = blockIdx.y;
  if (row == 0 && c == 0 && threadIdx.x == 0) *a.dev_status = 0;
  const T* rp = static_cast<const T*>(a.logits) + row * a.V;
  const int64_t j0 = (int64_t)c * a.len1;
  const int64_t j1 = min(a.V, j0 + a.len1);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  // this thread's ids rise along both loops, so a tie keeps the lower id
  auto take = [&](float x, int64_t j) {
    const float v = isfinite(x) ? x : __int_as_float(0x7fc00000);
    if (gbetter(bv, bi, v, (int)j)) {
      bv = v;
      bi = (int)j;
    }
  };
  int64_t jt = j0;
  if (a.vec_ok) {
    const int64_t nv = (j1 - j0) / VEC;
    const uint4* vp = reinterpret_cast<const uint4*>(rp + j0);
    for (int64_t v = threadIdx.x; v < nv; v += (int64_t)kNT * U) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t vi = v + (int64_t)u * kNT;
        if (vi < nv) raw[u] = __ldg(vp + vi);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t vi = v + (int64_t)u * kNT;
        if (vi < nv) {
          float x[VEC];
          Elem<T>::unpack16(raw[u], x);
#pragma unroll
          for (int e = 0; e < VEC; ++e) take(x[e], j0 + vi * VEC + e);
        }
      }
    }
    jt = j0 + nv * VEC;
  }
  for (int64_t j = jt + threadIdx.x; j < j1; j += kNT) take(Elem<T>::load(rp + j), j);
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_gmax(bv, bi);
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kNT / 32; ++w)
      if (gbetter(bv, bi, sv[w], si[w])) {
        bv = sv[w];
        bi = si[w];
      }
    a.part[row * a.C1 + c] = make_float2(bv, __int_as_float(bi));
  }
}

// grid (B): merge the chunk partials of the gamma+1 rows, walk, write
__global__ void __launch_bounds__(kNT) verify_greedy_finish_kernel(VArgs a) {
  __shared__ int choice[kMaxGamma + 1];
  __shared__ unsigned fail[2];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R;
  griddep_wait();  // the stats kernel has completed
  for (int i = warp; i < R; i += kNT / 32) {
    float v = -INFINITY;
    int idx = 0x7fffffff;
    const float2* pp = a.part + ((int64_t)b * R + i) * a.C1;
    for (int k = lane; k < a.C1; k += 32) {
      const float2 t = pp[k];
      if (gbetter(v, idx, t.x, __float_as_int(t.y))) {
        v = t.x;
        idx = __float_as_int(t.y);
      }
    }
    warp_gmax(v, idx);
    if (lane == 0) choice[i] = (v == v && idx >= 0 && (int64_t)idx < a.V) ? idx : -1;
  }
  __syncthreads();
  bool bad = false;
  if (tid < 64) {
    bool f = false;
    if (tid < a.gamma) {
      const int x = a.draft[(int64_t)b * a.gamma + tid];
      bad = !(x >= 0 && (int64_t)x < a.V);
      f = bad || x != choice[tid];
    }
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) fail[warp] = bal;
  }
  __syncthreads();
  const uint64_t mask = (uint64_t)fail[0] | ((uint64_t)fail[1] << 32);
  const int n = mask ? (__ffsll((long long)mask) - 1) : a.gamma;
  int flags = 0;
  for (int i = 0; i < R; ++i)
    if (choice[i] < 0) flags |= VT_DEV_NONFINITE;
  // a drafted token outside [0, V) stops the walk at its position
  if (__syncthreads_or(tid == n && tid < a.gamma && bad)) flags |= VT_DEV_BAD_DRAFT;
  if (a.out_accept_prob != nullptr && tid < a.gamma)
    a.out_accept_prob[(int64_t)b * a.gamma + tid] =
        (flags == 0 && tid <= n) ? (tid < n ? 1.f : 0.f) : __int_as_float(0x7fc00000);
  for (int i = tid; i < R; i += kNT) {
    int v = -1;
    if (flags == 0) {
      if (i < n) v = a.draft[(int64_t)b * a.gamma + i];
      else if (i == n) v = choice[n];
    }
    a.out_tokens[(int64_t)b * R + i] = v;
  }
  if (tid == 0) {
    a.out_n[b] = flags ? 0 : n;
    if (flags) atomicOr(a.dev_status, flags);
  }
}

// ------------------------------------------------------------ draft trees
// Greedy verification of a draft tree (VocabTrim section 4.1's EAGLE-2
// trees with the greedy target of section 4): N nodes in topological order,
// node i with a target id and a parent in {-1} or [0, i) (-1: the context);
// the target scores N + 1 rows (row 0 after the context, row i + 1 after
// node i).  Node i is accepted iff its parent is and its token is the
// target's choice at the parent's row; the block is the path to the
// deepest accepted node (ties to the lower node) and the choice there.
constexpr int kMaxTreeNodes = 255;

// one warp per row of partials (up to 32 rows at once)
constexpr int kTreeNT = 1024;

struct TreeArgs {
  const int* parent;    // [B][N], or one shared [N] when pstride == 0
  int64_t pstride;
  const int* tokens;    // [B][N]
  int N;
  int* out_path;        // [B][N] or nullptr
};

__global__ void __launch_bounds__(kTreeNT) verify_tree_finish_kernel(VArgs a, TreeArgs t) {
  __shared__ int choice[kMaxTreeNodes + 1];
  __shared__ unsigned char acc[kMaxTreeNodes];
  __shared__ unsigned char dep[kMaxTreeNodes];
  __shared__ int path[kMaxTreeNodes];
  __shared__ int spar[kMaxTreeNodes];  // the tree, staged once: the walk below
  __shared__ int stok[kMaxTreeNodes];  // is serial, so it reads shared memory only
  __shared__ int s_best, s_len, s_flags;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R, N = t.N;
  // inputs that the stats kernel of this call does not write (every older
  // kernel has completed): fetch before waiting
  for (int i = tid; i < N; i += kTreeNT) {
    spar[i] = t.parent[(int64_t)b * t.pstride + i];
    stok[i] = t.tokens[(int64_t)b * N + i];
  }
  griddep_wait();  // the stats kernel has completed
  for (int i = warp; i < R; i += kTreeNT / 32) {
    float v = -INFINITY;
    int idx = 0x7fffffff;
    const float2* pp = a.part + ((int64_t)b * R + i) * a.C1;
    for (int k = lane; k < a.C1; k += 32) {
      const float2 q = pp[k];
      if (gbetter(v, idx, q.x, __float_as_int(q.y))) {
        v = q.x;
        idx = __float_as_int(q.y);
      }
    }
    warp_gmax(v, idx);
    if (lane == 0) choice[i] = (v == v && idx >= 0 && (int64_t)idx < a.V) ? idx : -1;
  }
  __syncthreads();
  if (tid == 0) {
    // nodes in topological order: a parent's verdict is known before its children's
    int flags = 0, best = -1, best_depth = 0;
    for (int r = 0; r < R; ++r)
      if (choice[r] < 0) flags |= VT_DEV_NONFINITE;
    for (int i = 0; i < N && !flags; ++i) {
      const int p = spar[i];
      const int x = stok[i];
      if (p < -1 || p >= i || x < 0 || (int64_t)x >= a.V) {
        flags |= VT_DEV_BAD_DRAFT;
        break;
      }
      const bool ok = (p < 0 || acc[p]) && x == choice[p + 1];
      acc[i] = ok ? 1 : 0;
      dep[i] = (unsigned char)(p < 0 ? 1 : dep[p] + 1);
      if (ok && dep[i] > best_depth) {
        best = i;
        best_depth = dep[i];
      }
    }
    int len = 0;
    if (!flags) {
      for (int i = best; i >= 0; i = spar[i]) path[len++] = i;
      for (int k = 0; k < len / 2; ++k) {  // root first
        const int tmp = path[k];
        path[k] = path[len - 1 - k];
        path[len - 1 - k] = tmp;
      }
    }
    s_best = best;
    s_len = len;
    s_flags = flags;
  }
  __syncthreads();
  const int flags = s_flags, len = s_len, best = s_best;
  for (int i = tid; i < R; i += kTreeNT) {
    int v = -1;
    if (!flags) {
      if (i < len) v = stok[path[i]];
      else if (i == len) v = choice[best + 1];
    }
    a.out_tokens[(int64_t)b * R + i] = v;
  }
  if (t.out_path != nullptr)
    for (int i = tid; i < N; i += kTreeNT)
      t.out_path[(int64_t)b * N + i] = (!flags && i < len) ? path[i] : -1;
  if (tid == 0) {
    a.out_n[b] = flags ? 0 : len;
    if (flags) atomicOr(a.dev_status, flags);
  }
}

template <typename T>
int launch_verify_greedy(const VArgs& a, cudaStream_t s) {
  VT_RETURN_IF_CUDA(launch_pdl(verify_greedy_stats_kernel<T>,
                               dim3((unsigned)((int64_t)a.B * a.R), (unsigned)a.C1), s, a));
  VT_RETURN_IF_CUDA(launch_pdl(verify_greedy_finish_kernel, dim3((unsigned)a.B), s, a));
  return VT_OK;
}

template <typename T>
int launch_verify_tree(const VArgs& a, const TreeArgs& t, cudaStream_t s) {
  VT_RETURN_IF_CUDA(launch_pdl(verify_greedy_stats_kernel<T>,
                               dim3((unsigned)((int64_t)a.B * a.R), (unsigned)a.C1), s, a));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.B);
  cfg.blockDim = dim3(kTreeNT);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  VT_RETURN_IF_CUDA(cudaLaunchKernelEx(&cfg, verify_tree_finish_kernel, a, t));
  return VT_OK;
}


}  // namespace
}  // namespace vt

namespace vt {
namespace {

// Host-checkable argument errors of vt_verify (and vt_verify_noalloc).
int verify_check_args(const void* target_logits, int32_t logits_dtype, int32_t B, int32_t gamma,
                      int32_t V, const float* q, const int32_t* inv_map, int32_t K,
                      const int32_t* draft_tokens, const float* u_accept,
                      const float* u_resample, float temperature, const int32_t* out_tokens,
                      const int32_t* out_num_accepted, const int32_t* dev_status) {
  const bool greedy = temperature == 0.f;
  if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted || !dev_status)
    return VT_ERR_INVALID_ARG;
  if (!greedy && (!q || !inv_map || !u_accept || !u_resample)) return VT_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || gamma < 1 || gamma > kMaxGamma || V < 1 || K < 1 || K > V ||
      V > (1 << 22))
    return VT_ERR_INVALID_ARG;
  if (logits_dtype != VT_F32 && logits_dtype != VT_BF16) return VT_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return VT_ERR_INVALID_ARG;
  return VT_OK;
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_verify_workspace_bytes(int32_t B, int32_t gamma, int32_t V, int32_t K) {
  (void)K;
  if (B < 1 || gamma < 1 || V < 1) return 0;
  return vt::verify_layout(B, gamma, V).bytes;
}

extern "C" int vt_verify(const void* target_logits, int32_t logits_dtype, int32_t B, int32_t gamma,
                         int32_t V, const float* q, const int32_t* inv_map, int32_t K,
                         const int32_t* draft_tokens, const float* u_accept,
                         const float* u_resample, float temperature, int32_t* out_tokens,
                         int32_t* out_num_accepted, float* out_accept_prob, int32_t* dev_status,
                         void* workspace, size_t workspace_bytes, void* stream) {
  using namespace vt;
  // temperature 0: greedy verification (q, inv_map and the uniforms are not read)
  const bool greedy = temperature == 0.f;
  const int arg = verify_check_args(target_logits, logits_dtype, B, gamma, V, q, inv_map, K,
                                    draft_tokens, u_accept, u_resample, temperature, out_tokens,
                                    out_num_accepted, dev_status);
  if (arg != VT_OK) return arg;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  const VerifyLayout L = verify_layout(B, gamma, V);
  if (workspace_bytes < L.bytes) return VT_ERR_WORKSPACE;

  const size_t esize = (logits_dtype == VT_F32) ? 4 : 2;
  const int vec = (logits_dtype == VT_F32) ? 4 : 8;
  char* ws = static_cast<char*>(workspace);
  VArgs a;
  a.logits = target_logits;
  a.V = V;
  a.B = B;
  a.gamma = gamma;
  a.R = gamma + 1;
  a.K = K;
  a.q = q;
  a.inv_map = inv_map;
  a.draft = draft_tokens;
  a.u_acc = u_accept;
  a.u_res = u_resample;
  a.scale = greedy ? 1.f : VT_LOG2E / temperature;
  // stats chunks of 32 KB (at most kMaxChunks1 per row), aligned to the
  // 16-byte vector width
  int64_t len1 = std::max<int64_t>(kStatsBytes / (int64_t)esize,
                                   ((int64_t)V + kMaxChunks1 - 1) / kMaxChunks1);
  len1 = (len1 + vec - 1) / vec * vec;
  a.len1 = len1;
  a.C1 = (int)(((int64_t)V + len1 - 1) / len1);
  a.C2 = chunks2(V);
  set_finish_split(a);
  // 16-byte loads need every row to start on a 16-byte boundary; residual
  // tiles also load inv_map eight ids at a time
  a.vec_ok = ((reinterpret_cast<uintptr_t>(target_logits) & 15) == 0) &&
             (((int64_t)V * esize) % 16 == 0) && ((reinterpret_cast<uintptr_t>(inv_map) & 15) == 0);
  a.part = reinterpret_cast<float2*>(ws + L.part);
  a.pre = reinterpret_cast<float2*>(ws + L.pre);
  a.zpart = reinterpret_cast<float*>(ws + L.zpart);
  a.lpart = reinterpret_cast<int*>(ws + L.lpart);
  a.rdone = reinterpret_cast<unsigned*>(ws + L.rdone);
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.out_accept_prob = out_accept_prob;
  a.dev_status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (greedy) {
    if (logits_dtype == VT_F32) return launch_verify_greedy<float>(a, s);
    return launch_verify_greedy<uint16_t>(a, s);
  }
  if (logits_dtype == VT_F32) return launch_verify<float>(a, s);
  return launch_verify<uint16_t>(a, s);
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

// 2 MiB of scratch per device, resident for the life of the process.
static __device__ __align__(256) unsigned char g_noalloc_scratch[VT_VERIFY_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the calling thread's current
// context.  Host code only holds a stand-in for the symbol, and each context
// that loads the library gets its own copy of the array, so the address is
// looked up on every call: a cached address would outlive the context it
// belongs to (cudaDeviceReset, or a caller that switches to a context of its
// own on the same device).  The lookup is a host-side table query, not a
// stream operation.
int noalloc_scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return VT_ERR_CUDA;
  }
  *out = p;
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
  // the argument checks of vt_verify come first, so a bad argument reports
  // VT_ERR_INVALID_ARG here too; only a valid problem can exceed the scratch
  const int arg = verify_check_args(target_logits, logits_dtype, B, gamma, V, q, inv_map, K,
                                    draft_tokens, u_accept, u_resample, temperature, out_tokens,
                                    out_num_accepted, dev_status);
  if (arg != VT_OK) return arg;
  const size_t need = vt_verify_workspace_bytes(B, gamma, V, K);
  if (need > VT_VERIFY_NOALLOC_SCRATCH_BYTES) return VT_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int st = noalloc_scratch_address(&scratch);
  if (st != VT_OK) return st;
  return vt_verify(target_logits, logits_dtype, B, gamma, V, q, inv_map, K, draft_tokens,
                   u_accept, u_resample, temperature, out_tokens, out_num_accepted,
                   out_accept_prob, dev_status, scratch, VT_VERIFY_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" size_t vt_verify_tree_workspace_bytes(int32_t B, int32_t N, int32_t V) {
  if (B < 1 || N < 1 || N > vt::kMaxTreeNodes || V < 1) return 0;
  return vt_verify_workspace_bytes(B, N, V, 1);
}

extern "C" int vt_verify_tree(const void* target_logits, int32_t logits_dtype, int32_t B,
                              int32_t N, int32_t V, const int32_t* parent, int64_t parent_stride,
                              const int32_t* tokens, float temperature, int32_t* out_tokens,
                              int32_t* out_num_accepted, int32_t* out_path, int32_t* dev_status,
                              void* workspace, size_t workspace_bytes, void* stream) {
  using namespace vt;
  if (!target_logits || !parent || !tokens || !out_tokens || !out_num_accepted || !dev_status)
    return VT_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || N < 1 || N > kMaxTreeNodes || V < 1 || V > (1 << 22))
    return VT_ERR_INVALID_ARG;
  if (parent_stride != 0 && parent_stride < N) return VT_ERR_INVALID_ARG;
  if (logits_dtype != VT_F32 && logits_dtype != VT_BF16) return VT_ERR_INVALID_ARG;
  if (!std::isfinite(temperature) || temperature < 0.f) return VT_ERR_INVALID_ARG;
  if (temperature != 0.f) return VT_ERR_UNSUPPORTED;  // trees are verified greedily
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  const VerifyLayout L = verify_layout(B, N, V);
  if (workspace_bytes < L.bytes) return VT_ERR_WORKSPACE;
  const size_t esize = (logits_dtype == VT_F32) ? 4 : 2;
  const int vec = (logits_dtype == VT_F32) ? 4 : 8;
  VArgs a = {};
  a.logits = target_logits;
  a.V = V;
  a.B = B;
  a.gamma = N;
  a.R = N + 1;
  a.K = 1;
  a.scale = 1.f;
  int64_t len1 = std::max<int64_t>(kStatsBytes / (int64_t)esize,
                                   ((int64_t)V + kMaxChunks1 - 1) / kMaxChunks1);
  len1 = (len1 + vec - 1) / vec * vec;
  a.len1 = len1;
  a.C1 = (int)(((int64_t)V + len1 - 1) / len1);
  a.C2 = chunks2(V);
  set_finish_split(a);
  a.vec_ok = ((reinterpret_cast<uintptr_t>(target_logits) & 15) == 0) &&
             (((int64_t)V * esize) % 16 == 0);
  a.part = reinterpret_cast<float2*>(static_cast<char*>(workspace) + L.part);
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.dev_status = dev_status;
  TreeArgs t;
  t.parent = parent;
  t.pstride = parent_stride;
  t.tokens = tokens;
  t.N = N;
  t.out_path = out_path;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (logits_dtype == VT_F32) return launch_verify_tree<float>(a, t, s);
  return launch_verify_tree<uint16_t>(a, t, s);
}
