// Drafting through the VocabTrim head on sm_103a.
//
// Operation ("VocabTrim: Vocabulary Pruning for Efficient Speculative
// Decoding in LLMs", Algorithm 2, drafting; temperature as required by the
// "Speculative decoding" glossary, "Distributional exactness has
// conditions"):
//   z[b, j] = (hidden[b] . W_trim[j]) / T     over the K trimmed ids only
//   q[b, :] = softmax(z[b, :]);  token[b] = trim_ids[j*], j* = strict inverse
//   CDF of q[b] at u_b in ascending j (ascending target id).
//
// Kernels:
//  1. the projection, on the tensor cores when the shapes allow it
//     (head_umma_kernel in vt_umma.cuh: tcgen05 MMA, TMA-fed, accumulator in
//     tensor memory; batch <= 256, H a multiple of 8, 16-byte aligned rows),
//     otherwise draft_gemv on the CUDA cores: it streams W_trim once from HBM with 16-byte loads, four lanes
//     per row (64 contiguous bytes per row per step), the hidden tile in
//     shared memory (broadcast reads), fp32 FMA accumulation.  Its epilogue
//     stores z (scaled to base 2 for the softmax) and folds each CTA's rows
//     into per-row-of-batch online-softmax partials (max, sum 2^(z - max)).
//  2. draft_finalize grid (B, C chunks of several 1024-id passes): merges
//     the partials, writes q = 2^(z-m)/S in place; every CTA scans the
//     per-tile masses s_t 2^(m_t - m) in tile order (no CTA waits on
//     another) to find the tile where the running
//     mass passes u_b * S, and the CTA holding that tile scans its rows in
//     ascending id order to pick the token.
//  Both kernels are launched with programmatic dependent launch: the
//  projection streams its first W_trim stages while the previous kernel in
//  the stream drains.
#include <algorithm>
#include <cmath>

#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include "vt_common.cuh"
#include "vt_internal.h"
#include "vt_umma.cuh"

namespace cg = cooperative_groups;

namespace vt {
namespace {

constexpr int kGemvNT = 256;        // 8 warps
constexpr int kRowsPerWarp = 8;     // 4 lanes per row
constexpr int kGemvRowTile = 64;  // rows per CTA of the CUDA-core projection
constexpr int kFinNT = 256;

__device__ __forceinline__ void unpack_bf16x8(uint4 v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

// out[b, j] = out_scale * sum_h hidden[b, h] * W[j, h] for one tile of BT rows
// of the batch at a time.  part (optional) receives, per CTA and batch row,
// the online-softmax partial of the values written.
template <int BT, int UNROLL>
__global__ void __launch_bounds__(kGemvNT)
draft_gemv_kernel(const uint16_t* __restrict__ hidden, int B, int H,
                  const uint16_t* __restrict__ W, int K, float out_scale,
                  float* __restrict__ out, int64_t ldo, float2* __restrict__ part,
                  int* __restrict__ zero_ints, int nzero, int* __restrict__ status_to_zero,
                  int vec_ok, int greedy) {
  extern __shared__ __align__(16) uint16_t sh_h[];  // [BT][H]
  __shared__ MS sred[kGemvNT / 32][BT];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane & 3;         // which 16-byte slice of a 64-byte step
  const int rlane = lane >> 2;      // row within the warp's group of 8

  if (blockIdx.x == 0) {
    // tickets and status word of the finalize kernel, which starts only
    // after this grid has completed (same stream)
    for (int i = tid; i < nzero; i += kGemvNT) zero_ints[i] = 0;
    if (tid == 0 && status_to_zero != nullptr) *status_to_zero = 0;
  }

  for (int b0 = 0; b0 < B; b0 += BT) {
    const int bt = min(BT, B - b0);
    __syncthreads();
    // stage hidden rows b0..b0+bt (zero rows past bt)
    if (vec_ok) {
      const int hv = H / 8;
      for (int i = tid; i < BT * hv; i += kGemvNT) {
        const int b = i / hv, c = i - b * hv;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (b < bt) v = __ldg(reinterpret_cast<const uint4*>(hidden + (int64_t)(b0 + b) * H) + c);
        reinterpret_cast<uint4*>(sh_h + (int64_t)b * H)[c] = v;
      }
    } else {
      for (int i = tid; i < BT * H; i += kGemvNT) {
        const int b = i / H, c = i - b * H;
        sh_h[i] = (b < bt) ? __ldg(hidden + (int64_t)(b0 + b) * H + c) : (uint16_t)0;
      }
    }
    __syncthreads();

    float m[BT], s[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      m[b] = greedy ? -INFINITY : kNegBig;
      s[b] = greedy ? __int_as_float(0x7fffffff) : 0.f;
    }

    const int groups = (K + kRowsPerWarp - 1) / kRowsPerWarp;
    // one group of 8 consecutive rows per warp: CTA g covers rows [64g, 64g+64)
    for (int g = blockIdx.x * (kGemvNT / 32) + warp; g < groups; g += gridDim.x * (kGemvNT / 32)) {
      const int row = g * kRowsPerWarp + rlane;
      float acc[BT];
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[b] = 0.f;
      if (row < K) {
        const uint16_t* wr = W + (int64_t)row * H;
        if (vec_ok) {
          // 16-byte slices h = 8*sub + 32*t
          const int nsteps = H / 32;           // full 64-byte steps
          int t = 0;
          for (; t + UNROLL <= nsteps; t += UNROLL) {
            uint4 wv[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
              wv[u] = __ldg(reinterpret_cast<const uint4*>(wr + 32 * (t + u) + 8 * sub));
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
              float wf[8];
              unpack_bf16x8(wv[u], wf);
              const int h = 32 * (t + u) + 8 * sub;
#pragma unroll
              for (int b = 0; b < BT; ++b) {
                float hf[8];
                unpack_bf16x8(*reinterpret_cast<const uint4*>(sh_h + b * H + h), hf);
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[b] = fmaf(wf[k], hf[k], acc[b]);
              }
            }
          }
          for (; t < nsteps; ++t) {
            const int h = 32 * t + 8 * sub;
            float wf[8];
            unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(wr + h)), wf);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
              float hf[8];
              unpack_bf16x8(*reinterpret_cast<const uint4*>(sh_h + b * H + h), hf);
#pragma unroll
              for (int k = 0; k < 8; ++k) acc[b] = fmaf(wf[k], hf[k], acc[b]);
            }
          }
          // remaining H % 32 elements in 16-byte slices
          const int h = 32 * nsteps + 8 * sub;
          if (h < H) {
            float wf[8];
            unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(wr + h)), wf);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
              float hf[8];
              unpack_bf16x8(*reinterpret_cast<const uint4*>(sh_h + b * H + h), hf);
#pragma unroll
              for (int k = 0; k < 8; ++k) acc[b] = fmaf(wf[k], hf[k], acc[b]);
            }
          }
        } else {
          for (int h = sub; h < H; h += 4) {
            const float wf = bf16_bits_to_float(__ldg(wr + h));
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[b] = fmaf(wf, bf16_bits_to_float(sh_h[b * H + h]), acc[b]);
          }
        }
      }
      // reduce the four lanes of each row
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 1);
        acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], 2);
      }
      if (row < K && sub == 0) {
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          if (b < bt) {
            const float z = acc[b] * out_scale;
            out[(int64_t)(b0 + b) * ldo + row] = z;
            if (greedy) {
              // m = max z, s = its lowest row (rows rise along this loop)
              const float v = isfinite(z) ? z : __int_as_float(0x7fc00000);
              if (umma::argmax_better(m[b], __float_as_int(s[b]), v, row)) {
                m[b] = v;
                s[b] = __int_as_float(row);
              }
            } else {
              if (z > m[b]) {
                s[b] *= exp2_approx(m[b] - z);
                m[b] = z;
              }
              s[b] += exp2_approx(z - m[b]);
            }
          }
        }
      }
    }
    if (part != nullptr) {
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        if (greedy) {
          float v = m[b];
          int i = __float_as_int(s[b]);
          umma::warp_argmax(v, i);
          if (lane == 0) sred[warp][b] = MS{v, __int_as_float(i)};
        } else {
          MS v = warp_ms_reduce(MS{m[b], s[b]});
          if (lane == 0) sred[warp][b] = v;
        }
      }
      __syncthreads();
      if (tid < bt) {
        MS r = sred[0][tid];
#pragma unroll
        for (int w = 1; w < kGemvNT / 32; ++w) {
          if (greedy) {
            if (umma::argmax_better(r.m, __float_as_int(r.s), sred[w][tid].m,
                                    __float_as_int(sred[w][tid].s)))
              r = sred[w][tid];
          } else {
            r = ms_combine(r, sred[w][tid]);
          }
        }
        part[(int64_t)blockIdx.x * B + b0 + tid] = make_float2(r.m, r.s);
      }
    }
  }
}

struct FinArgs {
  float* q;          // in: z scaled to base 2; out: probabilities
  int64_t ldq;
  int B, K;
  const float2* part;  // [G][B] partials of consecutive row tiles
  int G;
  int tile_rows;       // rows per partial (64 or 128; divides kFinChunk)
  int passes;          // chunks of kFinChunk ids per CTA
  const float* u;
  const int* trim_ids;
  int* tokens;
  int64_t ldt;
  int* dev_status;
  int vec_ok;
};

constexpr int kFinChunk = kFinNT * 4;  // ids normalised per CTA and pass

// finalize passes per CTA.  A sampling CTA merges all of its row's partials
// and scans its tile masses whatever its share of the row, so a row is split
// over few CTAs: at least four passes each, and a grid of at most about 512
// CTAs (measured on the drafting step for B = 1..256: fewer, longer CTAs
// were faster down to these bounds).  The greedy finalize only merges the
// (max, row) partials and writes a one-hot row: up to about 1216 CTAs.
inline int fin_passes(int B, int K, bool greedy) {
  const int64_t p1 = (K + kFinChunk - 1) / kFinChunk;  // 1024-id passes per row
  const int64_t target = greedy ? 1216 : 512;
  int64_t r = std::max<int64_t>(greedy ? 1 : std::min<int64_t>(4, p1), (p1 * B + target - 1) / target);
  return (int)std::min(r, p1);
}

// the passes of one batch: loaded together (RB float4 loads in flight per
// thread), then weighted, drawn from and stored
template <int RB>
__device__ __forceinline__ void fin_load(float (&z)[RB][4], const float* qrow, int64_t j0, int p0,
                                         int np, int K, bool vec_ok) {
#pragma unroll
  for (int q = 0; q < RB; ++q) {
    const int64_t j = j0 + (int64_t)(p0 + q) * kFinChunk;
    if (p0 + q < np && vec_ok && j + 3 < K) {
      const float4 v = *reinterpret_cast<const float4*>(qrow + j);
      z[q][0] = v.x; z[q][1] = v.y; z[q][2] = v.z; z[q][3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) z[q][e] = (p0 + q < np && j + e < K) ? qrow[j + e] : kNegBig;
    }
  }
}

// Normalises q for a.passes consecutive chunks of 1024 ids of row b and, in
// the CTA whose chunks hold the sampled tile, draws the token.  The
// projection left one online-softmax partial (m_t, s_t) per tile of
// consecutive rows; the global (m, S) and the tile masses s_t 2^(m_t - m) in
// units of the global 2^m are therefore known to every CTA without waiting
// on any other: all CTAs of row b scan the tile masses in tile order to find
// the tile where the running mass passes u_b * S, and the warp holding that
// tile scans its rows (ascending id) to pick the row.  The chunks are
// streamed in batches of RB passes (four consecutive ids per thread and
// pass); the first batch is requested before the partials are merged.
template <int RB>
__global__ void __launch_bounds__(kFinNT) draft_finalize_kernel(FinArgs a) {
  __shared__ MS mred[kFinNT / 32];
  __shared__ float sred[kFinNT / 32];
  __shared__ int ired[kFinNT / 32];
  __shared__ int s_tile, s_last;
  __shared__ float s_before;
  constexpr int kRegTiles = 4;  // tile partials a thread keeps in registers
  const int b = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31;
  float* qrow = a.q + (int64_t)b * a.ldq;
  // the next kernel may launch now: it reads nothing this kernel writes
  // before its own griddepcontrol.wait, which waits for this whole grid
  griddep_launch_dependents();
  griddep_wait();  // the projection has completed

  // this CTA's passes [0, np) start at cbase; in pass p this thread holds
  // ids j0 + p * kFinChunk + [0, 4)
  const int64_t cbase = (int64_t)c * kFinChunk * a.passes;
  const int64_t j0 = cbase + 4 * (int64_t)tid;
  const int np = (int)min((int64_t)a.passes, (a.K - cbase + kFinChunk - 1) / kFinChunk);
  float z[RB][4];
  fin_load<RB>(z, qrow, j0, 0, np, a.K, a.vec_ok != 0);
  const int per = (a.G + kFinNT - 1) / kFinNT;
  const int t0 = tid * per, t1 = min(a.G, t0 + per);
  float2 pt[kRegTiles];
  MS mine{kNegBig, 0.f};
  for (int t = t0; t < t1; ++t) {
    const float2 p = a.part[(int64_t)t * a.B + b];
    if (t - t0 < kRegTiles) pt[t - t0] = p;
    mine = ms_combine(mine, MS{p.x, p.y});
  }
  const MS g = block_ms_reduce<kFinNT>(mine, mred);
  if (!(g.s > 0.f && isfinite(g.s) && isfinite(g.m))) {
    if (c == 0 && tid == 0) {
      a.tokens[(int64_t)b * a.ldt] = -1;
      atomicOr(a.dev_status, VT_DEV_NONFINITE);
    }
    return;
  }
  const float m = g.m, invS = 1.f / g.s;
  auto tile_part = [&](int t) -> float2 {
    return (t - t0 < kRegTiles) ? pt[t - t0] : a.part[(int64_t)t * a.B + b];
  };

  // tile holding the draw: scan of tile masses in tile order (the token is
  // chosen before this chunk of q is normalised)
  const float target = a.u[b] * g.s;
  float mass = 0.f;
  for (int t = t0; t < t1; ++t) {
    const float2 p = tile_part(t);
    mass += p.y * exp2_approx(p.x - m);
  }
  float excl, tot;
  const float incl = block_scan_incl<kFinNT>(mass, sred, excl, tot);
  const int first = block_min_int<kFinNT>(incl > target ? tid : kFinNT, ired);
  if (tid == 0) {
    s_tile = -1;
    s_before = 0.f;
    s_last = 0;
  }
  __syncthreads();
  if (tid == first) {
    // walk this thread's tiles; if rounding hides the crossing, fall back to
    // the last tile with mass in the range and its last weighted row
    float run = excl;
    int last_t = -1;
    for (int t = t0; t < t1; ++t) {
      const float2 p = tile_part(t);
      const float mt = p.y * exp2_approx(p.x - m);
      if (mt > 0.f) last_t = t;
      if (run + mt > target) {
        s_tile = t;
        s_before = run;
        break;
      }
      run += mt;
    }
    if (s_tile < 0) {
      s_tile = last_t;
      s_last = 1;
    }
  }
  __syncthreads();
  int tsel = s_tile;
  const float before = s_before;
  bool force_last = s_last != 0;
  if (first == kFinNT) {
    // u * S at or above the summed masses (rounding): last tile with mass
    tsel = -1;
    for (int t = a.G - 1; t >= 0 && tsel < 0; --t)
      if (a.part[(int64_t)t * a.B + b].y > 0.f) tsel = t;
    force_last = true;
  }
  const int64_t r0 = (int64_t)max(tsel, 0) * a.tile_rows;
  const bool owner_cta = tsel >= 0 && r0 >= cbase && r0 < cbase + (int64_t)kFinChunk * np;
  // a tile lies within one pass (tile_rows divides kFinChunk)
  const int opass = owner_cta ? (int)((r0 - cbase) / kFinChunk) : -1;
  const int owner_warp = owner_cta ? (int)(((r0 - cbase) % kFinChunk) / 4) >> 5 : -1;

#pragma unroll 1
  for (int p0 = 0; p0 < np; p0 += RB) {
    if (p0 > 0) fin_load<RB>(z, qrow, j0, p0, np, a.K, a.vec_ok != 0);
#pragma unroll
    for (int q = 0; q < RB; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        z[q][e] = (j0 + (int64_t)(p0 + q) * kFinChunk + e < a.K) ? exp2_approx(z[q][e] - m) : 0.f;
    if ((tid >> 5) == owner_warp && opass >= p0 && opass < p0 + RB) {
      // this batch holds the tile: its rows are consecutive threads of one warp
      const int64_t r1 = min((int64_t)a.K, r0 + a.tile_rows);
      const int64_t j = j0 + (int64_t)opass * kFinChunk;
      float w[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < RB; ++q)
        if (p0 + q == opass)
#pragma unroll
          for (int e = 0; e < 4; ++e) w[e] = z[q][e];
      float v = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j + e >= r0 && j + e < r1) v += w[e];
      float x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const float local = target - before;
      const unsigned hit = force_last ? 0u : __ballot_sync(0xffffffffu, x > local);
      int pick = -1;
      if (hit) {
        const int l = __ffs(hit) - 1;
        if (lane == l) {
          float acc = x - v;
          int lastp = -1;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (j + e < r0 || j + e >= r1) continue;
            if (w[e] > 0.f) lastp = (int)(j + e);
            acc += w[e];
            if (pick < 0 && acc > local) pick = (int)(j + e);
          }
          if (pick < 0) pick = lastp;
        }
        pick = __shfl_sync(0xffffffffu, pick, l);
      } else {
        // last row with weight in the tile
        int lp = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (j + e >= r0 && j + e < r1 && w[e] > 0.f) lp = (int)(j + e);
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        pick = lp;
      }
      if (lane == 0) a.tokens[(int64_t)b * a.ldt] = (pick >= 0) ? a.trim_ids[pick] : -1;
    }
    // normalise this batch in place
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      if (p0 + q >= np) continue;
      const int64_t j = j0 + (int64_t)(p0 + q) * kFinChunk;
      if (a.vec_ok && j + 3 < a.K) {
        *reinterpret_cast<float4*>(qrow + j) =
            make_float4(z[q][0] * invS, z[q][1] * invS, z[q][2] * invS, z[q][3] * invS);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (j + e < a.K) qrow[j + e] = z[q][e] * invS;
      }
    }
  }
}

struct GreedyFinArgs {
  float* q;            // in: raw logits z; out: one-hot at the greedy index
  int64_t ldq;
  int B, K;
  int passes;          // chunks of kFinChunk ids per CTA
  const float2* part;  // [G][B] (max z, its lowest row) of consecutive row tiles
  int G;
  const int* trim_ids;
  int* tokens;
  int64_t ldt;
  int* dev_status;
  int vec_ok;
};

// Greedy drafting (temperature 0): j* = the largest z of row b, ties to the
// lower trimmed index, from the projection's per-tile (max, row) partials;
// q[b, :] = one-hot at j*; token = trim_ids[j*].  Grid (B, chunks of
// a.passes x 1024 ids): every CTA merges the partials itself and writes its
// chunk of q.
__global__ void __launch_bounds__(kFinNT) draft_greedy_finalize_kernel(GreedyFinArgs a) {
  __shared__ float sv[kFinNT / 32];
  __shared__ int si[kFinNT / 32];
  const int b = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  griddep_launch_dependents();  // the next kernel waits for this grid before reading
  griddep_wait();               // the projection has completed
  float v = -INFINITY;
  int idx = 0x7fffffff;
  for (int t = tid; t < a.G; t += kFinNT) {
    const float2 p = a.part[(int64_t)t * a.B + b];
    const int pi = __float_as_int(p.y);
    if (umma::argmax_better(v, idx, p.x, pi)) {
      v = p.x;
      idx = pi;
    }
  }
  umma::warp_argmax(v, idx);
  if (lane == 0) {
    sv[warp] = v;
    si[warp] = idx;
  }
  __syncthreads();
  v = sv[0];
  idx = si[0];
  for (int w = 1; w < kFinNT / 32; ++w)
    if (umma::argmax_better(v, idx, sv[w], si[w])) {
      v = sv[w];
      idx = si[w];
    }
  const bool ok = (v == v) && idx >= 0 && idx < a.K;  // NaN: a non-finite z was seen
  float* qrow = a.q + (int64_t)b * a.ldq;
#pragma unroll 4
  for (int p = 0; p < a.passes; ++p) {
    const int64_t j = ((int64_t)c * a.passes + p) * kFinChunk + 4 * (int64_t)tid;
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = (ok && j + e == idx) ? 1.f : 0.f;
    if (a.vec_ok && j + 3 < a.K) {
      *reinterpret_cast<float4*>(qrow + j) = make_float4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j + e < a.K) qrow[j + e] = o[e];
    }
  }
  if (c == 0 && tid == 0) {
    a.tokens[(int64_t)b * a.ldt] = ok ? a.trim_ids[idx] : -1;
    if (!ok) atomicOr(a.dev_status, VT_DEV_NONFINITE);
  }
}

// ------------------------------------------------------ drafter top-k
// The drafter's k best trimmed candidates at one position (the expansion
// step of a draft tree, VocabTrim section 4.1): the k highest z, ties to the
// lower trimmed index, with log q = log softmax(z / T).  The projection
// writes z2 = z * log2(e) / T and the per-tile softmax partials; each CTA of
// topk_chunk takes 1024 ids and leaves its k best in order; topk_final
// merges the chunks' lists of a row and converts to log q.
constexpr int kTopkMax = 32;
constexpr int kTkNT = 256;               // 8 warps
constexpr int kTkE = 16;                 // ids per lane per chunk
constexpr int kTkSpan = kTkNT * kTkE;    // ids per CTA per pass
constexpr int kTkMaxCL = 8;              // CTAs per row (one cluster)
constexpr int kTkInsertMax = 6;          // more passing ids than this: sort them as a batch

struct TopkArgs {
  const float* z2;       // [B][K]
  int B, K, k;
  const float2* part;    // [G][B]
  int G;
  const int* trim_ids;
  int* out_ids;          // [B][k]
  float* out_logq;       // [B][k]
  int* dev_status;
};

// (value, index) order of the top-k: higher value first, then lower index
__device__ __forceinline__ bool vi_before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// A warp list: lane l holds the l-th entry of a list of 32 (value, index)
// pairs.  One compare-exchange stage of a bitonic network between lanes
// l and l ^ stride; blocks of `size` lanes run best first where
// (l & size) == 0.
__device__ __forceinline__ void wl_stage(float& v, int& x, int size, int stride, int lane) {
  const float pv = __shfl_xor_sync(0xffffffffu, v, stride);
  const int px = __shfl_xor_sync(0xffffffffu, x, stride);
  const bool keep_better = ((lane & size) == 0) == ((lane & stride) == 0);
  if (vi_before(pv, px, v, x) == keep_better) {
    v = pv;
    x = px;
  }
}

__device__ __forceinline__ void wl_sort(float& v, int& x, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) wl_stage(v, x, size, stride, lane);
}

// (v, x) <- the 32 best of the sorted lists (v, x) and (yv, yx) given in
// reverse (lane l holds entry 31 - l), sorted: the lanewise better of the two
// is a bitonic sequence holding the 32 best of both, which one bitonic merge
// network sorts
__device__ __forceinline__ void wl_merge_rev(float& v, int& x, float yv, int yx, int lane) {
  if (vi_before(yv, yx, v, x)) {
    v = yv;
    x = yx;
  }
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) wl_stage(v, x, 32, stride, lane);
}

// The drafter's k best per row b in one cluster of C CTAs (blockIdx.x =
// rank).  Each warp scans chunks of 512 ids (CTA r takes the passes
// r, r + C, ... of 4096 ids) keeping in a warp list the best entries seen.
// Per chunk: the k-th best of the 32 lanes' best ids bounds the chunk's k-th
// best from below, as does the list's k-th entry; the ids not below the
// better bound (usually about k) are gathered through shared memory, sorted
// as one warp list and merged into the list.  When more than 32 pass (ties),
// the chunk goes batch by batch instead: ids that beat the list's k-th entry
// enter it one at a time, or sorted as a batch when many do.  The warps'
// lists then merge pairwise through shared memory, the CTAs' lists in CTA 0
// through distributed shared memory, and lane r of CTA 0's warp 0 writes
// pick r.  Only the first k entries of a list are exact; they are all that
// is compared and output.
__global__ void __launch_bounds__(kTkNT) topk_cluster_kernel(TopkArgs a) {
  constexpr int NW = kTkNT / 32;
  __shared__ float sv[NW][32];
  __shared__ int sx[NW][32];
  __shared__ MS red[NW];
  __shared__ float gv[NW][32];  // a warp's gathered candidates
  __shared__ int gx[NW][32];
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank(), C = (int)cl.num_blocks();
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k1 = a.k - 1;
  griddep_wait();  // the projection has completed
  // the next kernel may start its prologue; it writes only after its own
  // wait, which waits for this whole grid
  griddep_launch_dependents();

  // CTA 0: this thread's share of the row's softmax normaliser
  MS g{kNegBig, 0.f};
  if (rank == 0)
    for (int t = tid; t < a.G; t += kTkNT) {
      const float2 p = a.part[(int64_t)t * a.B + b];
      g = ms_combine(g, MS{p.x, p.y});
    }

  const float* zr = a.z2 + (int64_t)b * a.K;
  float rv = -INFINITY;  // this warp's list
  int rx = 0x7fffffff;
  float tv = -INFINITY;  // its k-th entry
  int tx = 0x7fffffff;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int64_t base = (int64_t)rank * kTkSpan + 32 * kTkE * warp; base < a.K;
       base += (int64_t)C * kTkSpan) {
    float yv[kTkE];
#pragma unroll
    for (int e = 0; e < kTkE; ++e) {
      const int64_t j = base + 32 * e + lane;
      const float v = (j < a.K) ? zr[j] : -INFINITY;
      yv[e] = (v == v) ? v : -INFINITY;  // non-finite rows are flagged from the partials
    }
    // the lane's best id
    float bv = -INFINITY;
    int bx = 0x7fffffff;
#pragma unroll
    for (int e = 0; e < kTkE; ++e) {
      const int64_t j = base + 32 * e + lane;
      if (j < a.K && vi_before(yv[e], (int)j, bv, bx)) {
        bv = yv[e];
        bx = (int)j;
      }
    }
    if (!__any_sync(0xffffffffu, vi_before(bv, bx, tv, tx))) continue;  // nothing beats the list
    // cv: the better of the list's k-th entry and the k-th best lane best
    wl_sort(bv, bx, lane);
    float cv = __shfl_sync(0xffffffffu, bv, k1);
    int cx = __shfl_sync(0xffffffffu, bx, k1);
    if (vi_before(tv, tx, cv, cx)) {
      cv = tv;
      cx = tx;
    }
    unsigned msk[kTkE];
    int n = 0;
#pragma unroll
    for (int e = 0; e < kTkE; ++e) {
      const int64_t j = base + 32 * e + lane;
      msk[e] = __ballot_sync(0xffffffffu, j < a.K && !vi_before(cv, cx, yv[e], (int)j));
      n += __popc(msk[e]);
    }
    if (n <= 32) {
      int off = 0;
#pragma unroll
      for (int e = 0; e < kTkE; ++e) {
        if ((msk[e] >> lane) & 1u) {
          const int slot = off + __popc(msk[e] & lt_mask);
          gv[warp][slot] = yv[e];
          gx[warp][slot] = (int)(base + 32 * e + lane);
        }
        off += __popc(msk[e]);
      }
      __syncwarp();
      float qv = lane < n ? gv[warp][lane] : -INFINITY;
      int qx = lane < n ? gx[warp][lane] : 0x7fffffff;
      __syncwarp();
      wl_sort(qv, qx, lane);
      if (tx == 0x7fffffff) {  // the list is still empty (its k-th entry is padding)
        rv = qv;
        rx = qx;
      } else {
        wl_merge_rev(rv, rx, __shfl_sync(0xffffffffu, qv, 31 - lane),
                     __shfl_sync(0xffffffffu, qx, 31 - lane), lane);
      }
      tv = __shfl_sync(0xffffffffu, rv, k1);
      tx = __shfl_sync(0xffffffffu, rx, k1);
      continue;
    }
#pragma unroll
    for (int e = 0; e < kTkE; ++e) {
      const int64_t j = base + 32 * e + lane;
      const int yx = (j < a.K) ? (int)j : 0x7fffffff;
      const bool pass = vi_before(yv[e], yx, tv, tx);
      unsigned m = __ballot_sync(0xffffffffu, pass);
      if (m == 0u) continue;
      if (__popc(m) > kTkInsertMax) {
        float bv = pass ? yv[e] : -INFINITY;
        int bx = pass ? yx : 0x7fffffff;
        wl_sort(bv, bx, lane);
        wl_merge_rev(rv, rx, __shfl_sync(0xffffffffu, bv, 31 - lane),
                     __shfl_sync(0xffffffffu, bx, 31 - lane), lane);
      } else {
        while (m != 0u) {
          const int src = __ffs(m) - 1;
          m &= m - 1u;
          const float cv = __shfl_sync(0xffffffffu, yv[e], src);
          const int cx = __shfl_sync(0xffffffffu, yx, src);
          // the entries before the candidate are a prefix of the sorted list
          const int pos = __popc(__ballot_sync(0xffffffffu, vi_before(rv, rx, cv, cx)));
          const float uv = __shfl_up_sync(0xffffffffu, rv, 1);
          const int ux = __shfl_up_sync(0xffffffffu, rx, 1);
          if (lane == pos) {
            rv = cv;
            rx = cx;
          } else if (lane > pos) {
            rv = uv;
            rx = ux;
          }
        }
      }
      tv = __shfl_sync(0xffffffffu, rv, k1);
      tx = __shfl_sync(0xffffffffu, rx, k1);
    }
  }
  if (rank == 0) g = block_ms_reduce<kTkNT>(g, red);

  // the CTA's warps, pairwise: slot w <- merge(slot w, slot w + h)
  sv[warp][lane] = rv;
  sx[warp][lane] = rx;
  __syncthreads();
#pragma unroll
  for (int h = NW / 2; h >= 1; h >>= 1) {
    if (warp < h) {
      wl_merge_rev(rv, rx, sv[warp + h][31 - lane], sx[warp + h][31 - lane], lane);
      sv[warp][lane] = rv;
      sx[warp][lane] = rx;
    }
    __syncthreads();
  }
  cl.sync();  // every CTA's list is in its slot 0
  if (rank == 0 && warp > 0) {
    // warp c copies CTA c's list (an empty one past the cluster)
    float v = -INFINITY;
    int x = 0x7fffffff;
    if (warp < C) {
      v = cl.map_shared_rank(&sv[0][0], warp)[lane];
      x = cl.map_shared_rank(&sx[0][0], warp)[lane];
    }
    sv[warp][lane] = v;
    sx[warp][lane] = x;
    rv = v;
    rx = x;
  }
  cl.sync();  // CTA 0 has read the other CTAs' lists; they may exit
  if (rank != 0) return;
#pragma unroll
  for (int h = NW / 2; h >= 1; h >>= 1) {
    if (warp < h) {
      wl_merge_rev(rv, rx, sv[warp + h][31 - lane], sx[warp + h][31 - lane], lane);
      sv[warp][lane] = rv;
      sx[warp][lane] = rx;
    }
    __syncthreads();
  }
  if (warp == 0) {
    const bool ok = g.s > 0.f && isfinite(g.s) && isfinite(g.m);
    if (lane < a.k) {
      const bool have = ok && rx >= 0 && rx < a.K;
      a.out_ids[(int64_t)b * a.k + lane] = have ? a.trim_ids[rx] : -1;
      // log q = (z2 - m) ln 2 - ln S
      a.out_logq[(int64_t)b * a.k + lane] =
          have ? (rv - g.m) * 0.6931471805599453f - logf(g.s) : __int_as_float(0x7fc00000);
    }
    if (lane == 0 && !ok) atomicOr(a.dev_status, VT_DEV_NONFINITE);
  }
}

struct DraftWs {
  float2* part;
  int* status_sink;  // status word of calls that report none (vt_draft_logits)
  size_t bytes;
};

// partial groups: one per 64-row tile (CUDA-core path) or 128-row tile
int max_groups(int K) {
  return (K + kGemvRowTile - 1) / kGemvRowTile;
}

DraftWs carve_draft(void* base, int B, int K) {
  DraftWs w;
  size_t off = 0;
  auto take = [&](size_t n) {
    size_t o = off;
    off = align_up(off + n, 256);
    return o;
  };
  size_t o_part = take((size_t)max_groups(K) * B * sizeof(float2));
  size_t o_s = take(sizeof(int));
  char* p = static_cast<char*>(base);
  w.status_sink = reinterpret_cast<int*>(p + o_s);
  w.part = reinterpret_cast<float2*>(p + o_part);
  w.bytes = off;
  return w;
}

int gemv_bt(int B) {
  if (B >= 16) return 16;
  if (B >= 8) return 8;
  if (B >= 4) return 4;
  if (B >= 2) return 2;
  return 1;
}

template <int BT>
cudaError_t launch_gemv_bt(int grid, cudaStream_t s, const uint16_t* hidden, int B, int H,
                           const uint16_t* W, int K, float out_scale, float* out, int64_t ldo,
                           float2* part, int* zero_ints, int nzero, int* status_to_zero,
                           int vec_ok, int greedy) {
  const size_t smem = (size_t)BT * H * sizeof(uint16_t);
  auto kern = draft_gemv_kernel<BT, 4>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, kGemvNT, smem, s>>>(hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero,
                                   status_to_zero, vec_ok, greedy);
  return cudaGetLastError();
}

int launch_gemv(cudaStream_t s, const uint16_t* hidden, int B, int H, const uint16_t* W, int K,
                float out_scale, float* out, int64_t ldo, float2* part, int* zero_ints,
                int nzero, int* status_to_zero, int greedy, int* grid_out) {
  const int vec_ok = (H % 8 == 0) && ((reinterpret_cast<uintptr_t>(hidden) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(W) & 15) == 0);
  int bt = gemv_bt(B);
  // the hidden tile must fit in shared memory
  while (bt > 1 && (size_t)bt * H * 2 > 160 * 1024) bt >>= 1;
  if ((size_t)bt * H * 2 > 200 * 1024) return VT_ERR_UNSUPPORTED;
  // one CTA per 64 consecutive rows, so each partial covers one row tile
  const int rows_per_cta = (kGemvNT / 32) * kRowsPerWarp;
  const int grid = (K + rows_per_cta - 1) / rows_per_cta;
  *grid_out = grid;
  cudaError_t e;
  switch (bt) {
    case 16: e = launch_gemv_bt<16>(grid, s, hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero, status_to_zero, vec_ok, greedy); break;
    case 8: e = launch_gemv_bt<8>(grid, s, hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero, status_to_zero, vec_ok, greedy); break;
    case 4: e = launch_gemv_bt<4>(grid, s, hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero, status_to_zero, vec_ok, greedy); break;
    case 2: e = launch_gemv_bt<2>(grid, s, hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero, status_to_zero, vec_ok, greedy); break;
    default: e = launch_gemv_bt<1>(grid, s, hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero, status_to_zero, vec_ok, greedy); break;
  }
  return e == cudaSuccess ? VT_OK : VT_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // looked up once; the initialisation of a function-local static is
  // thread-safe, so concurrent first calls from several host threads agree
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 2-D tensor map of a row-major bf16 [rows, cols] matrix, boxes of
// 64 columns (128 bytes, 128-byte swizzle) x box_rows rows
bool make_bf16_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool umma_supported(const uint16_t* hidden, int B, int H, const uint16_t* W) {
  return B <= 256 && H % 8 == 0 && ((reinterpret_cast<uintptr_t>(hidden) & 15) == 0) &&
         ((reinterpret_cast<uintptr_t>(W) & 15) == 0) && tensor_map_encoder() != nullptr;
}

template <int BN, int TM>
int launch_umma_bn(cudaStream_t s, const CUtensorMap& mw, const CUtensorMap& mh,
                   umma::HeadArgs a, int tiles) {
  constexpr int stage = TM * umma::kABytes + BN * 128;
  // up to ~96 KB of stages for narrow batches: two CTAs per SM that still
  // fit beside the previous draft step's finalize CTAs (so the next
  // projection can start and prefetch while that finalize runs); ~200 KB
  // for wide ones (one CTA per SM)
  const int budget = (BN <= 64) ? 96 * 1024 : 200 * 1024;
  a.stages = std::max(2, std::min(umma::kMaxStages, budget / stage));
  // the ring also holds one transposed accumulator tile in the epilogue
  constexpr size_t kZt =
      (size_t)BN * umma::zt_pitch<BN, umma::kHeadThreads<BN>>() * sizeof(float);
  const size_t smem = std::max((size_t)a.stages * stage, kZt) + 1024;
  auto k = umma::head_umma_kernel<BN, TM>;
  VT_RETURN_IF_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((tiles + TM - 1) / TM));
  cfg.blockDim = dim3(umma::kHeadThreads<BN>);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  VT_RETURN_IF_CUDA(cudaLaunchKernelEx(&cfg, k, mw, mh, a));
  return VT_OK;
}

// z = out_scale * hidden @ W^T on the tensor cores; part[tile][b] partials
int launch_umma(cudaStream_t s, const uint16_t* hidden, int B, int H, const uint16_t* W, int K,
                float out_scale, float* out, int64_t ldo, float2* part, int* zero_ints, int nzero,
                int* status, int status_reset, int greedy, int hidden_ready, int* groups_out) {
  const int BN = (B <= 16) ? 16 : (B <= 32) ? 32 : (B <= 64) ? 64 : (B <= 128) ? 128 : 256;
  CUtensorMap mw, mh;
  if (!make_bf16_map(&mw, W, (uint64_t)K, (uint64_t)H, umma::kBM)) return VT_ERR_CUDA;
  if (!make_bf16_map(&mh, hidden, (uint64_t)B, (uint64_t)H, (uint32_t)BN)) return VT_ERR_CUDA;
  umma::HeadArgs a;
  a.B = B;
  a.H = H;
  a.K = K;
  a.out_scale = out_scale;
  a.out = out;
  a.ldo = ldo;
  a.part = part;
  a.zero_ints = zero_ints;
  a.nzero = nzero;
  a.status = status;
  a.status_reset = status_reset;
  a.stages = 2;
  a.greedy = greedy;
  a.hidden_ready = hidden_ready;
  const int tiles = (K + umma::kBM - 1) / umma::kBM;
  *groups_out = tiles;
  // wide batches: two tiles per CTA share each staged block of hidden states
  // (at B = 256 the hidden states re-read per 128-row tile outweigh W_trim)
  switch (BN) {
    case 16: return launch_umma_bn<16, 1>(s, mw, mh, a, tiles);
    case 32: return launch_umma_bn<32, 1>(s, mw, mh, a, tiles);
    case 64: return launch_umma_bn<64, 1>(s, mw, mh, a, tiles);
    case 128: return launch_umma_bn<128, 2>(s, mw, mh, a, tiles);
    default: return launch_umma_bn<256, 2>(s, mw, mh, a, tiles);
  }
}

// the projection through whichever engine the shapes allow; hidden_ready:
// no kernel still running writes the hidden states (see HeadArgs)
int launch_head(cudaStream_t s, const uint16_t* hidden, int B, int H, const uint16_t* W, int K,
                float out_scale, float* out, int64_t ldo, float2* part, int* zero_ints, int nzero,
                int* status, int status_reset, int greedy, int* groups_out, int* tile_rows_out,
                int hidden_ready = 0) {
  if (umma_supported(hidden, B, H, W)) {
    *tile_rows_out = umma::kBM;
    return launch_umma(s, hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero, status,
                       status_reset, greedy, hidden_ready, groups_out);
  }
  *tile_rows_out = kGemvRowTile;
  return launch_gemv(s, hidden, B, H, W, K, out_scale, out, ldo, part, zero_ints, nzero,
                     status_reset ? status : nullptr, greedy, groups_out);
}

// T > 0, or T == 0 where greedy drafting is allowed
int check_draft_args(const uint16_t* hidden, int B, int H, const uint16_t* W_trim, int K,
                     float T, bool allow_greedy) {
  if (!hidden || !W_trim) return VT_ERR_INVALID_ARG;
  if (B < 1 || B > 4096 || H < 1 || H > 65536 || K < 1) return VT_ERR_INVALID_ARG;
  if (!std::isfinite(T) || T < 0.f || (T == 0.f && !allow_greedy)) return VT_ERR_INVALID_ARG;
  return VT_OK;
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_draft_workspace_bytes(int32_t B, int32_t H, int32_t K) {
  (void)H;
  if (B < 1 || K < 1) return 0;
  return vt::carve_draft(nullptr, B, K).bytes;
}

extern "C" int vt_draft_logits(const uint16_t* hidden, int32_t B, int32_t H,
                               const uint16_t* W_trim, int32_t K, float temperature,
                               float* logits, int64_t ld_logits, void* workspace,
                               size_t workspace_bytes, void* stream) {
  using namespace vt;
  int st = check_draft_args(hidden, B, H, W_trim, K, temperature, false);
  if (st != VT_OK) return st;
  if (!logits || ld_logits < K) return VT_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  DraftWs ws = carve_draft(workspace, B, K);
  if (workspace_bytes < ws.bytes) return VT_ERR_WORKSPACE;
  int groups = 0, tile_rows = 0;
  return launch_head(static_cast<cudaStream_t>(stream), hidden, B, H, W_trim, K,
                     1.0f / temperature, logits, ld_logits, nullptr, nullptr, 0, ws.status_sink, 1, 0,
                     &groups, &tile_rows);
}

extern "C" int vt_draft_step(const uint16_t* hidden, int32_t B, int32_t H,
                             const uint16_t* W_trim, const int32_t* trim_ids, int32_t K,
                             const float* uniforms, float temperature, float* q, int64_t ldq,
                             int32_t* tokens, int64_t ld_tokens, int32_t* dev_status,
                             void* workspace, size_t workspace_bytes, void* stream) {
  return vt::draft_step_impl(hidden, B, H, W_trim, trim_ids, K, uniforms, temperature, q, ldq,
                             tokens, ld_tokens, dev_status, workspace, workspace_bytes, stream,
                             1, 0);
}

int vt::draft_step_impl(const uint16_t* hidden, int32_t B, int32_t H, const uint16_t* W_trim,
                        const int32_t* trim_ids, int32_t K, const float* uniforms,
                        float temperature, float* q, int64_t ldq, int32_t* tokens,
                        int64_t ld_tokens, int32_t* dev_status, void* workspace,
                        size_t workspace_bytes, void* stream, int status_reset,
                        int hidden_ready) {
  using namespace vt;
  int st = check_draft_args(hidden, B, H, W_trim, K, temperature, true);
  if (st != VT_OK) return st;
  const bool greedy = temperature == 0.f;
  if (!trim_ids || (!uniforms && !greedy) || !q || ldq < K || !tokens || ld_tokens < 1 ||
      !dev_status)
    return VT_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  DraftWs ws = carve_draft(workspace, B, K);
  if (workspace_bytes < ws.bytes) return VT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // with status_reset the projection zeroes the status word (its first CTA
  // runs before the finalize grid starts: same stream); without, the flags
  // of this step add to what earlier steps left
  int grid = 0, tile_rows = 0;
  st = launch_head(s, hidden, B, H, W_trim, K, greedy ? 1.0f : VT_LOG2E / temperature, q, ldq,
                   ws.part, nullptr, 0, dev_status, status_reset, greedy ? 1 : 0, &grid,
                   &tile_rows, hidden_ready);
  if (st != VT_OK) return st;
  if (greedy) {
    GreedyFinArgs ga;
    ga.q = q;
    ga.ldq = ldq;
    ga.B = B;
    ga.K = K;
    ga.part = ws.part;
    ga.G = grid;
    ga.trim_ids = trim_ids;
    ga.tokens = tokens;
    ga.ldt = ld_tokens;
    ga.dev_status = dev_status;
    ga.vec_ok = ((reinterpret_cast<uintptr_t>(q) & 15) == 0) && (ldq % 4 == 0);
    const int R = fin_passes(B, K, true);
    ga.passes = R;
    cudaLaunchConfig_t gcfg = {};
    gcfg.gridDim = dim3((unsigned)B, (unsigned)((K + kFinChunk * R - 1) / (kFinChunk * R)));
    gcfg.blockDim = dim3(kFinNT);
    gcfg.stream = s;
    cudaLaunchAttribute gattr[1];
    gattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    gattr[0].val.programmaticStreamSerializationAllowed = 1;
    gcfg.attrs = gattr;
    gcfg.numAttrs = 1;
    VT_RETURN_IF_CUDA(cudaLaunchKernelEx(&gcfg, draft_greedy_finalize_kernel, ga));
    return VT_OK;
  }

  FinArgs fa;
  fa.q = q;
  fa.ldq = ldq;
  fa.B = B;
  fa.K = K;
  fa.part = ws.part;
  fa.G = grid;
  fa.tile_rows = tile_rows;
  fa.u = uniforms;
  fa.trim_ids = trim_ids;
  fa.tokens = tokens;
  fa.ldt = ld_tokens;
  fa.dev_status = dev_status;
  fa.vec_ok = ((reinterpret_cast<uintptr_t>(q) & 15) == 0) && (ldq % 4 == 0);
  const int R = fin_passes(B, K, false);
  fa.passes = R;
  const int nchunk = (K + kFinChunk * R - 1) / (kFinChunk * R);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B, (unsigned)nchunk);
  cfg.blockDim = dim3(kFinNT);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto fk = R == 1 ? draft_finalize_kernel<1>
            : R == 2 ? draft_finalize_kernel<2> : draft_finalize_kernel<4>;
  VT_RETURN_IF_CUDA(cudaLaunchKernelEx(&cfg, fk, fa));
  return VT_OK;
}

extern "C" size_t vt_draft_topk_workspace_bytes(int32_t B, int32_t H, int32_t K, int32_t k) {
  if (B < 1 || K < 1 || k < 1 || k > vt::kTopkMax || k > K) return 0;
  return vt::align_up(vt_draft_workspace_bytes(B, H, K), 256) +
         vt::align_up((size_t)B * K * 4, 256);
}

extern "C" int vt_draft_topk(const uint16_t* hidden, int32_t B, int32_t H, const uint16_t* W_trim,
                             const int32_t* trim_ids, int32_t K, int32_t k, float temperature,
                             int32_t* out_ids, float* out_logq, int32_t* dev_status,
                             void* workspace, size_t workspace_bytes, void* stream) {
  using namespace vt;
  int st = check_draft_args(hidden, B, H, W_trim, K, temperature, false);
  if (st != VT_OK) return st;
  if (!trim_ids || !out_ids || !out_logq || !dev_status || k < 1 || k > kTopkMax || k > K)
    return VT_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  if (workspace_bytes < vt_draft_topk_workspace_bytes(B, H, K, k)) return VT_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  DraftWs dws = carve_draft(ws, B, K);
  const size_t off_z = align_up(vt_draft_workspace_bytes(B, H, K), 256);
  float* z2 = reinterpret_cast<float*>(ws + off_z);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int grid = 0, tile_rows = 0;
  st = launch_head(s, hidden, B, H, W_trim, K, VT_LOG2E / temperature, z2, K, dws.part, nullptr,
                   0, dev_status, 1, 0, &grid, &tile_rows);
  if (st != VT_OK) return st;
  TopkArgs a;
  a.z2 = z2;
  a.B = B;
  a.K = K;
  a.k = k;
  a.part = dws.part;
  a.G = grid;
  a.trim_ids = trim_ids;
  a.out_ids = out_ids;
  a.out_logq = out_logq;
  a.dev_status = dev_status;
  const int C = (int)std::min<int64_t>(kTkMaxCL, ((int64_t)K + kTkSpan - 1) / kTkSpan);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.stream = s;
  cfg.gridDim = dim3((unsigned)C, (unsigned)B);
  cfg.blockDim = dim3(kTkNT);
  VT_RETURN_IF_CUDA(cudaLaunchKernelEx(&cfg, topk_cluster_kernel, a));
  return VT_OK;
}
