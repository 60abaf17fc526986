// Trimmed-head projection on the 5th-generation tensor cores (sm_103a).
//
//   z[b, j] = out_scale * sum_h hidden[b, h] * W_trim[j, h]
//
// as one tcgen05 GEMM per 128-row tile of W_trim: the trimmed rows are the
// M = 128 operand, the batch is the N = BN operand (BN = batch rounded up to
// a multiple of 16, at most 256), H is the reduction.  Both operands are
// K-major bf16 and arrive by TMA (2-D tensor maps, 128-byte swizzle) into a
// ring of shared-memory stages; one thread issues the MMAs (accumulator in
// tensor memory, fp32), one thread issues the TMA loads, and all four warps
// read the accumulator back (tcgen05.ld, one TMEM lane quarter per warp) to
// scale and store z and fold each tile's rows into per-batch-row online-
// softmax partials (max, sum 2^(z - max)), or, for greedy drafting, into
// (max z, the lowest row holding it).
//
// The first ring stages of W_trim are requested before the kernel waits on
// the previous kernel in the stream (programmatic dependent launch); the
// hidden states come after that wait unless the caller knows that no kernel
// still running writes them (the drafting steps of a captured block), and
// all outputs always do.
//
// Every wait on an mbarrier is bounded: on expiry the kernel records
// VT_DEV_TIMEOUT, drains its own TMA copies (bounded), frees its tensor memory
// and returns.
#pragma once

#include <cuda.h>

#include "vt_common.cuh"

namespace vt {
namespace umma {

constexpr int kBM = 128;            // W_trim rows per tile (MMA M)
constexpr int kBK = 64;             // reduction elements per stage (128 bytes)
constexpr int kABytes = kBM * 128;  // one A stage: 128 rows x 128 bytes
constexpr int kMaxStages = 8;
constexpr int kThreads = 128;
// polls of an mbarrier before a wait gives up: an incomplete try_wait
// suspends for ~3.8 us on sm_103a, so this is about one second, far above
// any wait of a working pipeline (the longest, the epilogue's wait for the
// whole reduction, lasts tens of microseconds)
constexpr uint32_t kWaitLimit = 1u << 18;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// bounded wait for the phase with the given parity to complete: false once
// `limit` polls have found it incomplete
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte
// swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4 (not used by this layout)
//   bits 32-45 stride-dimension byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-47 descriptor version (1)
//   bits 61-63 swizzle mode (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator, both
// operands K-major, shape M x N.
//   bits 4-5 accumulator format (1 = f32); 7-9 A format (1 = bf16);
//   10-12 B format (1 = bf16); 15/16 A/B major (0 = K); 17-22 N >> 3;
//   24-28 M >> 4
__device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive on `bar` once every MMA issued so far by this thread has completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct HeadArgs {
  int B, H, K;
  float out_scale;
  float* out;        // [B, ldo]
  int64_t ldo;
  float2* part;      // [tiles][B] online-softmax partials, or nullptr
  int* zero_ints;    // zeroed by CTA 0 (tickets of the next kernel), or nullptr
  int nzero;
  int* status;       // zeroed by CTA 0 when status_reset, VT_DEV_TIMEOUT on expiry
  int status_reset;
  int stages;
  int greedy;        // part holds (max z, its lowest row) instead of (max, sum 2^(z-max))
  int hidden_ready;  // the hidden states were complete before the previous kernel in the
                     // stream started: they may be staged before the dependency wait
};

// (value, index) pairs of an argmax, ties to the lower index; a NaN value
// (non-finite input seen) wins every comparison so it reaches the result
__device__ __forceinline__ bool argmax_better(float v, int i, float w, int k) {
  if (v != v) return false;
  if (w != w) return true;
  return w > v || (w == v && k < i);
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    const int k = __shfl_xor_sync(0xffffffffu, i, o);
    if (argmax_better(v, i, w, k)) {
      v = w;
      i = k;
    }
  }
}

// one CTA per TM consecutive 128-row tiles of W_trim; BN = padded batch
// (16..256, step 16).  With TM = 2 the two tiles share every staged block of
// hidden states (two MMAs per step, one TMEM accumulator each), which halves
// the hidden-state traffic of wide batches.
template <int BN, int TM>
__global__ void __launch_bounds__(kThreads, 1)
head_umma_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                 HeadArgs a) {
  static_assert(TM == 1 || TM == 2, "one or two tiles per CTA");
  constexpr int kBBytes = BN * 128;
  constexpr int kAB = TM * kABytes;  // the A (W_trim) part of a stage
  constexpr int kNeed = TM * BN;     // accumulator columns
  constexpr uint32_t kCols = kNeed <= 32 ? 32 : (kNeed <= 64 ? 64 : (kNeed <= 128 ? 128 : (kNeed <= 256 ? 256 : 512)));
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int s_err;
  __shared__ MS red[4][BN];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.stages;
  const int stage_bytes = kAB + kBBytes;
  const int tile = blockIdx.x;
  const int m0 = tile * kBM * TM;
  const int nk = (a.H + kBK - 1) / kBK;
  // tiles start their reduction at different column blocks, so the rows
  // streamed at any moment are spread over column offsets (DRAM channels)
  const int rot = tile % nk;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&acc_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_err = 0;
    tma_prefetch_map(&map_w);
    tma_prefetch_map(&map_h);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  // Everything above overlaps the previous kernel's tail.  The producer also
  // fills the first stages with W_trim tiles before waiting on it: W_trim is
  // a weight, never written by the kernel just before this one (the kernels
  // of this library release their dependents only after their own wait, so
  // every older kernel has completed).  The hidden states join them when the
  // caller says no running kernel writes them (hidden_ready).  Everything
  // else -- every output -- waits for the previous kernel
  // (griddepcontrol.wait).
  if (warp == 0 && lane == 0) {
    // TMA producer
    const int pre = min(S, nk);
    for (int kb = 0; kb < pre; ++kb) {
      mbar_expect_tx(&full_bar[kb], (uint32_t)stage_bytes);
#pragma unroll
      for (int t = 0; t < TM; ++t)
        tma_load_2d(smem + (size_t)kb * stage_bytes + t * kABytes, &map_w,
                    ((kb + rot) % nk) * kBK, m0 + t * kBM, &full_bar[kb]);
      if (a.hidden_ready)
        tma_load_2d(smem + (size_t)kb * stage_bytes + kAB, &map_h, ((kb + rot) % nk) * kBK, 0,
                    &full_bar[kb]);
    }
    griddep_wait();
    if (!a.hidden_ready)
      for (int kb = 0; kb < pre; ++kb)
        tma_load_2d(smem + (size_t)kb * stage_bytes + kAB, &map_h, ((kb + rot) % nk) * kBK, 0,
                    &full_bar[kb]);
    int issued = pre;
    bool ok = true;
    for (int kb = pre; kb < nk && ok; ++kb) {
      const int s = kb % S;
      if (kb >= S && !mbar_wait(&empty_bar[s], ((kb / S) - 1) & 1)) {
        ok = false;
        break;
      }
      uint8_t* sa = smem + (size_t)s * stage_bytes;
      mbar_expect_tx(&full_bar[s], (uint32_t)stage_bytes);
      const int x = ((kb + rot) % nk) * kBK;
#pragma unroll
      for (int t = 0; t < TM; ++t) tma_load_2d(sa + t * kABytes, &map_w, x, m0 + t * kBM, &full_bar[s]);
      tma_load_2d(sa + kAB, &map_h, x, 0, &full_bar[s]);
      issued = kb + 1;
    }
    if (!ok) atomicExch(&s_err, 1);
    // drain: every issued copy has landed before this CTA may exit
    for (int kb = (issued > S ? issued - S : 0); kb < issued; ++kb)
      mbar_wait(&full_bar[kb % S], (kb / S) & 1);
  } else {
    griddep_wait();
    if (tile == 0 && warp >= 2) {
      for (int i = tid - 64; i < a.nzero; i += kThreads - 64) a.zero_ints[i] = 0;
      if (tid == 64 && a.status_reset) *a.status = 0;
    }
  }
  if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kBM, BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % S;
      if (!mbar_wait(&full_bar[s], (kb / S) & 1)) {
        atomicExch(&s_err, 1);
        break;
      }
      fence_after_sync();
      const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
      const uint64_t bdesc = sw128_desc(sa + kAB);
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        const uint64_t adesc = sw128_desc(sa + t * kABytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // +32 bytes along K per 16-element step (descriptor address field is >> 4)
          mma_bf16(tmem + (uint32_t)(t * BN), adesc + 2 * kk, bdesc + 2 * kk, idesc,
                   (kb > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit(&empty_bar[s]);
    }
    mma_commit(&acc_bar);
  }
  __syncwarp();

  // epilogue: all four warps; the next kernel may launch meanwhile
  const bool acc_ok = mbar_wait(&acc_bar, 0);
  griddep_launch_dependents();
  fence_after_sync();
  const int row = warp * 32 + lane;
#pragma unroll 1
  for (int t = 0; t < TM; ++t) {
    const int j = m0 + t * kBM + row;
    const int tt = tile * TM + t;  // this 128-row tile
    if (acc_ok) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(t * BN + c0), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int b = c0 + e;
          const float z = v[e] * a.out_scale;
          if (b < a.B && j < a.K) a.out[(int64_t)b * a.ldo + j] = z;
          if (a.part != nullptr && a.greedy) {
            float v = (j < a.K) ? (isfinite(z) ? z : __int_as_float(0x7fc00000)) : -INFINITY;
            int idx = (j < a.K) ? j : 0x7fffffff;
            warp_argmax(v, idx);
            if (lane == 0) red[warp][b] = MS{v, __int_as_float(idx)};
          } else if (a.part != nullptr) {
            MS m = (j < a.K) ? MS{z, 1.f} : MS{kNegBig, 0.f};
            m = warp_ms_reduce(m);
            if (lane == 0) red[warp][b] = m;
          }
        }
      }
    } else {
      atomicExch(&s_err, 1);
    }
    fence_before_sync();
    __syncthreads();
    if (a.part != nullptr && acc_ok && m0 + t * kBM < a.K) {
      for (int b = tid; b < a.B && b < BN; b += kThreads) {
        MS r = red[0][b];
        if (a.greedy) {
          float v = r.m;
          int idx = __float_as_int(r.s);
          for (int w = 1; w < 4; ++w) {
            const float wv = red[w][b].m;
            const int wi = __float_as_int(red[w][b].s);
            if (argmax_better(v, idx, wv, wi)) {
              v = wv;
              idx = wi;
            }
          }
          a.part[(int64_t)tt * a.B + b] = make_float2(v, __int_as_float(idx));
        } else {
          r = ms_combine(r, red[1][b]);
          r = ms_combine(r, red[2][b]);
          r = ms_combine(r, red[3][b]);
          a.part[(int64_t)tt * a.B + b] = make_float2(r.m, r.s);
        }
      }
    }
    __syncthreads();  // red is reused by the next tile
  }
  if (tid == 0 && s_err) atomicOr(a.status, VT_DEV_TIMEOUT);
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace umma
}  // namespace vt
