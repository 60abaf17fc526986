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

// 32 consecutive fp32 columns of this thread's TMEM lane; the wait is part
// of the same statement, so no use of the registers can precede it
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// threads of the projection CTA: wide batches (BN >= 128) add a second
// group of four warps, which reads the other half of the accumulator's
// columns (the same TMEM lanes) in the epilogue
template <int BN>
constexpr int kHeadThreads = BN >= 128 ? 256 : 128;

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

// Row pitch (floats) of the transposed tile: 128 rows plus 4 P, P = threads
// sharing a column in the reduction.  The P threads of a column read
// consecutive 16-byte groups and the next column starts P groups further
// along the banks, so a quarter warp's eight 16-byte reads hit 32 distinct
// banks; the row-major writes (one row per lane) are conflict-free at any
// pitch.
template <int BN, int NT>
__host__ __device__ constexpr int zt_pitch() {
  return kBM + 4 * (BN >= NT ? 1 : NT / BN);
}

// Per-column partials of one accumulator tile held transposed in shared
// memory (zt[b][r], r < nvalid rows of the tile starting at row r0):
// sampling, (max z, sum 2^(z - max)); greedy, (max z, its lowest row), a
// non-finite z counting as NaN, which wins.  P = NT/BN threads share a
// column (narrow batches), interleaved by 16-byte groups (see zt_pitch);
// with BN > NT each thread owns BN/NT columns.
template <int BN, int NT>
__device__ __forceinline__ void tile_partials(const float* zt, const HeadArgs& a, int nvalid,
                                              int r0, int tt, int tid) {
  constexpr int P = BN >= NT ? 1 : NT / BN;          // threads per column
  constexpr int CPT = BN > NT ? BN / NT : 1;         // columns per thread
  constexpr int NF = kBM / 4 / P;                    // 16-byte groups per thread
  const int p = tid % P;
#pragma unroll
  for (int cc = 0; cc < CPT; ++cc) {
    const int b = tid / P + cc * (NT / P);
    const float4* col = reinterpret_cast<const float4*>(zt + b * zt_pitch<BN, NT>());
    if (a.greedy) {
      float v = -INFINITY;
      int idx = 0x7fffffff;
#pragma unroll 4
      for (int k = 0; k < NF; ++k) {
        const int f = p + P * k;
        const float4 x4 = col[f];
        const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 4 * f + e;
          const float w = isfinite(xs[e]) ? xs[e] : __int_as_float(0x7fc00000);
          if (r < nvalid && argmax_better(v, idx, w, r0 + r)) {
            v = w;
            idx = r0 + r;
          }
        }
      }
#pragma unroll
      for (int o = P / 2; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        const int k = __shfl_xor_sync(0xffffffffu, idx, o);
        if (argmax_better(v, idx, w, k)) {
          v = w;
          idx = k;
        }
      }
      if (p == 0 && b < a.B) a.part[(int64_t)tt * a.B + b] = make_float2(v, __int_as_float(idx));
    } else {
      // two passes over the column: its max, then the sum of 2^(z - max);
      // a NaN or +inf z leaves the sum NaN
      float m = kNegBig;
#pragma unroll 4
      for (int k = 0; k < NF; ++k) {
        const int f = p + P * k;
        const float4 x4 = col[f];
        if (4 * f + 3 < nvalid) {
          m = fmaxf(m, fmaxf(fmaxf(x4.x, x4.y), fmaxf(x4.z, x4.w)));
        } else {
          const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (4 * f + e < nvalid) m = fmaxf(m, xs[e]);
        }
      }
#pragma unroll
      for (int o = P / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float s = 0.f;
#pragma unroll 4
      for (int k = 0; k < NF; ++k) {
        const int f = p + P * k;
        const float4 x4 = col[f];
        const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * f + e < nvalid) s += exp2_approx(xs[e] - m);
      }
#pragma unroll
      for (int o = P / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (p == 0 && b < a.B) a.part[(int64_t)tt * a.B + b] = make_float2(m, s);
    }
  }
}

// one CTA per TM consecutive 128-row tiles of W_trim; BN = padded batch
// (16..256, step 16).  With TM = 2 the two tiles share every staged block of
// hidden states (two MMAs per step, one TMEM accumulator each), which halves
// the hidden-state traffic of wide batches.
template <int BN, int TM>
__global__ void __launch_bounds__(kHeadThreads<BN>, 1)
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
  // a weight that no kernel still running writes.  The library's kernels
  // release their dependents only after their own wait, except the drafting
  // finalizes, which release on entry; neither they nor the projection
  // before them write W_trim, and the trim's gather, which does, releases
  // no dependent early.  The hidden states join them when the caller says
  // no running kernel writes them (hidden_ready).  Everything else -- every
  // output -- waits for the previous kernel (griddepcontrol.wait).
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
      for (int i = tid - 64; i < a.nzero; i += kHeadThreads<BN> - 64) a.zero_ints[i] = 0;
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

  // epilogue: all four warps; the next kernel may launch meanwhile.  The
  // threads agree on whether the accumulator is complete, so the barriers
  // below are reached by all of them or by none.
  const bool acc_ok = __syncthreads_and(mbar_wait(&acc_bar, 0) ? 1 : 0) != 0;
  griddep_launch_dependents();
  fence_after_sync();
  if (!acc_ok && tid == 0) s_err = 1;
  constexpr int NT = kHeadThreads<BN>;
  constexpr int CW = BN / (NT / 128);  // accumulator columns read by one warp group
  constexpr int CH = CW >= 32 ? 32 : 16;
  const int quad = warp & 3, col0 = (warp >> 2) * CW;
  const int row = quad * 32 + lane;  // TMEM lane = row of the tile
  // Once every MMA has completed the stage ring is idle (each stage was
  // consumed, so no copy is in flight): it holds one accumulator tile
  // transposed, zt[column b][row], so that the per-column partials are
  // reduced by threads that own whole columns rather than by a chain of
  // warp shuffles per column.
  float* zt = reinterpret_cast<float*>(smem);
#pragma unroll 1
  for (int t = 0; t < TM && acc_ok; ++t) {
    const int j = m0 + t * kBM + row;
    const int tt = tile * TM + t;  // this 128-row tile
#pragma unroll 1
    for (int c0 = col0; c0 < col0 + CW; c0 += CH) {
      float v[CH];
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(t * BN + c0);
      if constexpr (CH == 32) {
        tmem_ld32(taddr, v);
      } else {
        tmem_ld16(taddr, v);
      }
#pragma unroll
      for (int e = 0; e < CH; ++e) {
        const int b = c0 + e;
        const float z = v[e] * a.out_scale;
        if (b < a.B && j < a.K) a.out[(int64_t)b * a.ldo + j] = z;
        if (a.part != nullptr) zt[b * zt_pitch<BN, NT>() + row] = z;
      }
    }
    fence_before_sync();
    __syncthreads();
    if (a.part != nullptr && m0 + t * kBM < a.K)
      tile_partials<BN, NT>(zt, a, min(kBM, a.K - (m0 + t * kBM)), m0 + t * kBM, tt, tid);
    __syncthreads();  // zt is reused by the next tile
  }
  if (tid == 0 && s_err) atomicOr(a.status, VT_DEV_TIMEOUT);
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace umma
}  // namespace vt
