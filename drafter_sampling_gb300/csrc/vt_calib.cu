// VocabTrim calibration and head trimming on sm_103a.
//
// Operations ("VocabTrim: Vocabulary Pruning for Efficient Speculative
// Decoding in LLMs", section 3):
//  * Algorithm 1: c[t] += 1 for every token id t of the calibration stream.
//  * eq. (1): Top-K(c, k), here ranked by (count desc, id asc), and
//    W^Trim = W[Top-K(c,k), :] with rows in ascending id order; the index
//    mapper T_{d->t} of Algorithm 2 and its inverse.
//
// Kernels:
//  * hist:    grid-stride 16-byte loads of the id stream; lanes holding the
//             same id merge their increments (match.any) before one atomic,
//             so hot ids of a Zipf stream do not serialise a warp.
//  * radix:   stable LSD radix sort of (~count, id) by 8-bit digits: per-tile
//             digit counts, one exclusive scan, stable scatter.  Stability
//             makes equal counts keep ascending id order, which is the tie
//             rule.  Exact integer work: the result is bit-identical to a
//             sequential sort.
//  * trim:    mark the K ids in inv_map, one-block exclusive scan in id
//             order (writes trim_ids and inv_map), row gather of W.
#include <algorithm>

#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kHistNT = 256;
constexpr int kSortNT = 256;
constexpr int kSortItems = 8;
constexpr int kSortTile = kSortNT * kSortItems;
constexpr int kScanNT = 1024;

// ------------------------------------------------------------- histogram
__device__ __forceinline__ void count_one(int id, int V, unsigned* counts, int& bad) {
  const bool ok = (unsigned)id < (unsigned)V;
  if (!ok) bad = 1;
  const unsigned active = __activemask();
  // group the lanes that hold the same valid id; out-of-range ids form their
  // own groups keyed by a value no valid id can take
  const int key = ok ? id : -1 - (int)(threadIdx.x & 31);
  const unsigned peers = __match_any_sync(active, key);
  const int leader = __ffs(peers) - 1;
  if (ok && (int)(threadIdx.x & 31) == leader) atomicAdd(counts + id, (unsigned)__popc(peers));
}

__global__ void __launch_bounds__(kHistNT)
hist_kernel(const int* __restrict__ ids, int64_t n, int V, unsigned* __restrict__ counts,
            int* __restrict__ dev_status, int vec_ok) {
  int bad = 0;
  const int64_t stride = (int64_t)gridDim.x * kHistNT;
  const int64_t t0 = (int64_t)blockIdx.x * kHistNT + threadIdx.x;
  int64_t tail_start = 0;
  if (vec_ok) {
    const int64_t nv = n / 4;
    const int4* v4 = reinterpret_cast<const int4*>(ids);
    // every lane of a warp runs the same number of iterations so match.any
    // sees full warps; lanes past the end use the sentinel
    const int64_t warp_base = t0 - (threadIdx.x & 31);
    for (int64_t i0 = warp_base; i0 < nv; i0 += stride) {
      const int64_t i = i0 + (threadIdx.x & 31);
      int4 v = make_int4(0, 0, 0, 0);
      const bool in = i < nv;
      if (in) v = __ldg(v4 + i);
      const int vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int id = vals[k];
        const bool ok = in && (unsigned)id < (unsigned)V;
        if (in && !ok) bad = 1;
        const int key = ok ? id : -1 - (int)(threadIdx.x & 31);
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (ok && (int)(threadIdx.x & 31) == __ffs(peers) - 1)
          atomicAdd(counts + id, (unsigned)__popc(peers));
      }
    }
    tail_start = nv * 4;
  }
  for (int64_t i = tail_start + t0; i < n; i += stride) count_one(__ldg(ids + i), V, counts, bad);
  if (bad) atomicOr(dev_status, VT_DEV_BAD_ID);
}

// ----------------------------------------------------------- radix sort
__global__ void sort_init_kernel(const unsigned* __restrict__ counts, int V,
                                 unsigned* __restrict__ keys, int* __restrict__ vals) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < V) {
    keys[i] = ~counts[i];  // ascending ~count = descending count
    vals[i] = i;
  }
}

__global__ void __launch_bounds__(kSortNT)
sort_count_kernel(const unsigned* __restrict__ keys, int V, int shift, int ntiles,
                  int* __restrict__ ghist) {
  __shared__ int h[256];
  h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const int64_t i = base + it * kSortNT + threadIdx.x;
    if (i < V) atomicAdd(&h[(keys[i] >> shift) & 255u], 1);
  }
  __syncthreads();
  ghist[threadIdx.x * ntiles + blockIdx.x] = h[threadIdx.x];
}

// exclusive scan of n ints in place, one block
__global__ void __launch_bounds__(kScanNT) scan_ints_kernel(int* __restrict__ a, int n) {
  __shared__ int wsum[kScanNT / 32];
  const int per = (n + kScanNT - 1) / kScanNT;
  const int s = threadIdx.x * per;
  const int e = min(n, s + per);
  int local = 0;
  for (int i = s; i < e; ++i) local += a[i];
  // block exclusive scan of `local`
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int wpre = 0;
  for (int w = 0; w < warp; ++w) wpre += wsum[w];
  int run = wpre + x - local;
  for (int i = s; i < e; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
}

__global__ void __launch_bounds__(kSortNT)
sort_scatter_kernel(const unsigned* __restrict__ keys_in, const int* __restrict__ vals_in, int V,
                    int shift, int ntiles, const int* __restrict__ goff,
                    unsigned* __restrict__ keys_out, int* __restrict__ vals_out) {
  __shared__ int base_d[256];
  __shared__ int cnt_d[256];
  __shared__ int wc[kSortNT / 32][256];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  base_d[tid] = goff[tid * ntiles + blockIdx.x];
  cnt_d[tid] = 0;
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int it = 0; it < kSortItems; ++it) {
    for (int k = tid; k < (kSortNT / 32) * 256; k += kSortNT) (&wc[0][0])[k] = 0;
    __syncthreads();
    const int64_t i = base + it * kSortNT + tid;
    const bool valid = i < V;
    unsigned key = 0;
    int val = 0, d = 256;
    if (valid) {
      key = keys_in[i];
      val = vals_in[i];
      d = (key >> shift) & 255u;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const int rank = __popc(peers & lt_mask);
    if (valid && rank == 0) wc[warp][d] = __popc(peers);
    __syncthreads();
    if (valid) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += wc[w][d];
      const int pos = base_d[d] + cnt_d[d] + pre + rank;
      keys_out[pos] = key;
      vals_out[pos] = val;
    }
    __syncthreads();
    {
      int tot = 0;
#pragma unroll
      for (int w = 0; w < kSortNT / 32; ++w) tot += wc[w][tid];
      cnt_d[tid] += tot;
    }
    __syncthreads();
  }
}

__global__ void copy_ints_kernel(const int* __restrict__ src, int* __restrict__ dst, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = src[i];
}

// ------------------------------------------------------------------ trim
__global__ void trim_mark_kernel(const int* __restrict__ topk, int K, int V,
                                 int* __restrict__ flags, int* __restrict__ dev_status) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= K) return;
  const int id = topk[k];
  if ((unsigned)id >= (unsigned)V) {
    atomicOr(dev_status, VT_DEV_BAD_ID);
    return;
  }
  if (atomicAdd(flags + id, 1) != 0) atomicOr(dev_status, VT_DEV_DUPLICATE_ID);
}

// flags[id] != 0 marks a kept id.  One block scans in id order and writes
// trim_ids[pos] = id and inv_map[id] = pos (or -1), in place over flags.
__global__ void __launch_bounds__(kScanNT)
trim_scan_kernel(int* __restrict__ inv_map, int V, int K, int* __restrict__ trim_ids) {
  __shared__ int wsum[kScanNT / 32];
  __shared__ int s_total;
  const int per = (V + kScanNT - 1) / kScanNT;
  const int s = threadIdx.x * per;
  const int e = min(V, s + per);
  int local = 0;
  for (int i = s; i < e; ++i) local += (inv_map[i] != 0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int wpre = 0, tot = 0;
  for (int w = 0; w < kScanNT / 32; ++w) {
    if (w < warp) wpre += wsum[w];
    tot += wsum[w];
  }
  if (threadIdx.x == 0) s_total = tot;
  int run = wpre + x - local;
  for (int i = s; i < e; ++i) {
    if (inv_map[i] != 0) {
      if (run < K) trim_ids[run] = i;
      inv_map[i] = (run < K) ? run : -1;
      ++run;
    } else {
      inv_map[i] = -1;
    }
  }
  __syncthreads();
  // fewer than K distinct ids (bad input): pad trim_ids
  for (int p = s_total + threadIdx.x; p < K; p += kScanNT) trim_ids[p] = -1;
}

// one warp per trimmed row: W_trim[j, :] = W[trim_ids[j], :]
__global__ void __launch_bounds__(256)
trim_gather_kernel(const uint16_t* __restrict__ W, int H, const int* __restrict__ trim_ids, int K,
                   int V, uint16_t* __restrict__ W_trim, int vec_ok) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= K) return;
  const int id = trim_ids[warp];
  if ((unsigned)id >= (unsigned)V) return;
  const uint16_t* src = W + (int64_t)id * H;
  uint16_t* dst = W_trim + (int64_t)warp * H;
  if (vec_ok) {
    const int nv = H / 8;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    int i = lane;
    for (; i + 96 < nv; i += 128) {
      uint4 a = __ldg(s4 + i), b = __ldg(s4 + i + 32), c = __ldg(s4 + i + 64),
            d = __ldg(s4 + i + 96);
      d4[i] = a;
      d4[i + 32] = b;
      d4[i + 64] = c;
      d4[i + 96] = d;
    }
    for (; i < nv; i += 32) d4[i] = __ldg(s4 + i);
  } else {
    for (int i = lane; i < H; i += 32) dst[i] = __ldg(src + i);
  }
}

struct CalibWs {
  unsigned* keys[2];
  int* vals[2];
  int* ghist;
  size_t bytes;
};

CalibWs carve_calib(void* base, int V) {
  CalibWs w;
  size_t off = 0;
  auto take = [&](size_t n) {
    size_t o = off;
    off = align_up(off + n, 256);
    return o;
  };
  const int ntiles = (V + kSortTile - 1) / kSortTile;
  size_t k0 = take((size_t)V * 4), k1 = take((size_t)V * 4);
  size_t v0 = take((size_t)V * 4), v1 = take((size_t)V * 4);
  size_t gh = take((size_t)256 * ntiles * 4);
  char* p = static_cast<char*>(base);
  w.keys[0] = reinterpret_cast<unsigned*>(p + k0);
  w.keys[1] = reinterpret_cast<unsigned*>(p + k1);
  w.vals[0] = reinterpret_cast<int*>(p + v0);
  w.vals[1] = reinterpret_cast<int*>(p + v1);
  w.ghist = reinterpret_cast<int*>(p + gh);
  w.bytes = off;
  return w;
}

int num_sms() {
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

}  // namespace
}  // namespace vt

extern "C" size_t vt_calibrate_topk_workspace_bytes(int64_t n, int32_t V, int32_t K) {
  (void)n;
  (void)K;
  if (V < 1) return 0;
  return vt::carve_calib(nullptr, V).bytes;
}

extern "C" int vt_calibrate_topk(const int32_t* ids, int64_t n, int32_t V, int32_t K,
                                 uint32_t* counts, int32_t* topk_ids, int32_t* dev_status,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  using namespace vt;
  if (n < 0 || V < 1 || V > (1 << 30) || K < 1 || K > V) return VT_ERR_INVALID_ARG;
  if ((n > 0 && !ids) || !counts || !topk_ids || !dev_status) return VT_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  CalibWs ws = carve_calib(workspace, V);
  if (workspace_bytes < ws.bytes) return VT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  VT_RETURN_IF_CUDA(cudaMemsetAsync(counts, 0, (size_t)V * 4, s));
  VT_RETURN_IF_CUDA(cudaMemsetAsync(dev_status, 0, 4, s));
  if (n > 0) {
    const int vec_ok = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    int64_t want = (n / 4 + kHistNT - 1) / kHistNT;
    int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms() * 8));
    hist_kernel<<<grid, kHistNT, 0, s>>>(ids, n, V, counts, dev_status, vec_ok);
    VT_RETURN_IF_LAUNCH_FAILED();
  }
  sort_init_kernel<<<(V + 255) / 256, 256, 0, s>>>(counts, V, ws.keys[0], ws.vals[0]);
  VT_RETURN_IF_LAUNCH_FAILED();
  const int ntiles = (V + kSortTile - 1) / kSortTile;
  int cur = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    sort_count_kernel<<<ntiles, kSortNT, 0, s>>>(ws.keys[cur], V, shift, ntiles, ws.ghist);
    VT_RETURN_IF_LAUNCH_FAILED();
    scan_ints_kernel<<<1, kScanNT, 0, s>>>(ws.ghist, 256 * ntiles);
    VT_RETURN_IF_LAUNCH_FAILED();
    sort_scatter_kernel<<<ntiles, kSortNT, 0, s>>>(ws.keys[cur], ws.vals[cur], V, shift, ntiles,
                                                   ws.ghist, ws.keys[cur ^ 1], ws.vals[cur ^ 1]);
    VT_RETURN_IF_LAUNCH_FAILED();
    cur ^= 1;
  }
  copy_ints_kernel<<<(K + 255) / 256, 256, 0, s>>>(ws.vals[cur], topk_ids, K);
  VT_RETURN_IF_LAUNCH_FAILED();
  return VT_OK;
}

extern "C" int vt_trim_head(const uint16_t* W, int32_t V, int32_t H, const int32_t* topk_ids,
                            int32_t K, uint16_t* W_trim, int32_t* trim_ids, int32_t* inv_map,
                            int32_t* dev_status, void* stream) {
  using namespace vt;
  if (!W || !topk_ids || !W_trim || !trim_ids || !inv_map || !dev_status) return VT_ERR_INVALID_ARG;
  if (V < 1 || H < 1 || K < 1 || K > V) return VT_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VT_RETURN_IF_CUDA(cudaMemsetAsync(inv_map, 0, (size_t)V * 4, s));
  VT_RETURN_IF_CUDA(cudaMemsetAsync(dev_status, 0, 4, s));
  trim_mark_kernel<<<(K + 255) / 256, 256, 0, s>>>(topk_ids, K, V, inv_map, dev_status);
  VT_RETURN_IF_LAUNCH_FAILED();
  trim_scan_kernel<<<1, kScanNT, 0, s>>>(inv_map, V, K, trim_ids);
  VT_RETURN_IF_LAUNCH_FAILED();
  const int vec_ok = (H % 8 == 0) && ((reinterpret_cast<uintptr_t>(W) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(W_trim) & 15) == 0);
  const int64_t warps = K;
  trim_gather_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(W, H, trim_ids, K, V, W_trim,
                                                                         vec_ok);
  VT_RETURN_IF_LAUNCH_FAILED();
  return VT_OK;
}
