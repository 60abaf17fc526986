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
//  * hist:    the Zipf head of a token stream would serialise a plain atomic
//             histogram on a few addresses (the most frequent id alone is
//             ~13% of the stream).  A sample of the first 256K ids picks the
//             hot ids (sample count >= sample/4096); the main pass keeps a
//             bitmap and a small hash table of them in shared memory and
//             counts hot ids in per-CTA shared counters, cold ids with
//             global atomics; lanes holding the same id merge first
//             (match.any).  The sample only decides where an id is counted,
//             so the counts are exact whatever it picks.
//  * radix:   stable LSD radix sort of (~count, id) by 8-bit digits: per-tile
//             digit counts, one exclusive scan, stable scatter.  Stability
//             makes equal counts keep ascending id order, which is the tie
//             rule.  Exact integer work: the result is bit-identical to a
//             sequential sort.
//  * trim:    mark the K ids in inv_map, exclusive scan in id order (tile
//             counts, then tile-local scans that write trim_ids and inv_map),
//             row gather of W.
#include <algorithm>

#include "vt_common.cuh"

namespace vt {
namespace {

constexpr int kHistNT = 256;
constexpr int kSortNT = 256;
constexpr int kSortItems = 2;
constexpr int kSortTile = kSortNT * kSortItems;
constexpr int kScanNT = 1024;
constexpr int kHotMax = 8192;            // hot ids counted in shared memory
constexpr int64_t kSample = 1 << 17;     // ids in the hot-id sample
constexpr unsigned kSampleThr = 2;       // sample count that makes an id hot
constexpr int kHotBitmapMaxV = 1 << 19;  // bitmap + prefix of hot ids fit in 96 KB

// sample histogram of the first `ns` ids (warp-aggregated global atomics)
__global__ void __launch_bounds__(kHistNT)
hist_sample_kernel(const int* __restrict__ ids, int64_t ns, int V, unsigned* __restrict__ tmp) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kHistNT;
  for (int64_t i0 = (int64_t)blockIdx.x * kHistNT + threadIdx.x - lane; i0 < ns; i0 += stride) {
    const int64_t i = i0 + lane;
    const int id = (i < ns) ? __ldg(ids + i) : -1;
    const bool ok = (unsigned)id < (unsigned)V;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? id : -1 - lane);
    if (ok && lane == __ffs(peers) - 1) atomicAdd(tmp + id, (unsigned)__popc(peers));
  }
}

// ids whose sample count reaches `thr` (at most kHotMax, any order)
__global__ void hot_select_kernel(const unsigned* __restrict__ tmp, int V, unsigned thr,
                                  int* __restrict__ hot_list, int* __restrict__ hot_n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < V && tmp[i] >= thr) {
    const int slot = atomicAdd(hot_n, 1);
    if (slot < kHotMax) hot_list[slot] = i;
  }
}

// Hot ids: a bitmap over [0, V) in shared memory, and their slot = the rank
// of their bit (per-word prefix counts + popc), so the shared counters are
// indexed without a search.  Hot ids take shared atomics (contention stays
// inside one SM); the rest take global atomics, where no address is hot.
__global__ void __launch_bounds__(kHistNT)
hist_main_kernel(const int* __restrict__ ids, int64_t n, int V, const int* __restrict__ hot_list,
                 const int* __restrict__ hot_n, unsigned* __restrict__ counts,
                 int* __restrict__ dev_status, int vec_ok, int use_hot) {
  extern __shared__ unsigned smem[];
  const int nwords = (V + 31) / 32;
  unsigned* bitmap = smem;                                              // [nwords]
  unsigned short* prefix = reinterpret_cast<unsigned short*>(smem + nwords);  // [nwords]
  unsigned* hcnt = smem + nwords + (nwords + 1) / 2;                    // [kHotMax]
  __shared__ int wsum[kHistNT / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (use_hot) {
    for (int w = tid; w < nwords; w += kHistNT) bitmap[w] = 0;
    for (int h = tid; h < kHotMax; h += kHistNT) hcnt[h] = 0;
    __syncthreads();
    const int nh = min(*hot_n, kHotMax);
    for (int sl = tid; sl < nh; sl += kHistNT) {
      const int id = hot_list[sl];
      atomicOr(&bitmap[id >> 5], 1u << (id & 31));
    }
    __syncthreads();
    // prefix[w] = number of hot ids in words before w
    const int per = (nwords + kHistNT - 1) / kHistNT;
    const int w0 = tid * per, w1 = min(nwords, w0 + per);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bitmap[w]);
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int run = x - c;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int w = w0; w < w1; ++w) {
      prefix[w] = (unsigned short)run;
      run += __popc(bitmap[w]);
    }
    __syncthreads();
  }
  int bad = 0;
  auto count = [&](int id) {
    if ((unsigned)id >= (unsigned)V) {
      bad = 1;
      return;
    }
    if (use_hot) {
      const unsigned word = bitmap[id >> 5];
      const unsigned bit = 1u << (id & 31);
      if (word & bit) {
        atomicAdd(&hcnt[prefix[id >> 5] + __popc(word & (bit - 1))], 1u);
        return;
      }
    }
    atomicAdd(counts + id, 1u);
  };
  const int64_t stride = (int64_t)gridDim.x * kHistNT;
  const int64_t t0 = (int64_t)blockIdx.x * kHistNT + tid;
  int64_t tail_start = 0;
  if (vec_ok) {
    const int64_t nv = n / 4;
    const int4* v4 = reinterpret_cast<const int4*>(ids);
    int64_t i = t0;
    for (; i + stride < nv; i += 2 * stride) {
      const int4 a = __ldg(v4 + i), b = __ldg(v4 + i + stride);
      count(a.x); count(a.y); count(a.z); count(a.w);
      count(b.x); count(b.y); count(b.z); count(b.w);
    }
    if (i < nv) {
      const int4 a = __ldg(v4 + i);
      count(a.x); count(a.y); count(a.z); count(a.w);
    }
    tail_start = nv * 4;
  }
  for (int64_t i = tail_start + t0; i < n; i += stride) count(__ldg(ids + i));
  if (bad) atomicOr(dev_status, VT_DEV_BAD_ID);
  if (use_hot) {
    __syncthreads();
    // flush: each set bit of the bitmap is one hot id with its slot
    for (int w = tid; w < nwords; w += kHistNT) {
      unsigned word = bitmap[w];
      int slot = prefix[w];
      while (word) {
        const int b = __ffs(word) - 1;
        word &= word - 1;
        const unsigned c = hcnt[slot++];
        if (c) atomicAdd(counts + w * 32 + b, c);
      }
    }
  }
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

// exclusive scan of ghist in blocks of kScanBlock entries: each block scans
// its entries in place (block-local offsets) and writes its total; the
// scatter kernel adds the totals of the blocks before.
constexpr int kScanBlock = kScanNT * 4;

__global__ void __launch_bounds__(kScanNT)
scan_blocks_kernel(int* __restrict__ a, int n, int* __restrict__ btot) {
  __shared__ int wsum[kScanNT / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t j = (int64_t)blockIdx.x * kScanBlock + 4 * threadIdx.x;
  int v[4], c = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[e] = (j + e < n) ? a[j + e] : 0;
    c += v[e];
  }
  int x = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int run = x - c, tot = 0;
  for (int w = 0; w < kScanNT / 32; ++w) {
    if (w < warp) run += wsum[w];
    tot += wsum[w];
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (j + e < n) a[j + e] = run;
    run += v[e];
  }
  if (threadIdx.x == 0) btot[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kSortNT)
sort_scatter_kernel(const unsigned* __restrict__ keys_in, const int* __restrict__ vals_in, int V,
                    int shift, int ntiles, const int* __restrict__ goff,
                    const int* __restrict__ btot, int nblk,
                    unsigned* __restrict__ keys_out, int* __restrict__ vals_out) {
  __shared__ int base_d[256];
  __shared__ int cnt_d[256];
  __shared__ int wc[kSortNT / 32][256];
  __shared__ int bpre[64];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    int r = 0;
    for (int k = 0; k < nblk; ++k) {
      bpre[k] = r;
      r += btot[k];
    }
  }
  __syncthreads();
  {
    const int e = tid * ntiles + blockIdx.x;
    base_d[tid] = goff[e] + bpre[e / kScanBlock];
  }
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

// zero the counts, the sample histogram, the hot-id count and the status
__global__ void calib_zero_kernel(unsigned* __restrict__ counts, unsigned* __restrict__ tmp, int V,
                                  int* __restrict__ hot_n, int* __restrict__ dev_status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < V) {
    counts[i] = 0;
    tmp[i] = 0;
  }
  if (i == 0) {
    *hot_n = 0;
    *dev_status = 0;
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

// flags[id] != 0 marks a kept id.  Two passes over tiles of kTrimTile ids:
// count the kept ids of each tile, then every tile adds the counts of the
// tiles before it, scans its own flags in id order and writes
// trim_ids[pos] = id and inv_map[id] = pos (or -1), in place over flags.
constexpr int kTrimNT = 256;
constexpr int kTrimTile = kTrimNT * 4;

__device__ __forceinline__ int block_excl_scan_int(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) pre += wsum[w];
    tot += wsum[w];
  }
  __syncthreads();
  total = tot;
  return pre + x - v;
}

__global__ void __launch_bounds__(kTrimNT)
trim_tilecount_kernel(const int* __restrict__ flags, int V, int* __restrict__ tcount) {
  __shared__ int wsum[kTrimNT / 32];
  const int64_t j = (int64_t)blockIdx.x * kTrimTile + 4 * threadIdx.x;
  int c = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) c += (j + e < V && flags[j + e] != 0);
  int total;
  block_excl_scan_int(c, wsum, total);
  if (threadIdx.x == 0) tcount[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kTrimNT)
trim_write_kernel(int* __restrict__ inv_map, int V, int K, const int* __restrict__ tcount,
                  int ntiles, int* __restrict__ trim_ids) {
  __shared__ int wsum[kTrimNT / 32];
  __shared__ int s_pre, s_all;
  // kept ids in the tiles before this one, and in all tiles
  int pre = 0, all = 0;
  for (int t = threadIdx.x; t < ntiles; t += kTrimNT) {
    const int c = tcount[t];
    if (t < (int)blockIdx.x) pre += c;
    all += c;
  }
  int tp, ta;
  block_excl_scan_int(pre, wsum, tp);
  block_excl_scan_int(all, wsum, ta);
  if (threadIdx.x == 0) {
    s_pre = tp;
    s_all = ta;
  }
  __syncthreads();
  const int64_t j = (int64_t)blockIdx.x * kTrimTile + 4 * threadIdx.x;
  int f[4], c = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[e] = (j + e < V) ? (inv_map[j + e] != 0) : 0;
    c += f[e];
  }
  int total;
  int run = s_pre + block_excl_scan_int(c, wsum, total);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (j + e >= V) break;
    if (f[e]) {
      if (run < K) trim_ids[run] = (int)(j + e);
      inv_map[j + e] = (run < K) ? run : -1;
      ++run;
    } else {
      inv_map[j + e] = -1;
    }
  }
  // fewer than K distinct ids (bad input): pad trim_ids
  if (blockIdx.x == 0)
    for (int p = s_all + threadIdx.x; p < K; p += kTrimNT) trim_ids[p] = -1;
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
  int* btot;       // [64] block totals of the offset scan
  unsigned* tmp;   // sample histogram [V]
  int* hot_list;   // [kHotMax]
  int* hot_n;      // [1]
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
  size_t bt = take(64 * 4);
  size_t tm = take((size_t)V * 4);
  size_t hl = take((size_t)kHotMax * 4);
  size_t hn = take(4);
  char* p = static_cast<char*>(base);
  w.btot = reinterpret_cast<int*>(p + bt);
  w.tmp = reinterpret_cast<unsigned*>(p + tm);
  w.hot_list = reinterpret_cast<int*>(p + hl);
  w.hot_n = reinterpret_cast<int*>(p + hn);
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

  calib_zero_kernel<<<(V + 255) / 256, 256, 0, s>>>(counts, ws.tmp, V, ws.hot_n, dev_status);
  VT_RETURN_IF_LAUNCH_FAILED();
  if (n > 0) {
    const int vec_ok = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    const int use_hot = V <= kHotBitmapMaxV;
    if (use_hot) {
      const int64_t ns = std::min<int64_t>(n, kSample);
      const unsigned thr = kSampleThr;
      hist_sample_kernel<<<(unsigned)((ns + kHistNT - 1) / kHistNT), kHistNT, 0, s>>>(ids, ns, V,
                                                                                   ws.tmp);
      VT_RETURN_IF_LAUNCH_FAILED();
      hot_select_kernel<<<(V + 255) / 256, 256, 0, s>>>(ws.tmp, V, thr, ws.hot_list, ws.hot_n);
      VT_RETURN_IF_LAUNCH_FAILED();
    }
    const int nwords = (V + 31) / 32;
    const size_t smem = use_hot ? ((size_t)nwords + (nwords + 1) / 2 + kHotMax) * 4 : 0;
    if (smem > 48 * 1024)
      VT_RETURN_IF_CUDA(cudaFuncSetAttribute(hist_main_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem));
    const int64_t want = (n / 4 + kHistNT - 1) / kHistNT;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms() * 8));
    hist_main_kernel<<<grid, kHistNT, smem, s>>>(ids, n, V, ws.hot_list, ws.hot_n, counts,
                                                 dev_status, vec_ok, use_hot);
    VT_RETURN_IF_LAUNCH_FAILED();
  }
  sort_init_kernel<<<(V + 255) / 256, 256, 0, s>>>(counts, V, ws.keys[0], ws.vals[0]);
  VT_RETURN_IF_LAUNCH_FAILED();
  const int ntiles = (V + kSortTile - 1) / kSortTile;
  const int nblk = (256 * ntiles + kScanBlock - 1) / kScanBlock;
  if (nblk > 64) return VT_ERR_UNSUPPORTED;
  int cur = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    sort_count_kernel<<<ntiles, kSortNT, 0, s>>>(ws.keys[cur], V, shift, ntiles, ws.ghist);
    VT_RETURN_IF_LAUNCH_FAILED();
    scan_blocks_kernel<<<nblk, kScanNT, 0, s>>>(ws.ghist, 256 * ntiles, ws.btot);
    VT_RETURN_IF_LAUNCH_FAILED();
    sort_scatter_kernel<<<ntiles, kSortNT, 0, s>>>(ws.keys[cur], ws.vals[cur], V, shift, ntiles,
                                                   ws.ghist, ws.btot, nblk, ws.keys[cur ^ 1],
                                                   ws.vals[cur ^ 1]);
    VT_RETURN_IF_LAUNCH_FAILED();
    cur ^= 1;
  }
  copy_ints_kernel<<<(K + 255) / 256, 256, 0, s>>>(ws.vals[cur], topk_ids, K);
  VT_RETURN_IF_LAUNCH_FAILED();
  return VT_OK;
}

extern "C" size_t vt_trim_head_workspace_bytes(int32_t V, int32_t K) {
  (void)K;
  if (V < 1) return 0;
  return vt::align_up((size_t)((V + vt::kTrimTile - 1) / vt::kTrimTile) * 4, 256);
}

extern "C" int vt_trim_head(const uint16_t* W, int32_t V, int32_t H, const int32_t* topk_ids,
                            int32_t K, uint16_t* W_trim, int32_t* trim_ids, int32_t* inv_map,
                            int32_t* dev_status, void* workspace, size_t workspace_bytes,
                            void* stream) {
  using namespace vt;
  if (!W || !topk_ids || !W_trim || !trim_ids || !inv_map || !dev_status) return VT_ERR_INVALID_ARG;
  if (V < 1 || V > (1 << 30) || H < 1 || K < 1 || K > V) return VT_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  if (workspace_bytes < vt_trim_head_workspace_bytes(V, K)) return VT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VT_RETURN_IF_CUDA(cudaMemsetAsync(inv_map, 0, (size_t)V * 4, s));
  VT_RETURN_IF_CUDA(cudaMemsetAsync(dev_status, 0, 4, s));
  trim_mark_kernel<<<(K + 255) / 256, 256, 0, s>>>(topk_ids, K, V, inv_map, dev_status);
  VT_RETURN_IF_LAUNCH_FAILED();
  const int ntiles = (V + kTrimTile - 1) / kTrimTile;
  int* tcount = static_cast<int*>(workspace);  // kept-id count of each tile
  trim_tilecount_kernel<<<ntiles, kTrimNT, 0, s>>>(inv_map, V, tcount);
  VT_RETURN_IF_LAUNCH_FAILED();
  trim_write_kernel<<<ntiles, kTrimNT, 0, s>>>(inv_map, V, K, tcount, ntiles, trim_ids);
  VT_RETURN_IF_LAUNCH_FAILED();
  const int vec_ok = (H % 8 == 0) && ((reinterpret_cast<uintptr_t>(W) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(W_trim) & 15) == 0);
  const int64_t warps = K;
  trim_gather_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(W, H, trim_ids, K, V, W_trim,
                                                                         vec_ok);
  VT_RETURN_IF_LAUNCH_FAILED();
  return VT_OK;
}
