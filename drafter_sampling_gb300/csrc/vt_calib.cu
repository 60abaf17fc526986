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
//             ~13% of the stream).  A sample of the first 128K ids picks the
//             hot ids (sample count >= 2) and the most frequent one; the main
//             pass (one CTA per SM) counts the most frequent id in registers,
//             the other hot ids in shared counters found through a bitmap-
//             and-rank table, and cold ids with global atomics.  The sample
//             only decides where an id is counted, so the counts are exact
//             whatever it picks.
//  * radix:   stable LSD radix sort of (~count, id) by 8-bit digits: per-tile
//             digit counts, one exclusive scan, stable scatter.  Stability
//             makes equal counts keep ascending id order, which is the tie
//             rule.  Exact integer work: the result is bit-identical to a
//             sequential sort.
//  * trim:    mark the K ids in inv_map, exclusive scan in id order (tile
//             counts, then tile-local scans that write trim_ids and inv_map),
//             row gather of W.
#include <algorithm>
#include <atomic>
#include <cooperative_groups.h>
#include <utility>

#include "vt_common.cuh"

namespace cg = cooperative_groups;

namespace vt {
namespace {

constexpr int kMainNT = 1024;           // main pass: one CTA of 32 warps per SM
constexpr int kHotMax = 8192;            // hot ids counted in shared memory
constexpr int64_t kSample = 1 << 17;     // ids in the hot-id sample
constexpr unsigned kSampleThr = 2;       // sample count that makes an id hot
constexpr int kHotBitmapMaxV = 1 << 19;  // lookup table + hot counters fit in 160 KB

// Sample histogram of the first `ns` ids.  Each CTA merges its kSampleIds
// ids in a small open-addressing table in shared memory first, so a frequent
// id costs one global atomic per CTA, not one per warp.
constexpr int kSampleNT = 1024;
constexpr int kSampleIds = 2048;   // ids per CTA
constexpr int kHashBits = 12;
constexpr int kHashSlots = 1 << kHashBits;  // > kSampleIds: every insert finds a slot

__global__ void __launch_bounds__(kSampleNT)
hist_sample_kernel(const int* __restrict__ ids, int64_t ns, int V, unsigned* __restrict__ tmp) {
  __shared__ int hkey[kHashSlots];
  __shared__ unsigned hval[kHashSlots];
  for (int i = threadIdx.x; i < kHashSlots; i += kSampleNT) {
    hkey[i] = -1;
    hval[i] = 0u;
  }
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSampleIds;
  for (int e = threadIdx.x; e < kSampleIds; e += kSampleNT) {
    const int64_t i = base + e;
    if (i >= ns) break;
    const int id = __ldg(ids + i);
    if ((unsigned)id >= (unsigned)V) continue;
    unsigned h = ((unsigned)id * 2654435761u) >> (32 - kHashBits);
    for (int probe = 0; probe < kHashSlots; ++probe) {
      const int k = atomicCAS(&hkey[h], -1, id);
      if (k == -1 || k == id) {
        atomicAdd(&hval[h], 1u);
        break;
      }
      h = (h + 1u) & (kHashSlots - 1);
    }
  }
  __syncthreads();
  // the ids are read above without waiting (no kernel just before this one
  // writes them); the sample table they are added to is zeroed by it
  griddep_wait();
  griddep_launch_dependents();
  for (int i = threadIdx.x; i < kHashSlots; i += kSampleNT) {
    const int id = hkey[i];
    if (id >= 0) atomicAdd(tmp + id, hval[i]);
  }
}

// Ids whose sample count reaches `thr` (at most kHotMax kept, any order; one
// slot reservation per CTA), and the most frequent sampled id (ties: the
// smaller id) as the key (count << 32) | (0xffffffff - id).
constexpr int kSelNT = 256;

__global__ void __launch_bounds__(kSelNT)
hot_select_kernel(const unsigned* __restrict__ tmp, int V, unsigned thr, int* __restrict__ hot_list,
                  int* __restrict__ hot_n, unsigned long long* __restrict__ top_key) {
  __shared__ int wcnt[kSelNT / 32];
  __shared__ unsigned long long wkey[kSelNT / 32];
  __shared__ int sbase;
  griddep_wait();  // the sample counts are complete
  griddep_launch_dependents();
  const int i = blockIdx.x * kSelNT + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned c = (i < V) ? tmp[i] : 0u;
  const bool hot = c >= thr;
  const unsigned mask = __ballot_sync(0xffffffffu, hot);
  unsigned long long key = hot ? ((unsigned long long)c << 32) | (0xffffffffu - (unsigned)i) : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
    key = other > key ? other : key;
  }
  if (lane == 0) {
    wcnt[warp] = __popc(mask);
    wkey[warp] = key;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tot = 0;
    unsigned long long km = 0ull;
    for (int w = 0; w < kSelNT / 32; ++w) {
      tot += wcnt[w];
      km = wkey[w] > km ? wkey[w] : km;
    }
    sbase = tot ? atomicAdd(hot_n, tot) : 0;
    if (km) atomicMax(top_key, km);
  }
  __syncthreads();
  if (hot) {
    int slot = sbase + __popc(mask & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) slot += wcnt[w];
    if (slot < kHotMax) hot_list[slot] = i;
  }
}

// Main pass, one CTA per SM.  Hot ids are found through a lookup table in
// shared memory, one 32-bit word per 16 ids: the low half is the bitmap of
// the hot ids among 16w..16w+15, the high half the number of hot ids below
// 16w, so an id's hot-counter slot is one 4-byte load and a popc away; a
// zero word after the table answers every id >= V.  The most frequent
// sampled id is counted in a register (it alone would put several lanes of
// most warps on one shared counter); other hot ids take shared atomics; cold
// ids, where no address is hot, global atomics.  Out-of-range ids are
// detected once, from the largest id seen.  Every CTA adds its nonzero hot
// counters to `counts` at the end.
constexpr int kLutIds = 16;  // ids per lookup word

template <bool HOT>
__global__ void __launch_bounds__(kMainNT, 1)
hist_main_kernel(const int* __restrict__ ids, int64_t n, int V, const int* __restrict__ hot_list,
                 const int* __restrict__ hot_n, const unsigned long long* __restrict__ top_key,
                 unsigned* __restrict__ counts, int* __restrict__ dev_status, int vec_ok) {
  extern __shared__ unsigned lut[];  // [nwords + 1]
  const int nwords = (V + kLutIds - 1) / kLutIds;
  unsigned* hcnt = lut + nwords + 1;  // [kHotMax]
  __shared__ int wsum[kMainNT / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned top = 0u;
  bool use_top = false;  // a most frequent sampled id exists
  if (HOT) {
    for (int w = tid; w <= nwords; w += kMainNT) lut[w] = 0u;
    for (int h = tid; h < kHotMax; h += kMainNT) hcnt[h] = 0u;
  }
  griddep_wait();  // the hot ids are selected and the counts zeroed
  griddep_launch_dependents();
  if (HOT) {
    const unsigned long long tk = *top_key;
    if (tk != 0ull) {
      top = 0xffffffffu - (unsigned)(tk & 0xffffffffull);
      use_top = top < (unsigned)V;
    }
    __syncthreads();
    const int nh = min(*hot_n, kHotMax);
    for (int sl = tid; sl < nh; sl += kMainNT) {
      const int id = hot_list[sl];
      atomicOr(&lut[id / kLutIds], 1u << (id & (kLutIds - 1)));
    }
    __syncthreads();
    // high half of lut[w] = number of hot ids in the words before w (< 2^13)
    const int per = (nwords + kMainNT - 1) / kMainNT;
    const int w0 = tid * per, w1 = min(nwords, w0 + per);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(lut[w]);
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
      const unsigned bits = lut[w];
      lut[w] = bits | ((unsigned)run << 16);
      run += __popc(bits);
    }
    __syncthreads();
  }
  const unsigned uV = (unsigned)V, last = (unsigned)nwords;
  unsigned umax = 0u;  // largest id seen (as unsigned: negative ids are huge)
  unsigned ctop = 0u;
  auto lookup = [&](unsigned uid) -> unsigned {
    return HOT ? lut[min(uid / kLutIds, last)] : 0u;
  };
  auto count1 = [&](unsigned uid, unsigned e) {
    umax = max(umax, uid);
    const unsigned bit = 1u << (uid & (kLutIds - 1));
    const bool is_top = HOT && use_top && uid == top;
    const bool hot = !is_top && (e & bit) != 0u;
    const bool cold = !is_top && (e & bit) == 0u && uid < uV;
    ctop += is_top ? 1u : 0u;
    if (hot) atomicAdd(&hcnt[(e >> 16) + __popc(e & (bit - 1u))], 1u);
    if (cold) atomicAdd(counts + uid, 1u);
  };
  // eight ids: all table loads first, then the counter updates
  auto count8 = [&](const unsigned* v) {
    unsigned e[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) e[k] = lookup(v[k]);
#pragma unroll
    for (int k = 0; k < 8; ++k) count1(v[k], e[k]);
  };
  const int64_t stride = (int64_t)gridDim.x * kMainNT;
  const int64_t t0 = (int64_t)blockIdx.x * kMainNT + tid;
  int64_t tail_start = 0;
  if (vec_ok) {
    const int64_t nv = n / 4;
    const uint4* v4 = reinterpret_cast<const uint4*>(ids);
    int64_t i = t0;
    for (; i + 3 * stride < nv; i += 4 * stride) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = __ldg(v4 + i + u * stride);
      const unsigned a0[8] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w};
      count8(a0);
      const unsigned a1[8] = {q[2].x, q[2].y, q[2].z, q[2].w, q[3].x, q[3].y, q[3].z, q[3].w};
      count8(a1);
    }
    for (; i < nv; i += stride) {
      const uint4 q = __ldg(v4 + i);
      count1(q.x, lookup(q.x));
      count1(q.y, lookup(q.y));
      count1(q.z, lookup(q.z));
      count1(q.w, lookup(q.w));
    }
    tail_start = nv * 4;
  }
  for (int64_t i = tail_start + t0; i < n; i += stride) {
    const unsigned uid = (unsigned)__ldg(ids + i);
    count1(uid, lookup(uid));
  }
  if (umax >= uV) atomicOr(dev_status, VT_DEV_BAD_ID);
  if (HOT) {
    // the register counter of the top id: warp sums, one atomic per warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ctop += __shfl_xor_sync(0xffffffffu, ctop, o);
    if (lane == 0 && use_top && ctop != 0u) atomicAdd(counts + top, ctop);
    __syncthreads();
    // flush: each set bit of the table is one hot id with its slot
    for (int w = tid; w < nwords; w += kMainNT) {
      const unsigned e = lut[w];
      unsigned bits = e & 0xffffu;
      int slot = (int)(e >> 16);
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1u;
        const unsigned c = hcnt[slot++];
        if (c) atomicAdd(counts + w * kLutIds + b, c);
      }
    }
  }
}

// ----------------------------------------------------------- radix sort
// Stable LSD radix sort of the keys ~c[t] (ascending ~count = descending
// count; equal counts keep ascending id order), values t.  Counts are at most
// n, so only the low `bits` = bit length of n bits of ~count vary: they are
// sorted in P passes of D <= 10 bits (P * D >= bits).  One launch per pass:
// tiles of 2048 keys take a ticket in launch order; each ranks its keys by
// digit (per-warp ballots and counters: within a tile keys keep index order),
// publishes its digit counts, then adds up the counts of the tiles with
// smaller tickets (which are running or done, so every wait ends), reorders
// its keys by digit in shared memory and writes each digit's run to its
// place.  The global digit counts of every pass come from one pass over the
// counts beforehand.
constexpr int kRsNT = 1024;
// keys per thread: 2048-key tiles (63 at V = 128256) measured 3.3 us per
// calibrate call faster than 4096-key tiles; 1024 keys were no faster and
// 8192 keys 14 us slower
constexpr int kRsItems = 2;
constexpr int kRsTile = kRsNT * kRsItems;    // keys per tile
constexpr int kRsWarps = kRsNT / 32;
constexpr int kRsMaxD = 10;                  // digit bits: radix <= 1024
constexpr int kRsMaxPasses = 4;
constexpr int kRsMaxV = 1 << 22;
// reads of an unpublished digit count before a tile gives up (a relaxed L2
// read takes ~160 ns when nothing else runs: under a second in all, since
// a thread that gave up once polls no further count)
constexpr uint32_t kRsSpinLimit = 1u << 22;

struct SortPlan {
  int passes, D, radix, ntiles;
};

SortPlan sort_plan(int64_t n, int V) {
  const unsigned long long cmax = (unsigned long long)std::min<int64_t>(n, 0xffffffffll);
  int bits = 1;
  while (bits < 32 && (cmax >> bits) != 0ull) ++bits;
  SortPlan p;
  p.passes = (bits + kRsMaxD - 1) / kRsMaxD;
  p.D = (bits + p.passes - 1) / p.passes;
  p.radix = 1 << p.D;
  p.ntiles = (V + kRsTile - 1) / kRsTile;
  return p;
}

__device__ __forceinline__ unsigned rs_digit(unsigned key, int shift, int radix) {
  return (key >> shift) & (unsigned)(radix - 1);
}

// global digit counts of every pass: ghist[p * radix + d]
__global__ void __launch_bounds__(kRsNT)
sort_hist_kernel(const unsigned* __restrict__ counts, int V, int passes, int D,
                 unsigned* __restrict__ ghist) {
  __shared__ unsigned sh[kRsMaxPasses << kRsMaxD];
  griddep_wait();  // the counts are complete
  const int radix = 1 << D;
  for (int i = threadIdx.x; i < (passes << D); i += kRsNT) sh[i] = 0u;
  const int64_t base = (int64_t)blockIdx.x * kRsTile;
  const int lane = threadIdx.x & 31;
  unsigned key[kRsItems];
  bool valid[kRsItems];
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const int64_t i = base + r * kRsNT + threadIdx.x;
    valid[r] = i < V;
    key[r] = valid[r] ? ~counts[i] : 0u;
  }
  __syncthreads();
  // most counts are small, so most keys share their high digits: a warp
  // whose keys all have the same digit adds once
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const unsigned vmask = __ballot_sync(0xffffffffu, valid[r]);
    for (int p = 0; p < passes; ++p) {
      const unsigned d = rs_digit(key[r], p * D, radix);
      const unsigned d0 = __shfl_sync(0xffffffffu, d, 0);
      if (__all_sync(0xffffffffu, d == d0 || !valid[r])) {
        if (lane == 0 && vmask) atomicAdd(&sh[p * radix + d0], (unsigned)__popc(vmask));
      } else if (valid[r]) {
        atomicAdd(&sh[p * radix + d], 1u);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < (passes << D); i += kRsNT)
    if (sh[i]) atomicAdd(ghist + i, sh[i]);
}

__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// exclusive scan of one value per thread over the block (kRsNT threads)
__device__ __forceinline__ unsigned rs_block_excl(unsigned v, unsigned* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  unsigned pre = 0u;
  for (int w = 0; w < warp; ++w) pre += wsum[w];
  __syncthreads();
  return pre + x - v;
}

struct SortPassArgs {
  const unsigned* counts;   // pass 0 reads keys ~counts[i] and values i
  const unsigned* keys_in;
  const int* vals_in;
  unsigned* keys_out;       // not written by the last pass
  int* vals_out;
  int* topk_ids;            // written by the last pass: ranks < K
  unsigned* keys_last;      // the last pass also writes the sorted keys here, if not null
  int K;
  int V;
  int shift;
  int first, last;
  const unsigned* ghist;    // [radix] global digit counts of this pass
  unsigned* status;         // [ntiles][radix] (1 << 31 | tile count) once published
  int* ticket;
  int* dev_status;
};

template <int D>
__global__ void __launch_bounds__(kRsNT, 1) sort_pass_kernel(SortPassArgs a) {
  constexpr int R = 1 << D;
  extern __shared__ unsigned rs_smem[];
  unsigned* whist = rs_smem;                // [kRsWarps][R]: warp counts, then warp offsets
  unsigned* tstart = whist + kRsWarps * R;  // [R] first slot of digit d in the tile's order
  unsigned* gpos = tstart + R;              // [R] global position of that slot
  unsigned* skey = gpos + R;                // [kRsTile] keys in tile order
  int* sval = reinterpret_cast<int*>(skey + kRsTile);
  __shared__ int s_tile;
  __shared__ unsigned wsum[kRsWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_wait();  // the previous pass (or the counts) is complete
  if (tid == 0) s_tile = atomicAdd(a.ticket, 1);
  for (int i = tid; i < kRsWarps * R; i += kRsNT) whist[i] = 0u;
  __syncthreads();
  const int tile = s_tile;
  const int64_t tbase = (int64_t)tile * kRsTile;
  const int tcnt = (int)((int64_t)a.V - tbase < (int64_t)kRsTile ? (int64_t)a.V - tbase : (int64_t)kRsTile);

  // load (warp-striped: item r of lane l is key 128 w + 32 r + l of the tile)
  unsigned key[kRsItems];
  int val[kRsItems];
  unsigned rd[kRsItems];  // (rank within the warp << 11) | digit; digit == R: no key
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const int j = warp * (32 * kRsItems) + 32 * r + lane;
    const bool valid = j < tcnt;
    const int64_t i = tbase + j;
    if (a.first) {
      key[r] = valid ? ~a.counts[i] : 0u;
      val[r] = (int)i;
    } else {
      key[r] = valid ? a.keys_in[i] : 0u;
      val[r] = valid ? a.vals_in[i] : 0;
    }
    rd[r] = valid ? ((key[r] >> a.shift) & (unsigned)(R - 1)) : (unsigned)R;
  }
  // rank: lanes with the same digit found with one ballot per digit bit
  unsigned* wh = whist + warp * R;
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const unsigned d = rd[r];
    const bool valid = d < (unsigned)R;
    unsigned peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int b = 0; b < D; ++b) {
      const unsigned m = __ballot_sync(0xffffffffu, (d >> b) & 1u);
      peers &= ((d >> b) & 1u) ? m : ~m;
    }
    const unsigned before = valid ? wh[d] : 0u;
    rd[r] = ((before + __popc(peers & lt)) << 11) | d;
    __syncwarp();
    if (valid && (peers & lt) == 0u) wh[d] = before + __popc(peers);
    __syncwarp();
  }
  __syncthreads();

  // per digit: warp offsets, the tile count (published), tile and global starts
  unsigned tc = 0u;
  if (tid < R) {
    unsigned run = 0u;
    for (int w = 0; w < kRsWarps; ++w) {
      const unsigned c = whist[w * R + tid];
      whist[w * R + tid] = run;
      run += c;
    }
    tc = run;
    st_relaxed_u32(a.status + (int64_t)tile * R + tid, 0x80000000u | tc);
  }
  const unsigned ts = rs_block_excl(tc, wsum);
  const unsigned gx = rs_block_excl(tid < R ? a.ghist[tid] : 0u, wsum);
  if (tid < R) {
    tstart[tid] = ts;
    gpos[tid] = gx;
  }
  __syncthreads();
  // counts of the tiles before this one: kRsNT / R threads per digit, each
  // with up to 16 loads in flight (a count not yet published is polled)
  bool timed_out = false;
  {
    constexpr int tpd = (kRsNT / R) > 0 ? (kRsNT / R) : 1;
    const int d = tid % R, h = tid / R;
    unsigned part = 0u;
    for (int t0 = h; t0 < tile; t0 += 16 * tpd) {
      unsigned v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = t0 + j * tpd;
        v[j] = (t < tile) ? ld_relaxed_u32(a.status + (int64_t)t * R + d) : 0x80000000u;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = t0 + j * tpd;
        const unsigned* sp = a.status + (int64_t)t * R + d;
        v[j] = poll_published(sp, v[j], timed_out ? 0u : kRsSpinLimit);
        if ((v[j] >> 31) == 0u) timed_out = true;
        part += v[j] & 0x7fffffffu;
      }
    }
    if (part != 0u) atomicAdd(&gpos[d], part);
  }
  if (timed_out) atomicOr(a.dev_status, VT_DEV_TIMEOUT);
  // reorder the tile by digit in shared memory (stable)
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const unsigned d = rd[r] & 2047u;
    if (d >= (unsigned)R) continue;
    const unsigned slot = tstart[d] + whist[warp * R + d] + (rd[r] >> 11);
    skey[slot] = key[r];
    sval[slot] = val[r];
  }
  __syncthreads();
  // write out: consecutive slots of one digit go to consecutive positions
  for (int j = tid; j < tcnt; j += kRsNT) {
    const unsigned k = skey[j];
    const unsigned d = (k >> a.shift) & (unsigned)(R - 1);
    const unsigned pos = gpos[d] + ((unsigned)j - tstart[d]);
    if (pos >= (unsigned)a.V) continue;  // only after a timed-out wait
    if (a.last) {
      if (pos < (unsigned)a.K) {
        a.topk_ids[pos] = sval[j];
        if (a.keys_last != nullptr) a.keys_last[pos] = k;
      }
    } else {
      a.keys_out[pos] = k;
      a.vals_out[pos] = sval[j];
    }
  }
}

template <int D>
cudaError_t launch_sort_pass(const SortPassArgs& a, int ntiles, cudaStream_t s);

// zero the counts, the sample histogram, the hot-id count, the top key, the
// status word and the sort's tickets, digit counts and tile counts
__global__ void calib_zero_kernel(unsigned* __restrict__ counts, unsigned* __restrict__ tmp, int V,
                                  int* __restrict__ hot_n, unsigned long long* __restrict__ top_key,
                                  int* __restrict__ dev_status, unsigned* __restrict__ zero_words,
                                  int64_t nzero) {
  griddep_wait();  // the previous kernel may still read what is zeroed here
  griddep_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t i = t0; i < V; i += stride) {
    counts[i] = 0u;
    tmp[i] = 0u;
  }
  for (int64_t i = t0; i < nzero; i += stride) zero_words[i] = 0u;
  if (t0 == 0) {
    *hot_n = 0;
    *top_key = 0ull;
    *dev_status = 0;
  }
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

// Index mapper in one cluster of kIdxCL CTAs (V <= kIdxMaxV).  CTA r keeps
// the bitmap of the kept ids among words [r * slice, (r + 1) * slice) in its
// shared memory: every CTA reads all of topk_ids and marks the ids of its
// slice (atomicOr's old value reports duplicates), scans its slice, learns
// the kept-id counts of the other slices through distributed shared memory,
// and writes, in ascending id order, its part of trim_ids and of a rank
// table (bitmap word, kept ids before it) from which the gather kernel
// writes inv_map.
constexpr int kIdxNT = 1024;
constexpr int kIdxCL = 8;
constexpr int kIdxMaxV = 1 << 20;  // 16 KB of bitmap per CTA
constexpr int kIdxBatch = 16;      // topk loads in flight per thread

__global__ void __cluster_dims__(kIdxCL, 1, 1) __launch_bounds__(kIdxNT, 1)
trim_index_kernel(const int* __restrict__ topk, int K, int V, int* __restrict__ trim_ids,
                  uint2* __restrict__ table, int* __restrict__ dev_status) {
  extern __shared__ unsigned bm[];  // [slice] bitmap words, then [slice] local prefix
  __shared__ int wsum[kIdxNT / 32];
  __shared__ int s_total;           // kept ids in this CTA's slice
  __shared__ int s_tot[kIdxCL];     // kept ids in every slice
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwords = (V + 31) >> 5;
  const int slice = (nwords + kIdxCL - 1) / kIdxCL;
  unsigned* pre = bm + slice;
  const int wbeg = rank * slice, wend = min(nwords, wbeg + slice);
  griddep_wait();  // topk_ids come from the previous kernel
  for (int w = tid; w < slice; w += kIdxNT) bm[w] = 0u;
  if (rank == 0 && tid == 0) *dev_status = 0;
  __syncthreads();
  int flags = 0;
  for (int k0 = tid; k0 < K; k0 += kIdxNT * kIdxBatch) {
    int id[kIdxBatch];
#pragma unroll
    for (int r = 0; r < kIdxBatch; ++r) {
      const int k = k0 + r * kIdxNT;
      id[r] = (k < K) ? __ldg(topk + k) : -1;
    }
#pragma unroll
    for (int r = 0; r < kIdxBatch; ++r) {
      if (k0 + r * kIdxNT >= K) continue;  // past the end
      if ((unsigned)id[r] >= (unsigned)V) {
        flags |= VT_DEV_BAD_ID;
        continue;
      }
      const int w = id[r] >> 5;
      if (w < wbeg || w >= wend) continue;  // another CTA's slice
      const unsigned bit = 1u << (id[r] & 31);
      if (atomicOr(&bm[w - wbeg], bit) & bit) flags |= VT_DEV_DUPLICATE_ID;
    }
  }
  if (flags && (rank == 0 || (flags & VT_DEV_DUPLICATE_ID))) atomicOr(dev_status, flags);
  __syncthreads();

  // local exclusive prefix of every word of the slice, in word order
  int base = 0;
  for (int r0 = wbeg; r0 < wend; r0 += kIdxNT) {
    const int w = r0 + tid;
    const int c = (w < wend) ? __popc(bm[w - wbeg]) : 0;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int run = base + x - c, rtot = 0;
    for (int v = 0; v < kIdxNT / 32; ++v) {
      if (v < warp) run += wsum[v];
      rtot += wsum[v];
    }
    if (w < wend) pre[w - wbeg] = (unsigned)run;
    __syncthreads();
    base += rtot;
  }
  if (tid == 0) s_total = base;
  cl.sync();
  if (tid < kIdxCL) s_tot[tid] = *cl.map_shared_rank(&s_total, tid);
  cl.sync();  // every remote read is done: CTAs may leave from here on
  int before = 0, total = 0;
  for (int q = 0; q < kIdxCL; ++q) {
    if (q < rank) before += s_tot[q];
    total += s_tot[q];
  }
  // table and trim_ids: a warp takes 32 consecutive words; for each of them
  // lane l keeps id 32 w + l, so the word's kept ids land at consecutive
  // positions (one coalesced store)
  for (int r0 = wbeg; r0 < wend; r0 += kIdxNT) {
    const int w = r0 + tid;
    const unsigned bits = (w < wend) ? bm[w - wbeg] : 0u;
    const int run = before + ((w < wend) ? (int)pre[w - wbeg] : 0);
    if (w < wend) table[w] = make_uint2(bits, (unsigned)run);
    for (int j = 0; j < 32; ++j) {
      const unsigned wj = __shfl_sync(0xffffffffu, bits, j);
      const int pj = __shfl_sync(0xffffffffu, run, j);
      if ((wj >> lane) & 1u) {
        const int pos = pj + __popc(wj & ((1u << lane) - 1u));
        if (pos < K) trim_ids[pos] = (r0 + warp * 32 + j) * 32 + lane;
      }
    }
  }
  // fewer than K distinct ids (bad input): pad trim_ids
  if (rank == kIdxCL - 1)
    for (int p = total + tid; p < K; p += kIdxNT) trim_ids[p] = -1;
}

// one warp per trimmed row: W_trim[j, :] = W[trim_ids[j], :].  With a rank
// table, thread g < V of the grid also writes inv_map[g].  This kernel
// releases no dependent early: the projection kernel requests W_trim tiles
// before its own dependency wait.
__global__ void __launch_bounds__(256)
trim_gather_kernel(const uint16_t* __restrict__ W, int H, const int* __restrict__ trim_ids, int K,
                   int V, uint16_t* __restrict__ W_trim, int vec_ok, const uint2* __restrict__ table,
                   int* __restrict__ inv_map) {
  griddep_wait();  // trim_ids (and the rank table) are complete
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (table != nullptr && g < V) {
    const uint2 e = table[g >> 5];
    const unsigned bit = 1u << (g & 31);
    inv_map[g] = (e.x & bit) ? (int)(e.y + __popc(e.x & (bit - 1u))) : -1;
  }
  const int warp = (int)(g >> 5);
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
  unsigned* tmp;   // sample histogram [V]
  int* hot_list;   // [kHotMax]
  int* hot_n;      // [1]
  unsigned long long* top_key;  // [1] most frequent sampled id, packed with its count
  // sort state, zeroed before each call (one contiguous block):
  int* tickets;                 // [kRsMaxPasses]
  unsigned* ghist;              // [passes][radix]
  unsigned* status;             // [passes][ntiles][radix]
  unsigned* zero_base;
  size_t bytes;
};

// Workspace sized for the largest sort plan (4 passes, radix 1024); the
// zeroed block is laid out for the plan actually used.
CalibWs carve_calib(void* base, int V, const SortPlan* plan) {
  CalibWs w;
  size_t off = 0;
  auto take = [&](size_t n) {
    size_t o = off;
    off = align_up(off + n, 256);
    return o;
  };
  const size_t ntiles = (size_t)(V + kRsTile - 1) / kRsTile;
  size_t k0 = take((size_t)V * 4), k1 = take((size_t)V * 4);
  size_t v0 = take((size_t)V * 4), v1 = take((size_t)V * 4);
  size_t tm = take((size_t)V * 4);
  size_t hl = take((size_t)kHotMax * 4);
  size_t hn = take(4);
  size_t tk = take(8);
  const size_t zmax = 256 + (size_t)kRsMaxPasses * (1u << kRsMaxD) * 4 +
                      (size_t)kRsMaxPasses * ntiles * (1u << kRsMaxD) * 4;
  size_t zb = take(zmax);
  char* p = static_cast<char*>(base);
  w.tmp = reinterpret_cast<unsigned*>(p + tm);
  w.hot_list = reinterpret_cast<int*>(p + hl);
  w.hot_n = reinterpret_cast<int*>(p + hn);
  w.top_key = reinterpret_cast<unsigned long long*>(p + tk);
  w.keys[0] = reinterpret_cast<unsigned*>(p + k0);
  w.keys[1] = reinterpret_cast<unsigned*>(p + k1);
  w.vals[0] = reinterpret_cast<int*>(p + v0);
  w.vals[1] = reinterpret_cast<int*>(p + v1);
  w.zero_base = reinterpret_cast<unsigned*>(p + zb);
  w.tickets = reinterpret_cast<int*>(p + zb);
  if (plan != nullptr) {
    const size_t gh = (size_t)plan->passes * plan->radix * 4;
    w.ghist = reinterpret_cast<unsigned*>(p + zb + 256);
    w.status = reinterpret_cast<unsigned*>(p + zb + align_up(256 + gh, 256));
  } else {
    w.ghist = nullptr;
    w.status = nullptr;
  }
  w.bytes = off;
  return w;
}

// words of the zeroed block that `plan` uses
int64_t calib_zero_words(int V, const SortPlan& plan) {
  const size_t gh = (size_t)plan.passes * plan.radix * 4;
  const size_t st = (size_t)plan.passes * plan.ntiles * plan.radix * 4;
  (void)V;
  return (int64_t)((align_up(256 + gh, 256) + st) / 4);
}

// launch with programmatic stream serialisation: the kernel may start while
// the previous one drains and waits (griddepcontrol.wait) before reading
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

int num_sms() {
  // per device, filled on first use; concurrent first calls store the same
  // value (relaxed atomics, so there is no data race)
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace
}  // namespace vt

namespace vt {
namespace {
template <int D>
cudaError_t launch_sort_pass(const SortPassArgs& a, int ntiles, cudaStream_t s) {
  constexpr int R = 1 << D;
  const size_t smem = ((size_t)kRsWarps * R + 2 * R + 2 * (size_t)kRsTile) * 4;
  cudaError_t e = cudaFuncSetAttribute(sort_pass_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(sort_pass_kernel<D>, dim3((unsigned)ntiles), dim3(kRsNT), smem, s, a);
}
}  // namespace
}  // namespace vt

extern "C" size_t vt_calibrate_topk_workspace_bytes(int64_t n, int32_t V, int32_t K) {
  (void)n;
  (void)K;
  if (V < 1 || V > vt::kRsMaxV) return 0;
  return vt::carve_calib(nullptr, V, nullptr).bytes;
}

namespace vt {
namespace {
// counts, then the K best-ranked ids; with want_keys the last sort pass also
// leaves the sorted keys (~count, rank order) in the workspace (*keys_out)
int calibrate_impl(const int32_t* ids, int64_t n, int32_t V, int32_t K, uint32_t* counts,
                   int32_t* topk_ids, int32_t* dev_status, void* workspace,
                   size_t workspace_bytes, void* stream, bool want_keys,
                   const unsigned** keys_out) {
  if (n < 0 || V < 1 || V > (1 << 30) || K < 1 || K > V) return VT_ERR_INVALID_ARG;
  if ((n > 0 && !ids) || !counts || !topk_ids || !dev_status) return VT_ERR_INVALID_ARG;
  if (V > kRsMaxV) return VT_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return VT_ERR_WORKSPACE;
  const SortPlan plan = sort_plan(n, V);
  CalibWs ws = carve_calib(workspace, V, &plan);
  if (workspace_bytes < ws.bytes) return VT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the last pass reads keys[(P) & 1] and writes nothing else: keys[(P - 1) & 1] is free
  unsigned* keys_last = want_keys ? ws.keys[(plan.passes - 1) & 1] : nullptr;
  if (keys_out != nullptr) *keys_out = keys_last;

  const int64_t nzero = calib_zero_words(V, plan);
  const int64_t zwork = std::max<int64_t>(V, nzero);
  const int zgrid = (int)std::min<int64_t>((zwork + 255) / 256, 4096);
  VT_RETURN_IF_CUDA(launch_pdl(calib_zero_kernel, dim3((unsigned)zgrid), dim3(256), 0, s, counts,
                               ws.tmp, (int)V, ws.hot_n, ws.top_key, dev_status, ws.zero_base,
                               nzero));
  if (n > 0) {
    const int vec_ok = (reinterpret_cast<uintptr_t>(ids) & 15) == 0;
    const int use_hot = V <= kHotBitmapMaxV;
    if (use_hot) {
      const int64_t ns = std::min<int64_t>(n, kSample);
      const unsigned thr = kSampleThr;
      VT_RETURN_IF_CUDA(launch_pdl(hist_sample_kernel,
                                   dim3((unsigned)((ns + kSampleIds - 1) / kSampleIds)),
                                   dim3(kSampleNT), 0, s, ids, ns, (int)V, ws.tmp));
      VT_RETURN_IF_CUDA(launch_pdl(hot_select_kernel, dim3((unsigned)((V + kSelNT - 1) / kSelNT)),
                                   dim3(kSelNT), 0, s, (const unsigned*)ws.tmp, (int)V, thr,
                                   ws.hot_list, ws.hot_n, ws.top_key));
    }
    const int64_t want = (n / 4 + kMainNT - 1) / kMainNT;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms()));
    if (use_hot) {
      const size_t smem = ((size_t)(V + kLutIds - 1) / kLutIds + 1 + kHotMax) * 4;
      VT_RETURN_IF_CUDA(cudaFuncSetAttribute(hist_main_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem));
      VT_RETURN_IF_CUDA(launch_pdl(hist_main_kernel<true>, dim3((unsigned)grid), dim3(kMainNT),
                                   smem, s, ids, n, (int)V, (const int*)ws.hot_list,
                                   (const int*)ws.hot_n, (const unsigned long long*)ws.top_key,
                                   counts, dev_status, vec_ok));
    } else {
      VT_RETURN_IF_CUDA(launch_pdl(hist_main_kernel<false>, dim3((unsigned)grid), dim3(kMainNT),
                                   0, s, ids, n, (int)V, (const int*)ws.hot_list,
                                   (const int*)ws.hot_n, (const unsigned long long*)ws.top_key,
                                   counts, dev_status, vec_ok));
    }
  }

  // Top-K: radix sort of (~count, id), one launch per pass
  VT_RETURN_IF_CUDA(launch_pdl(sort_hist_kernel, dim3((unsigned)plan.ntiles), dim3(kRsNT), 0, s,
                               (const unsigned*)counts, (int)V, plan.passes, plan.D, ws.ghist));
  for (int p = 0; p < plan.passes; ++p) {
    SortPassArgs a;
    a.counts = counts;
    a.keys_in = ws.keys[(p + 1) & 1];
    a.vals_in = ws.vals[(p + 1) & 1];
    a.keys_out = ws.keys[p & 1];
    a.vals_out = ws.vals[p & 1];
    a.topk_ids = topk_ids;
    a.keys_last = keys_last;
    a.K = K;
    a.V = V;
    a.shift = p * plan.D;
    a.first = p == 0;
    a.last = p == plan.passes - 1;
    a.ghist = ws.ghist + (size_t)p * plan.radix;
    a.status = ws.status + (size_t)p * plan.ntiles * plan.radix;
    a.ticket = ws.tickets + p;
    a.dev_status = dev_status;
    cudaError_t e;
    switch (plan.D) {
      case 1: e = launch_sort_pass<1>(a, plan.ntiles, s); break;
      case 2: e = launch_sort_pass<2>(a, plan.ntiles, s); break;
      case 3: e = launch_sort_pass<3>(a, plan.ntiles, s); break;
      case 4: e = launch_sort_pass<4>(a, plan.ntiles, s); break;
      case 5: e = launch_sort_pass<5>(a, plan.ntiles, s); break;
      case 6: e = launch_sort_pass<6>(a, plan.ntiles, s); break;
      case 7: e = launch_sort_pass<7>(a, plan.ntiles, s); break;
      case 8: e = launch_sort_pass<8>(a, plan.ntiles, s); break;
      case 9: e = launch_sort_pass<9>(a, plan.ntiles, s); break;
      default: e = launch_sort_pass<10>(a, plan.ntiles, s); break;
    }
    VT_RETURN_IF_CUDA(e);
  }
  return VT_OK;
}

// Top-P / minimum-frequency selection over the sorted keys (~count, rank
// order).  select_sums: per 1024 ranks, the sum of the counts and how many
// reach min_count.  select_find: one CTA scans the chunk sums, finds the
// chunk where the running sum reaches P * total, and scans that chunk.
constexpr int kSelChunk = 1024;

__global__ void __launch_bounds__(kSelChunk)
select_sums_kernel(const unsigned* __restrict__ keys, int V, unsigned min_count,
                   unsigned long long* __restrict__ csum, int* __restrict__ ccnt) {
  __shared__ unsigned long long ws[kSelChunk / 32];
  __shared__ int wc[kSelChunk / 32];
  griddep_wait();  // the sort is complete
  const int r = blockIdx.x * kSelChunk + threadIdx.x;
  const unsigned c = (r < V) ? ~keys[r] : 0u;
  unsigned long long v = c;
  int k = (r < V && c >= min_count) ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v += __shfl_xor_sync(0xffffffffu, v, o);
    k += __shfl_xor_sync(0xffffffffu, k, o);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    ws[warp] = v;
    wc[warp] = k;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    int n = 0;
    for (int w = 0; w < kSelChunk / 32; ++w) {
      t += ws[w];
      n += wc[w];
    }
    csum[blockIdx.x] = t;
    ccnt[blockIdx.x] = n;
  }
}

// inclusive block scan of one u64 per thread (kSelChunk threads)
__device__ __forceinline__ unsigned long long sel_scan(unsigned long long v,
                                                       unsigned long long* wsum,
                                                       unsigned long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  unsigned long long pre = 0, tot = 0;
  for (int w = 0; w < kSelChunk / 32; ++w) {
    if (w < warp) pre += wsum[w];
    tot += wsum[w];
  }
  __syncthreads();
  total = tot;
  return pre + x;
}

// mode 0: Top-P; mode 1: minimum count
__global__ void __launch_bounds__(kSelChunk)
select_find_kernel(const unsigned* __restrict__ keys, int V, int nchunks, int mode, double P,
                   const unsigned long long* __restrict__ csum, const int* __restrict__ ccnt,
                   int* __restrict__ k_out) {
  __shared__ unsigned long long wsum[kSelChunk / 32];
  __shared__ int imin[kSelChunk / 32];
  __shared__ int s_chunk;
  __shared__ unsigned long long s_base;
  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nchunks + kSelChunk - 1) / kSelChunk;  // chunks per thread, in order
  const int c0 = tid * per, c1 = min(nchunks, c0 + per);
  if (mode == 1) {
    long long n = 0;
    for (int c = c0; c < c1; ++c) n += ccnt[c];
    unsigned long long tot;
    sel_scan((unsigned long long)n, wsum, tot);
    if (tid == 0) *k_out = (int)tot;
    return;
  }
  unsigned long long mine = 0;
  for (int c = c0; c < c1; ++c) mine += csum[c];
  unsigned long long total;
  const unsigned long long incl = sel_scan(mine, wsum, total);
  if (total == 0ull) {
    if (tid == 0) *k_out = 0;
    return;
  }
  const double thr = P * (double)total;
  // the first chunk whose running sum reaches thr
  int cand = 0x7fffffff;
  unsigned long long run = incl - mine;
  for (int c = c0; c < c1; ++c) {
    run += csum[c];
    if ((double)run >= thr) {
      cand = c;
      break;
    }
  }
  int m = cand;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) imin[warp] = m;
  __syncthreads();
  if (tid == 0) {
    int mm = imin[0];
    for (int w = 1; w < kSelChunk / 32; ++w) mm = min(mm, imin[w]);
    s_chunk = mm;
  }
  __syncthreads();
  const int cs = s_chunk;
  // the base of chunk cs, recomputed by the thread that owns it
  if (cs >= c0 && cs < c1) {
    unsigned long long b = incl - mine;
    for (int c = c0; c < cs; ++c) b += csum[c];
    s_base = b;
  }
  __syncthreads();
  // scan the chunk's counts in rank order
  const int r = cs * kSelChunk + tid;
  const unsigned long long cnt = (cs < nchunks && r < V) ? (unsigned long long)(~keys[r]) : 0ull;
  unsigned long long ctot;
  const unsigned long long cin = sel_scan(cnt, wsum, ctot) + s_base;
  const int hit = ((double)cin >= thr && cnt > 0ull) ? tid : 0x7fffffff;
  m = hit;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) imin[warp] = m;
  __syncthreads();
  if (tid == 0) {
    int mm = imin[0];
    for (int w = 1; w < kSelChunk / 32; ++w) mm = min(mm, imin[w]);
    *k_out = cs * kSelChunk + mm + 1;
  }
}

// the calibration workspace followed by the chunk sums and counts
size_t select_workspace_bytes(int64_t n, int32_t V) {
  (void)n;
  if (V < 1 || V > kRsMaxV) return 0;
  const size_t nchunks = (size_t)(V + kSelChunk - 1) / kSelChunk;
  return carve_calib(nullptr, V, nullptr).bytes + align_up(nchunks * 8, 256) +
         align_up(nchunks * 4, 256);
}

int select_impl(const int32_t* ids, int64_t n, int32_t V, int mode, double P, unsigned min_count,
                uint32_t* counts, int32_t* ranked_ids, int32_t* k_out, int32_t* dev_status,
                void* workspace, size_t workspace_bytes, void* stream) {
  if (!k_out) return VT_ERR_INVALID_ARG;
  const size_t need = select_workspace_bytes(n, V);
  if (need == 0) return V > kRsMaxV ? VT_ERR_UNSUPPORTED : VT_ERR_INVALID_ARG;
  if (workspace_bytes < need) return VT_ERR_WORKSPACE;
  const unsigned* keys = nullptr;
  int st = calibrate_impl(ids, n, V, V, counts, ranked_ids, dev_status, workspace, workspace_bytes,
                          stream, true, &keys);
  if (st != VT_OK) return st;
  const SortPlan plan = sort_plan(n, V);
  const CalibWs ws = carve_calib(workspace, V, &plan);
  char* extra = static_cast<char*>(workspace) + ws.bytes;
  const int nchunks = (V + kSelChunk - 1) / kSelChunk;
  unsigned long long* csum = reinterpret_cast<unsigned long long*>(extra);
  int* ccnt = reinterpret_cast<int*>(extra + align_up((size_t)nchunks * 8, 256));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  VT_RETURN_IF_CUDA(launch_pdl(select_sums_kernel, dim3((unsigned)nchunks), dim3(kSelChunk), 0, s,
                               keys, (int)V, min_count, csum, ccnt));
  VT_RETURN_IF_CUDA(launch_pdl(select_find_kernel, dim3(1), dim3(kSelChunk), 0, s, keys, (int)V,
                               nchunks, mode, P, (const unsigned long long*)csum,
                               (const int*)ccnt, k_out));
  return VT_OK;
}
}  // namespace
}  // namespace vt

extern "C" int vt_calibrate_topk(const int32_t* ids, int64_t n, int32_t V, int32_t K,
                                 uint32_t* counts, int32_t* topk_ids, int32_t* dev_status,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return vt::calibrate_impl(ids, n, V, K, counts, topk_ids, dev_status, workspace,
                            workspace_bytes, stream, false, nullptr);
}

extern "C" size_t vt_calibrate_select_workspace_bytes(int64_t n, int32_t V) {
  return vt::select_workspace_bytes(n, V);
}

extern "C" int vt_calibrate_top_p(const int32_t* ids, int64_t n, int32_t V, double P,
                                  uint32_t* counts, int32_t* ranked_ids, int32_t* k_out,
                                  int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (!(P > 0.0 && P <= 1.0)) return VT_ERR_INVALID_ARG;
  return vt::select_impl(ids, n, V, 0, P, 0u, counts, ranked_ids, k_out, dev_status, workspace,
                         workspace_bytes, stream);
}

extern "C" int vt_calibrate_min_count(const int32_t* ids, int64_t n, int32_t V,
                                      uint32_t min_count, uint32_t* counts, int32_t* ranked_ids,
                                      int32_t* k_out, int32_t* dev_status, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return vt::select_impl(ids, n, V, 1, 0.0, min_count, counts, ranked_ids, k_out, dev_status,
                         workspace, workspace_bytes, stream);
}
extern "C" size_t vt_trim_head_workspace_bytes(int32_t V, int32_t K) {
  (void)K;
  if (V < 1) return 0;
  // rank table (8 bytes per 32 ids) when V <= kIdxMaxV, else tile counts
  const size_t table = (size_t)((V + 31) / 32) * 8;
  const size_t tiles = (size_t)((V + vt::kTrimTile - 1) / vt::kTrimTile) * 4;
  return vt::align_up(std::max(table, tiles), 256);
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
  const int vec_ok = (H % 8 == 0) && ((reinterpret_cast<uintptr_t>(W) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(W_trim) & 15) == 0);
  const int64_t gthreads = std::max<int64_t>((int64_t)K * 32, V);
  const unsigned ggrid = (unsigned)((gthreads + 255) / 256);
  if (V <= kIdxMaxV) {
    // index mapper in one CTA, then the gather (which also writes inv_map)
    uint2* table = static_cast<uint2*>(workspace);
    const size_t smem = (size_t)(((V + 31) / 32 + kIdxCL - 1) / kIdxCL) * 8;
    VT_RETURN_IF_CUDA(launch_pdl(trim_index_kernel, dim3(kIdxCL), dim3(kIdxNT), smem, s, topk_ids,
                                 (int)K, (int)V, trim_ids, table, dev_status));
    VT_RETURN_IF_CUDA(launch_pdl(trim_gather_kernel, dim3(ggrid), dim3(256), 0, s, W, (int)H,
                                 (const int*)trim_ids, (int)K, (int)V, W_trim, vec_ok,
                                 (const uint2*)table, inv_map));
    return VT_OK;
  }
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
  trim_gather_kernel<<<ggrid, 256, 0, s>>>(W, H, trim_ids, K, V, W_trim, vec_ok, nullptr, nullptr);
  VT_RETURN_IF_LAUNCH_FAILED();
  return VT_OK;
}
