// Exact top-K selection by radix digits.
//
// sglang PR 48224 page (sgl-amd-mono #86): each row's "exact top-2048" (section
// Motivation, first paragraph) is chosen by radix selection over slices of the
// row's keys, with the first digit radix_key >> 26 counted in 64 bins during the
// scoring (section Motivation, fourth bullet; section Modifications, commit 4);
// the later digits, the counts and the placement follow in the selection.
//
// Order of keys: the 64-bit composite (radix_key(score) << 32) | ~position,
// larger first, i.e. score descending and, among equal scores, position
// ascending.  The top K composites are exactly the wanted set, so ties at the
// k-th value go to the lowest positions.
//
// The 12-bit histogram of the radix keys (fused into the scoring kernel; built
// by hist12_kernel when idx_topk gets bare scores) gives, for every 12-bit bin,
// the number of keys in higher bins: its exclusive prefix from the top.  The bin
// T holding the k-th key is where that prefix crosses K, and every key in a
// higher bin b belongs at output slots [prefix(b), prefix(b) + count(b)).
//   collect  one CTA per slice of a row (up to kSlice keys, sized so that the grid
//            is about four CTAs per SM): the slice is copied to
//            shared memory while one warp finds T from the row's 64-bin first
//            digit and the 64 twelve-bit bins of that digit.  Keys above T (the
//            winners) are appended to the row's winner list; keys in T (the
//            candidates) to its candidate list, and counted in a 1024-bin
//            histogram of their next 10 bits (the second digit).
//   finish   two CTAs per row.  One sorts the winner list into the first output
//            slots (the winners are fewer than K).  The other takes the
//            candidates whose second digit is above the one holding the k-th
//            key, picks the rest from that digit's bin by the remaining 42 bits,
//            places them by second digit after the winners, orders each digit's
//            few keys by rank, and writes -1 past min(K, bound).  A row with more
//            candidates than the list holds (thousands of equal scores) is
//            resolved digit by digit over the row's scores instead.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kSlice = 8192;              // largest slice (the page's limit)
constexpr int kSliceStep = 1024;          // slices are multiples of this (4 keys x 256 threads)
constexpr int kCollectThreads = 256;
constexpr int kWinList = IDX_MAX_K;        // winners of one slice (at most K)
constexpr int kCandList = 4096;            // candidates of one slice kept in shared memory
constexpr int kCollectSmem = kSlice * 4 + (kWinList + kCandList) * 2;
// Requested per collect CTA: more than a fifth of an SM's shared memory, so that
// at most four CTAs share an SM and the grid spreads over all SMs.
constexpr int kCollectSmemAlloc = 52 * 1024;
constexpr int kThreads = 512;              // hist12 and finish
constexpr int kSortCap = IDX_MAX_K;        // power of two
constexpr int kTilesPerWarp = kSortCap / 64 / (kThreads / 32);   // 64-key sort tiles per warp
constexpr int kFinishSmem = (kTieCap + kSortCap) * 8 + 2 * 4096 * 4;   // candidates, the keys to sort, buckets
// Requested by each finish CTA while the grid has no more CTAs than the device has
// SMs: more than half an SM's shared memory, so that the scheduler gives every CTA
// an SM of its own instead of packing two on one.  Larger grids ask for what the
// kernel uses, so that two CTAs share an SM and the grid needs fewer waves.
constexpr int kFinishSmemAlloc = 120 * 1024;
static_assert(kFinishSmem <= kFinishSmemAlloc, "finish shared memory");
constexpr uint32_t kNoBin = 0xFFFFFFFFu;
static_assert(kTilesPerWarp >= 1 && kSortCap % 64 == 0, "sort tiles");
static_assert(kCollectSmem <= kCollectSmemAlloc, "collect shared memory");

__device__ __forceinline__ unsigned long long composite(uint32_t key, int64_t pos) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}

// The selection's output for slot j of a row: the position, and the score when the
// caller asked for it (recovered exactly from the composite key's radix key).
__device__ __forceinline__ void put(const SelectArgs &a, int64_t at, unsigned long long c) {
  a.out_idx[at] = static_cast<int32_t>(~static_cast<uint32_t>(c & 0xFFFFFFFFull));
  if (a.out_score != nullptr) a.out_score[at] = radix_key_value(static_cast<uint32_t>(c >> 32));
}

__device__ __forceinline__ int nslices(int32_t bound) { return bound > 0 ? (bound + kSlice - 1) / kSlice : 1; }

// Block-wide exclusive scan of v (every thread must call).
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t *scratch /* 33 */, uint32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t x = lane < static_cast<int>(blockDim.x >> 5) ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
    scratch[lane] = x;
  }
  __syncthreads();
  const uint32_t excl = incl - v + (warp > 0 ? scratch[warp - 1] : 0u);
  *total = scratch[(blockDim.x >> 5) - 1];
  __syncthreads();
  return excl;
}

// Among nbins bins taken in descending bin order, the bin holding the need-th key:
// above < need <= above + hist[bin], above = keys in higher bins.  Block-wide.
__device__ void find_bin(const uint32_t *hist, int nbins, uint32_t need, uint32_t *out_bin, uint32_t *out_above,
                         uint32_t *scratch /* >= 36 words */) {
  const int per = (nbins + blockDim.x - 1) / blockDim.x;
  const int tid = threadIdx.x;
  if (tid == 0) {
    scratch[34] = 0u;
    scratch[35] = 0u;
  }
  uint32_t sum = 0;
  for (int m = 0; m < per; ++m) {
    const int i = tid * per + m;
    if (i < nbins) sum += hist[nbins - 1 - i];
  }
  uint32_t total;
  const uint32_t excl = block_excl_scan(sum, scratch, &total);
  if (excl < need && need <= excl + sum) {
    uint32_t above = excl;
    for (int m = 0; m < per; ++m) {
      const int i = tid * per + m;
      if (i >= nbins) break;
      const uint32_t c = hist[nbins - 1 - i];
      if (above + c >= need) {
        scratch[34] = static_cast<uint32_t>(nbins - 1 - i);
        scratch[35] = above;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
  *out_bin = scratch[34];
  *out_above = scratch[35];
  __syncthreads();
}

// ---------------------------------------------------------------------------- idx_topk front
__global__ void select_clear_kernel(const SelectArgs a, const int32_t *row_bound) {
  const int r = blockIdx.x;
  const Workspace &ws = a.ws;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) ws.hist12[static_cast<int64_t>(r) * kHistBins + i] = 0u;
  for (int i = threadIdx.x; i < kSubBins; i += blockDim.x) ws.hist_sub[static_cast<int64_t>(r) * kSubBins + i] = 0u;
  if (threadIdx.x < 64) ws.hist64[static_cast<int64_t>(r) * 64 + threadIdx.x] = 0u;
  if (threadIdx.x < sizeof(RowSelect) / 4) reinterpret_cast<uint32_t *>(&ws.rowsel[r])[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    const int32_t b = row_bound[r];
    const int32_t be = max(0, min(b, a.max_bound));
    if (be != b) flag_status(ws.status, kStatusBadBound);
    ws.bound_eff[r] = be;
  }
}

// The 12-bit histogram of given scores and its 64-bin marginal (one slice of a
// row per CTA).
__global__ void __launch_bounds__(kThreads) hist12_kernel(const SelectArgs a) {
  __shared__ uint32_t h[kHistBins];
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (static_cast<int>(blockIdx.x) >= nslices(B)) return;
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) h[i] = 0u;
  __syncthreads();
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int n = static_cast<int>(min(static_cast<int64_t>(B), begin + kSlice) - begin);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld + begin;
  // every load of the thread goes out before any is counted
  constexpr int kPer = kSlice / kThreads;
  float x[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = i * kThreads + threadIdx.x;
    x[i] = j < n ? __ldcs(row + j) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (i * kThreads + static_cast<int>(threadIdx.x) < n) atomicAdd(&h[radix_key(x[i]) >> 20], 1u);
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += kThreads)
    if (h[i]) atomicAdd(&a.ws.hist12[static_cast<int64_t>(r) * kHistBins + i], h[i]);
  // marginal: warp w sums first digits w, w + 16, ...
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int d = warp; d < 64; d += kThreads / 32) {
    const uint32_t c = __reduce_add_sync(0xffffffffu, h[d * 64 + lane] + h[d * 64 + 32 + lane]);
    if (lane == 0 && c) atomicAdd(&a.ws.hist64[static_cast<int64_t>(r) * 64 + d], c);
  }
}

// The bin holding the need-th key of 64 counts taken from the top, by one warp:
// lane l holds count[63 - l] and count[31 - l].  Returns the bin (or kNoBin when
// the counts sum below need) and the keys in higher bins.
__device__ __forceinline__ uint32_t warp_find64(uint32_t c_hi, uint32_t c_lo, uint32_t need, uint32_t *above) {
  const int lane = threadIdx.x & 31;
  uint32_t inc_hi = c_hi, inc_lo = c_lo;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(0xffffffffu, inc_hi, o);
    const uint32_t b = __shfl_up_sync(0xffffffffu, inc_lo, o);
    if (lane >= o) {
      inc_hi += a;
      inc_lo += b;
    }
  }
  const uint32_t tot_hi = __shfl_sync(0xffffffffu, inc_hi, 31);
  inc_lo += tot_hi;
  const uint32_t m_hi = __ballot_sync(0xffffffffu, inc_hi >= need);
  const uint32_t m_lo = __ballot_sync(0xffffffffu, inc_lo >= need);
  if (m_hi) {
    const int l = __ffs(m_hi) - 1;
    *above = __shfl_sync(0xffffffffu, inc_hi - c_hi, l);
    return 63u - l;
  }
  if (m_lo) {
    const int l = __ffs(m_lo) - 1;
    *above = __shfl_sync(0xffffffffu, inc_lo - c_lo, l);
    return 31u - l;
  }
  *above = __shfl_sync(0xffffffffu, inc_lo, 31);
  return kNoBin;
}

// ---------------------------------------------------------------------------- collect
__global__ void __launch_bounds__(kCollectThreads) collect_kernel(const SelectArgs a) {
  extern __shared__ __align__(128) unsigned char csm[];
  float *vals = reinterpret_cast<float *>(csm);                               // [kSlice]
  uint16_t *wlist = reinterpret_cast<uint16_t *>(csm + kSlice * 4);           // [kWinList]
  uint16_t *clist = wlist + kWinList;                                         // [kCandList]
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t scratch[36];
  __shared__ uint32_t nwin, ncand;
  __shared__ uint32_t wbase_s, cbase_s;
  __shared__ int abort_flag;

  grid_dependency_wait();   // scores and histogram come from the previous launch
  grid_dependency_trigger();
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int32_t B = a.bound[r];
  const int slice = a.slice;
  if (static_cast<int>(blockIdx.x) >= (B > 0 ? (B + slice - 1) / slice : 1)) return;
  const Workspace &ws = a.ws;
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * slice;
  const int n = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(B), begin + slice) - begin));
  const float *src = a.scores + static_cast<int64_t>(r) * a.ld + begin;

  // 1. the slice into shared memory (one bulk copy when the rows are 16-byte aligned)
  const uint32_t bytes = (static_cast<uint32_t>(n) * 4u + 15u) & ~15u;
  if (tid == 0) {
    nwin = 0u;
    ncand = 0u;
    abort_flag = 0;
    if (a.bulk_rows) {
      mbar_init(&bar, 1);
      fence_barrier_init();
      mbar_arrive_expect_tx(&bar, bytes);
      if (bytes > 0u) bulk_load(vals, src, bytes, &bar);
    }
  }
  if (!a.bulk_rows)
    for (int i = tid; i < n; i += kCollectThreads) vals[i] = __ldcg(src + i);

  // 2. meanwhile: the bin T holding the K-th key, from the row's 64-bin first
  //    digit and that digit's 64 twelve-bit bins (one warp, two dependent loads).
  if (threadIdx.x < 32) {
    uint32_t T = kNoBin;
    if (B > a.K) {
      const uint32_t *h64 = ws.hist64 + static_cast<int64_t>(r) * 64;
      uint32_t above_d;
      const uint32_t D = warp_find64(__ldcg(&h64[63 - tid]), __ldcg(&h64[31 - tid]), static_cast<uint32_t>(a.K),
                                     &above_d);
      if (D != kNoBin) {
        const uint32_t *h12 = ws.hist12 + static_cast<int64_t>(r) * kHistBins + D * 64;
        uint32_t above_f;
        const uint32_t f = warp_find64(__ldcg(&h12[63 - tid]), __ldcg(&h12[31 - tid]),
                                       static_cast<uint32_t>(a.K) - above_d, &above_f);
        if (f != kNoBin) T = D * 64 + f;
      }
    }
    if (tid == 0) {
      scratch[34] = T;
      if (blockIdx.x == 0) ws.rowsel[r].T = T;
    }
  }
  __syncthreads();
  const uint32_t T = scratch[34];

  // 3. classify the slice
  if (a.bulk_rows) {
    if (!mbar_wait(&bar, 0, a.wait_limit_ns, &abort_flag)) {
      flag_status(ws.status, kStatusTimeout);
      // The status reports the launch failed.  Before the CTA's shared memory is
      // released, wait once more (again with a limit) for the copy still in
      // flight to land.
      int never = 0;
      mbar_wait(&bar, 0, a.wait_limit_ns, &never);
      return;
    }
  } else {
    __syncthreads();
  }
  {
    // The bins become float thresholds (radix_key is monotone, and -0.0 and +0.0
    // compare equal as floats as they share a key): a winner is x >= fw (its bin
    // above T), a candidate fc <= x < fw (its bin T).  NaN thresholds take nothing.
    const float kNegInf = __uint_as_float(0xFF800000u);
    auto key_floor = [&](uint32_t k) {   // the smallest non-NaN float whose radix key is >= k
      if (k < 0x00800000u) return kNegInf;   // keys below that of -max are -inf's and NaNs'
      return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu) : __uint_as_float(~k);
    };
    const float kNaN = __uint_as_float(0x7FC00000u);
    const float fw = T == kNoBin ? kNegInf
                                 : (T + 1u < static_cast<uint32_t>(kHistBins) ? key_floor((T + 1u) << 20) : kNaN);
    const float fc = T == kNoBin ? kNaN : key_floor(T << 20);
    const float4 *v4 = reinterpret_cast<const float4 *>(vals);
    const int nq = slice / 4 / kCollectThreads;   // this thread's key quads, at most 8
    auto masks = [&](int i, uint32_t &wm, uint32_t &cm) {
      const int q = i * kCollectThreads + tid;
      const float4 x = v4[q];
      const float xs[4] = {x.x, x.y, x.z, x.w};
      wm = 0u;
      cm = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = 4 * q + e < n;
        const bool w = xs[e] >= fw;
        wm |= static_cast<uint32_t>(in && w) << e;
        cm |= static_cast<uint32_t>(in && !w && xs[e] >= fc) << e;
      }
    };
    // pass 1: count this thread's winners and candidates, remember the quads holding any.
    // Nearly every key is below both thresholds: a whole quad inside the slice with no
    // key at or above the lower one (fc, or fw when fc takes nothing) is passed over
    // after four compares.
    const float flo = fc == fc ? fc : fw;
    uint32_t qmask = 0u, cw = 0u, cc = 0u;
    for (int i = 0; i < nq; ++i) {
      const int q = i * kCollectThreads + tid;
      if (4 * q + 3 < n) {
        const float4 x = v4[q];
        if (!(x.x >= flo || x.y >= flo || x.z >= flo || x.w >= flo)) continue;
      }
      uint32_t wm, cm;
      masks(i, wm, cm);
      if (wm | cm) {
        qmask |= 1u << i;
        cw += __popc(wm);
        cc += __popc(cm);
      }
    }
    // offsets in the slice's two lists (16-bit fields: at most kSlice keys of each)
    uint32_t tot;
    const uint32_t ex = block_excl_scan((cw << 16) | cc, scratch, &tot);
    uint32_t wpos = ex >> 16, cpos = ex & 0xFFFFu;
    // One thread reserves both runs on the row's lists (two atomics in flight
    // together); their round trip runs under pass 2.  More candidates than one
    // slice keeps: the finish resolves the row from its scores.
    uint32_t wb = 0u, cb = 0u;
    if (tid == 0) {
      const uint32_t nw0 = min(tot >> 16, static_cast<uint32_t>(kWinList)), nc0 = tot & 0xFFFFu;
      nwin = tot >> 16;
      ncand = nc0;
      wb = nw0 > 0u ? atomicAdd(&ws.rowsel[r].win_count, nw0) : 0u;
      cb = nc0 > 0u ? atomicAdd(&ws.rowsel[r].tie_count, nc0 <= static_cast<uint32_t>(kCandList)
                                                          ? nc0 : static_cast<uint32_t>(kTieCap) + 1u)
                    : 0u;
    }
    // pass 2: the marked quads again, writing the keys' offsets within the slice
    while (qmask) {
      const int i = __ffs(qmask) - 1;
      qmask &= qmask - 1u;
      uint32_t wm, cm;
      masks(i, wm, cm);
      const int j0 = 4 * (i * kCollectThreads + tid);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((wm >> e) & 1u) {
          if (wpos < static_cast<uint32_t>(kWinList)) wlist[wpos] = static_cast<uint16_t>(j0 + e);
          ++wpos;
        }
        if ((cm >> e) & 1u) {
          if (cpos < static_cast<uint32_t>(kCandList)) clist[cpos] = static_cast<uint16_t>(j0 + e);
          ++cpos;
        }
      }
    }
    if (tid == 0) {
      wbase_s = wb;
      cbase_s = cb;
    }
  }
  __syncthreads();

  // 4. winners onto the row's winner list; candidates onto its candidate list
  const uint32_t nw = min(nwin, static_cast<uint32_t>(kWinList));
  const uint32_t nc = ncand;
  unsigned long long *win = ws.win + static_cast<int64_t>(r) * a.K;
  for (uint32_t i = tid; i < nw; i += kCollectThreads) {
    const uint32_t slot = wbase_s + i;
    if (slot < static_cast<uint32_t>(a.K)) {
      const int j = wlist[i];
      win[slot] = composite(radix_key(vals[j]), begin + j);
    }
  }
  if (nc > static_cast<uint32_t>(kCandList)) return;
  unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
  uint32_t *hsub = ws.hist_sub + static_cast<int64_t>(r) * kSubBins;
  for (uint32_t i = tid; i < nc; i += kCollectThreads) {
    const int j = clist[i];
    const uint32_t key = radix_key(vals[j]);
    atomicAdd(&hsub[(key >> 10) & (kSubBins - 1)], 1u);
    const uint32_t slot = cbase_s + i;
    if (slot < static_cast<uint32_t>(kTieCap)) tie[slot] = composite(key, begin + j);
  }
}

// ---------------------------------------------------------------------------- finish
// Sorting n keys (n a power of two, 64 <= n <= kSortCap) in descending order:
// every warp first sorts 64-key tiles in registers (lane l holds keys l and l + 32;
// a bitonic network unrolled at compile time: in-thread swaps for stride 32,
// shuffles below), then log2(n / 64) merge rounds double the sorted runs.  In a
// round each key finds its place in the merged run by a binary search for its
// rank in the partner run (equal keys: the left run's go first), so a round is
// one pass and one barrier.
template <int SIZE, int STRIDE>
__device__ __forceinline__ void tile_stage(unsigned long long &a, unsigned long long &b, int lane) {
  if constexpr (STRIDE == 32) {   // in-thread pair (l, l + 32); SIZE == 64 sorts the whole tile descending
    const bool sw = a < b;
    const unsigned long long x = a, y = b;
    a = sw ? y : x;
    b = sw ? x : y;
  } else {
    const bool lo = (lane & STRIDE) == 0;
    const bool desc_a = (lane & SIZE) == 0;
    const bool desc_b = ((lane + 32) & SIZE) == 0;
    const unsigned long long ya = __shfl_xor_sync(0xffffffffu, a, STRIDE);
    const unsigned long long yb = __shfl_xor_sync(0xffffffffu, b, STRIDE);
    a = ((a < ya) == (lo == desc_a)) ? ya : a;
    b = ((b < yb) == (lo == desc_b)) ? yb : b;
  }
}

template <int SIZE, int STRIDE>
__device__ __forceinline__ void tile_merge(unsigned long long &a, unsigned long long &b, int lane) {
  tile_stage<SIZE, STRIDE>(a, b, lane);
  if constexpr (STRIDE > 1) tile_merge<SIZE, STRIDE / 2>(a, b, lane);
}

template <int SIZE>
__device__ __forceinline__ void tile_sort(unsigned long long &a, unsigned long long &b, int lane) {
  tile_merge<SIZE, SIZE / 2>(a, b, lane);
  if constexpr (SIZE < 64) tile_sort<SIZE * 2>(a, b, lane);
}

// Sorts s[0, n) descending with tmp[0, n) as scratch; returns the buffer that holds
// the result.  Every thread of the block (kThreads) must call.
__device__ unsigned long long *block_sort_desc(unsigned long long *s, unsigned long long *tmp, int n) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kPerThread = kSortCap / kThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ntiles = n >> 6;
  {
    unsigned long long a[kTilesPerWarp], b[kTilesPerWarp];
#pragma unroll
    for (int j = 0; j < kTilesPerWarp; ++j) {
      const int t = warp + j * kWarps;
      if (t < ntiles) {
        a[j] = s[t * 64 + lane];
        b[j] = s[t * 64 + 32 + lane];
      }
    }
#pragma unroll
    for (int j = 0; j < kTilesPerWarp; ++j)
      if (warp + j * kWarps < ntiles) tile_sort<2>(a[j], b[j], lane);
#pragma unroll
    for (int j = 0; j < kTilesPerWarp; ++j) {
      const int t = warp + j * kWarps;
      if (t < ntiles) {
        s[t * 64 + lane] = a[j];
        s[t * 64 + 32 + lane] = b[j];
      }
    }
  }
  __syncthreads();
  unsigned long long *src = s, *dst = tmp;
  for (int lg = 6; (1 << lg) < n; ++lg) {
    const int m = 1 << lg;
    unsigned long long x[kPerThread];
    const unsigned long long *other[kPerThread];
    bool left[kPerThread];
    int pos[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int i = min(k * kThreads + static_cast<int>(threadIdx.x), n - 1);
      x[k] = src[i];
      other[k] = src + (((i >> lg) ^ 1) << lg);
      left[k] = ((i >> lg) & 1) == 0;
      pos[k] = 0;
    }
    // pos = number of partner keys placed before x (binary lifting over a sorted run)
    for (int step = m >> 1; step > 0; step >>= 1) {
#pragma unroll
      for (int k = 0; k < kPerThread; ++k) {
        if (k * kThreads >= n) break;   // uniform over the block
        const unsigned long long v = other[k][pos[k] + step - 1];
        if (left[k] ? v > x[k] : v >= x[k]) pos[k] += step;
      }
    }
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      if (k * kThreads >= n) break;
      const unsigned long long v = other[k][pos[k]];
      if (left[k] ? v > x[k] : v >= x[k]) pos[k] += 1;
      const int i = k * kThreads + static_cast<int>(threadIdx.x);
      if (i < n) dst[((i >> (lg + 1)) << (lg + 1)) + (i & (m - 1)) + pos[k]] = x[k];
    }
    __syncthreads();
    unsigned long long *t = src;
    src = dst;
    dst = t;
  }
  return src;
}

__device__ __forceinline__ int sort_size(int n);

// Sorts s[0, n) descending (1 <= n <= kSortCap) by an order-preserving bucket pass:
// the keys' top 32 bits (the radix key of the score) relative to their minimum, cut
// to 12 bits (the span's top 12 significant bits), give 4096 buckets; a counting
// pass places each bucket's keys in a contiguous group, and each key's rank
// among the members of its group (all 64 bits compared) gives its final slot.
// A key's rank costs one compare per member of its group, so groups of up to
// kGroupMax keys are ranked this way; when some group holds more (many equal or
// near-equal scores) the segment is sorted by block_sort_desc instead.  tmp[] (kSortCap keys)
// and start[], cur[] (4096 words each) are scratch.  Each key leaves through
// emit(slot, key) with its slot in the descending order, from whichever thread
// ranked it.  Every thread of the block must call.
constexpr int kBuckets = 4096;
constexpr int kGroupMax = 256;

template <typename Emit>
__device__ void block_bucket_sort_desc(unsigned long long *s, unsigned long long *tmp, int n, uint32_t *start,
                                       uint32_t *cur, uint32_t *scratch, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // 1. range of the 32-bit score keys
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t k = static_cast<uint32_t>(s[i] >> 32);
    lo = min(lo, k);
    hi = max(hi, k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  for (int i = tid; i < kBuckets; i += kThreads) {
    start[i] = 0u;
    cur[i] = 0u;
  }
  if (lane == 0) {
    scratch[warp] = lo;
    scratch[16 + warp] = hi;
  }
  __syncthreads();
  lo = 0xFFFFFFFFu;
  hi = 0u;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    lo = min(lo, scratch[w]);
    hi = max(hi, scratch[16 + w]);
  }
  const uint32_t span = hi - lo;
  const int shift = span < static_cast<uint32_t>(kBuckets) ? 0 : 32 - __clz(static_cast<int>(span >> 12));
  // 2. bucket counts
  for (int i = tid; i < n; i += kThreads)
    atomicAdd(&start[(static_cast<uint32_t>(s[i] >> 32) - lo) >> shift], 1u);
  __syncthreads();
  // 3. start of each bucket's group, buckets taken from the top; the largest group
  constexpr int per = kBuckets / kThreads;
  uint32_t c[per], sum = 0u, big = 0u;
#pragma unroll
  for (int m = 0; m < per; ++m) {
    c[m] = start[kBuckets - 1 - (tid * per + m)];
    sum += c[m];
    big = max(big, c[m]);
  }
  uint32_t total;
  uint32_t run = block_excl_scan(sum, scratch, &total);
#pragma unroll
  for (int m = 0; m < per; ++m) {
    start[kBuckets - 1 - (tid * per + m)] = run;
    run += c[m];
  }
  const bool fallback = __syncthreads_or(big > static_cast<uint32_t>(kGroupMax)) != 0;
  if (fallback) {
    const int p2 = sort_size(n);
    for (int i = n + tid; i < p2; i += kThreads) s[i] = 0ull;
    __syncthreads();
    const unsigned long long *sorted = block_sort_desc(s, tmp, p2);
    for (int i = tid; i < n; i += kThreads) emit(i, sorted[i]);
    return;
  }
  // 4. each key into its group (arbitrary order within the group)
  for (int i = tid; i < n; i += kThreads) {
    const unsigned long long x = s[i];
    const uint32_t b = (static_cast<uint32_t>(x >> 32) - lo) >> shift;
    tmp[start[b] + atomicAdd(&cur[b], 1u)] = x;
  }
  __syncthreads();
  // 5. rank within the group
  for (int i = tid; i < n; i += kThreads) {
    const unsigned long long x = tmp[i];
    const uint32_t b = (static_cast<uint32_t>(x >> 32) - lo) >> shift;
    const uint32_t g0 = start[b], g1 = start[b] + cur[b];
    uint32_t r = 0u;
    for (uint32_t j = g0; j < g1; ++j) r += tmp[j] > x ? 1u : 0u;
    emit(static_cast<int>(g0 + r), x);   // the key's final slot, straight out
  }
}

__device__ __forceinline__ int sort_size(int n) {
  int p = 64;
  while (p < n) p <<= 1;
  return p;
}

// Digits of the low 52 composite bits, most significant first: two of 10 bits
// (the score bits below the shared 12-bit bin) and three of 11, 11 and 10 bits
// (the inverted position, for exact ties).
__device__ __forceinline__ int digit_shift(int d) {
  return d == 0 ? 42 : d == 1 ? 32 : d == 2 ? 21 : d == 3 ? 10 : 0;
}
__device__ __forceinline__ int digit_width(int d) { return d < 2 ? 10 : d < 4 ? 11 : 10; }

__device__ __forceinline__ unsigned long long low52(unsigned long long c) { return c & ((1ull << 52) - 1); }

// Threshold on the low 52 bits such that exactly `need` of the keys yielded by
// `candidate(i, valid)` (valid = false to skip) are >= it, by digits d0..4 of
// the low 52 bits, starting at digit `d0` (the keys agree on the digits above
// it).  Bits of the returned threshold above digit d0 are 0.
template <typename Get>
__device__ unsigned long long select_threshold(int64_t n, uint32_t need, Get candidate, uint32_t *h /* 2048 */,
                                               uint32_t *scratch, int d0) {
  const int top = digit_shift(d0) + digit_width(d0);
  unsigned long long pre = 0ull;
  for (int d = d0; d < 5; ++d) {
    const int sh = digit_shift(d), wd = digit_width(d);
    const int nb = 1 << wd;
    const unsigned long long upper = ((1ull << (top - sh - wd)) - 1) << (sh + wd);   // digits d0 .. d-1
    for (int i = threadIdx.x; i < nb; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      bool valid;
      const unsigned long long v = candidate(i, valid);
      if (!valid || (v & upper) != pre) continue;
      atomicAdd(&h[(v >> sh) & (nb - 1u)], 1u);
    }
    __syncthreads();
    uint32_t bin, above;
    find_bin(h, nb, need, &bin, &above, scratch);
    const uint32_t cnt = h[bin];
    need -= above;
    pre |= static_cast<unsigned long long>(bin) << sh;
    __syncthreads();
    if (cnt == need) break;            // the whole bin is taken: the lower bits of pre stay 0
  }
  return pre;
}

// Appends `take` lanes' keys to list[] at slots counted by *counter (shared).
__device__ __forceinline__ void warp_push64(bool take, unsigned long long value, unsigned long long *list,
                                            uint32_t *counter, uint32_t cap) {
  const uint32_t ballot = __ballot_sync(0xffffffffu, take);
  if (ballot == 0u) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(ballot) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(ballot)));
  base = __shfl_sync(0xffffffffu, base, leader);
  const uint32_t at = base + __popc(ballot & ((1u << lane) - 1u));
  if (take && at < cap) list[at] = value;
}

__global__ void __launch_bounds__(kThreads) finish_kernel(const SelectArgs a) {
  extern __shared__ unsigned long long sm[];
  unsigned long long *cand = sm;               // [kTieCap]
  unsigned long long *sel = sm + kTieCap;      // [kSortCap]
  uint32_t *bstart = reinterpret_cast<uint32_t *>(sel + kSortCap);   // [kBuckets]
  uint32_t *bcur = bstart + kBuckets;                                // [kBuckets]
  __shared__ uint32_t hbuf[2048];
  __shared__ uint32_t scratch[36];
  __shared__ uint32_t count_s;
  grid_dependency_wait();   // every collect slice has placed its keys
  const int part = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const Workspace &ws = a.ws;
  const int32_t B = a.bound[r];
  const int K = a.K;
  const int nout = min(K, max(B, 0));
  const RowSelect &rs = ws.rowsel[r];
  int32_t *out = a.out_idx + static_cast<int64_t>(r) * K;

  if (part == 0) {
    // The winners (keys above T, fewer than K) are the first output slots: one
    // bucket sort of the row's whole winner list.  The list is read whole together
    // with its length (one round trip, not two); entries past the length are unused.
    const unsigned long long *win = ws.win + static_cast<int64_t>(r) * K;
    constexpr int kPer = IDX_MAX_K / kThreads;
    unsigned long long wv[kPer];
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int i = m * kThreads + tid;
      wv[m] = i < K ? __ldcg(&win[i]) : 0ull;
    }
    const uint32_t nw = min(__ldcg(&rs.win_count), static_cast<uint32_t>(nout));
    if (nw == 0u) return;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const uint32_t i = static_cast<uint32_t>(m * kThreads + tid);
      if (i < nw) sel[i] = wv[m];
    }
    __syncthreads();
    block_bucket_sort_desc(sel, cand, static_cast<int>(nw), bstart, bcur, scratch,
                           [&](int slot, unsigned long long x) { put(a, static_cast<int64_t>(r) * K + slot, x); });
    return;
  }

  // The threshold bin's part: the `need` best candidates after the winners.
  const uint32_t above = min(__ldcg(&rs.win_count), static_cast<uint32_t>(nout));
  const uint32_t nt = __ldcg(&rs.tie_count);
  const uint32_t T = __ldcg(&rs.T);
  const unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
  unsigned long long tv[kTieCap / kThreads];   // the list is read whole, before its length is known
#pragma unroll
  for (int m = 0; m < kTieCap / kThreads; ++m) tv[m] = __ldcg(&tie[m * kThreads + tid]);
  for (int i = tid; i < kSubBins; i += kThreads) hbuf[i] = __ldcg(&ws.hist_sub[static_cast<int64_t>(r) * kSubBins + i]);
  if (tid == 0) count_s = 0;
  const uint32_t need = static_cast<uint32_t>(nout) - above;
  for (int j = nout + tid; j < K; j += kThreads) {
    out[j] = -1;
    if (a.out_score != nullptr) a.out_score[static_cast<int64_t>(r) * K + j] = __uint_as_float(0xFF800000u);
  }
  if (need == 0) return;
  if (nt <= static_cast<uint32_t>(kTieCap)) {
#pragma unroll
    for (int m = 0; m < kTieCap / kThreads; ++m)
      if (static_cast<uint32_t>(m * kThreads + tid) < nt) cand[m * kThreads + tid] = tv[m];
    __syncthreads();
    // Second digit.  The candidates' 1024-bin histogram, summed from the top,
    // gives each bin's first slot among the candidates; S2 is the bin holding
    // the need-th.  Every bin above S2 is taken whole, S2 in part.
    __shared__ uint32_t gmax_s;
    if (tid == 0) {
      gmax_s = 0u;
      scratch[34] = 0u;
      scratch[35] = 0u;
    }
    const int b0 = kSubBins - 1 - 2 * tid, b1 = b0 - 1;   // this thread's two bins, highest first
    const uint32_t c0 = tid < kSubBins / 2 ? hbuf[b0] : 0u;
    const uint32_t c1 = tid < kSubBins / 2 ? hbuf[b1] : 0u;
    uint32_t total;
    const uint32_t e0 = block_excl_scan(c0 + c1, scratch, &total);
    const uint32_t e1 = e0 + c0;
    if (tid < kSubBins / 2) {
      bstart[b0] = e0;
      bstart[b1] = e1;
      bcur[b0] = 0u;
      bcur[b1] = 0u;
      if (e0 < need && need <= e1) {
        scratch[34] = static_cast<uint32_t>(b0);
        scratch[35] = e0;
      } else if (e1 < need && need <= e1 + c1) {
        scratch[34] = static_cast<uint32_t>(b1);
        scratch[35] = e1;
      }
      // the largest group of equal 22-bit prefixes among the keys taken
      const uint32_t g0 = e0 < need ? min(c0, need - e0) : 0u;
      const uint32_t g1 = e1 < need ? min(c1, need - e1) : 0u;
      if (max(g0, g1) > 0u) atomicMax(&gmax_s, max(g0, g1));
    }
    __syncthreads();
    const uint32_t S2 = scratch[34];
    const uint32_t need2 = need - scratch[35];
    const uint32_t cnt2 = hbuf[S2];
    const uint32_t gmax = gmax_s;
    __syncthreads();
    // the rest of S2's bin, by the 42 bits below the second digit (skipped when the whole bin goes)
    unsigned long long th42 = 0ull;
    if (need2 < cnt2)
      th42 = select_threshold(static_cast<int64_t>(nt), need2,
                              [&](int64_t i, bool &valid) {
                                const unsigned long long v = low52(cand[i]);
                                valid = (v >> 42) == S2;
                                return v;
                              },
                              hbuf, scratch, 1);
    // each taken key into its second-digit bin's slots (any order within the bin)
    for (uint32_t i = tid; i < nt; i += kThreads) {
      const unsigned long long c = cand[i];
      const unsigned long long v = low52(c);
      const uint32_t sub = static_cast<uint32_t>(v >> 42);
      if (sub > S2 || (sub == S2 && (v & ((1ull << 42) - 1)) >= th42)) {
        const uint32_t slot = bstart[sub] + atomicAdd(&bcur[sub], 1u);
        if (slot < need) sel[slot] = c;
      }
    }
    __syncthreads();
    if (gmax <= static_cast<uint32_t>(kGroupMax)) {
      // order within each bin by the rank among its members (all 64 bits compared)
      for (uint32_t i = tid; i < need; i += kThreads) {
        const unsigned long long x = sel[i];
        const uint32_t sub = static_cast<uint32_t>(low52(x) >> 42);
        const uint32_t g0 = bstart[sub], g1 = g0 + bcur[sub];
        uint32_t rank = 0u;
        for (uint32_t j = g0; j < g1; ++j) rank += sel[j] > x ? 1u : 0u;
        put(a, static_cast<int64_t>(r) * K + above + g0 + rank, x);
      }
      return;
    }
    if (tid == 0) count_s = need;   // many equal prefixes: sort the taken keys below
  } else {
    // Too many keys in the threshold bin for the list: digits over the row's scores.
    __syncthreads();
    const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
    const unsigned long long th = select_threshold(
        static_cast<int64_t>(B), need,
        [&](int64_t pos, bool &valid) {
          const uint32_t key = radix_key(row[pos]);
          valid = (key >> 20) == T;
          return low52(composite(key, pos));
        },
        hbuf, scratch, 0);
    __syncthreads();
    for (int64_t p0 = tid & ~31; p0 < B; p0 += kThreads) {
      const int64_t pos = p0 + (tid & 31);
      bool take = false;
      unsigned long long c = 0ull;
      if (pos < B) {
        const uint32_t key = radix_key(row[pos]);
        c = composite(key, pos);
        take = (key >> 20) == T && low52(c) >= th;
      }
      warp_push64(take, c, sel, &count_s, static_cast<uint32_t>(kSortCap));
    }
  }
  __syncthreads();
  const int n = min(static_cast<int>(count_s), static_cast<int>(need));
  block_bucket_sort_desc(sel, cand, n, bstart, bcur, scratch, [&](int slot, unsigned long long x) {
    put(a, static_cast<int64_t>(r) * K + above + slot, x);
  });
}

}  // namespace

cudaError_t launch_select_clear(const SelectArgs &a, const int32_t *row_bound, cudaStream_t stream) {
  select_clear_kernel<<<a.R, 256, 0, stream>>>(a, row_bound);
  return cudaGetLastError();
}

cudaError_t launch_hist12(const SelectArgs &a, cudaStream_t stream) {
  const int ns = max(1, (a.max_bound + kSlice - 1) / kSlice);
  hist12_kernel<<<dim3(ns, a.R), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

// Slice length for the collect grid: about four CTAs per SM over all rows,
// a multiple of kSliceStep, at most kSlice.
int collect_slice(const SelectArgs &a) {
  const int64_t keys = static_cast<int64_t>(a.R) * (a.max_bound > 1 ? a.max_bound : 1);
  const int64_t ctas = 4LL * (a.num_sms > 1 ? a.num_sms : 1);
  int64_t s = (keys + ctas - 1) / ctas;
  s = (s + kSliceStep - 1) / kSliceStep * kSliceStep;
  if (s < kSliceStep) s = kSliceStep;
  if (s > kSlice) s = kSlice;
  return static_cast<int>(s);
}

cudaError_t launch_collect(const SelectArgs &a_in, cudaStream_t stream) {
  static std::mutex mu;
  static bool done[128] = {};
  const cudaError_t es = once_per_device(mu, done, [] {
    const cudaError_t e1 =
        cudaFuncSetAttribute(finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFinishSmemAlloc);
    if (e1 != cudaSuccess) return e1;
    return cudaFuncSetAttribute(collect_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCollectSmemAlloc);
  });
  if (es != cudaSuccess) return es;
  SelectArgs a = a_in;
  a.slice = collect_slice(a);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int ns = max(1, (a.max_bound + a.slice - 1) / a.slice);
  cfg.gridDim = dim3(ns, a.R);
  cfg.blockDim = dim3(kCollectThreads);
  cfg.dynamicSmemBytes = kCollectSmemAlloc;
  cudaError_t e = cudaLaunchKernelEx(&cfg, collect_kernel, a);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(2, a.R);   // per row: the winners' CTA and the candidates' CTA
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 2 * a.R > a.num_sms ? kFinishSmem : kFinishSmemAlloc;
  return cudaLaunchKernelEx(&cfg, finish_kernel, a);
}

}  // namespace idx
