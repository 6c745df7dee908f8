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
//   collect  one CTA per slice of kSlice keys of a row: each key above T is
//            written straight into its bin's slots (a per-bin cursor orders keys
//            within the bin arbitrarily); each key in T is appended to the row's
//            candidate list.
//   finish   kParts CTAs per row sort the winners' bin-aligned segments in place
//            (bins are contiguous ranges of slots, so segments sort
//            independently); one more CTA per row picks the K - prefix(T) best
//            candidates by radix digits of their remaining 52 bits, sorts them
//            into the slots after the winners and writes -1 past min(K, bound).
//            A row with more candidates than the list holds (thousands of equal
//            scores) is resolved digit by digit over the row's scores instead.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kSlice = 8192;
constexpr int kThreads = 512;
constexpr int kPer = kSlice / kThreads;
constexpr int kParts = 4;                 // winner segments per row
constexpr int kSortCap = IDX_MAX_K;       // power of two
constexpr int kFinishSmem = kTieCap * 8;  // candidates (the sort buffer reuses the front)
constexpr uint32_t kNoBin = 0xFFFFFFFFu;

__device__ __forceinline__ unsigned long long composite(uint32_t key, int64_t pos) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
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

// The row's 12-bit bin layout: off[b] = keys in bins above b (into shared
// memory), the threshold bin T (kNoBin when the row keeps all its keys) and the
// number of keys above T.  Block-wide.
__device__ void row_layout(const uint32_t *hist_g, int32_t B, int K, uint32_t *off, uint32_t *scratch,
                           uint32_t *T, uint32_t *above) {
  constexpr int per = kHistBins / kThreads;
  uint32_t c[per];
  uint32_t sum = 0;
#pragma unroll
  for (int m = 0; m < per; ++m) {          // this thread's bins, highest first
    c[m] = __ldcg(&hist_g[kHistBins - 1 - (threadIdx.x * per + m)]);
    sum += c[m];
  }
  uint32_t total;
  uint32_t run = block_excl_scan(sum, scratch, &total);
  if (threadIdx.x == 0) {
    scratch[34] = kNoBin;
    scratch[35] = static_cast<uint32_t>(max(B, 0));
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < per; ++m) {
    const int b = kHistBins - 1 - (threadIdx.x * per + m);
    off[b] = run;
    if (B > K && run < static_cast<uint32_t>(K) && static_cast<uint32_t>(K) <= run + c[m]) {
      scratch[34] = static_cast<uint32_t>(b);
      scratch[35] = run;
    }
    run += c[m];
  }
  __syncthreads();
  *T = scratch[34];
  *above = scratch[35];
  __syncthreads();
}

// ---------------------------------------------------------------------------- idx_topk front
__global__ void select_clear_kernel(const SelectArgs a, const int32_t *row_bound) {
  const int r = blockIdx.x;
  const Workspace &ws = a.ws;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
    ws.hist12[static_cast<int64_t>(r) * kHistBins + i] = 0u;
    ws.cursor[static_cast<int64_t>(r) * kHistBins + i] = 0u;
  }
  if (threadIdx.x < sizeof(RowSelect) / 4) reinterpret_cast<uint32_t *>(&ws.rowsel[r])[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    const int32_t b = row_bound[r];
    const int32_t be = max(0, min(b, a.max_bound));
    if (be != b) flag_status(ws.status, kStatusBadBound);
    ws.bound_eff[r] = be;
  }
}

// The 12-bit histogram of given scores (one slice of a row per CTA).
__global__ void __launch_bounds__(kThreads) hist12_kernel(const SelectArgs a) {
  __shared__ uint32_t h[kHistBins];
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (static_cast<int>(blockIdx.x) >= nslices(B)) return;
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) h[i] = 0u;
  __syncthreads();
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int64_t end = min(static_cast<int64_t>(B), begin + kSlice);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
  for (int64_t pos = begin + threadIdx.x; pos < end; pos += kThreads) atomicAdd(&h[radix_key(row[pos]) >> 20], 1u);
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += kThreads)
    if (h[i]) atomicAdd(&a.ws.hist12[static_cast<int64_t>(r) * kHistBins + i], h[i]);
}

// ---------------------------------------------------------------------------- collect
__device__ __forceinline__ void warp_append(bool take, unsigned long long value, unsigned long long *dst,
                                            uint32_t *counter, uint32_t cap) {
  const uint32_t ballot = __ballot_sync(0xffffffffu, take);
  if (ballot == 0u) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(ballot) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(ballot)));
  base = __shfl_sync(0xffffffffu, base, leader);
  const uint32_t idx = base + __popc(ballot & ((1u << lane) - 1u));
  if (take && idx < cap) dst[idx] = value;
}

__global__ void __launch_bounds__(kThreads) collect_kernel(const SelectArgs a) {
  __shared__ uint32_t off[kHistBins];
  __shared__ uint32_t scratch[36];
  grid_dependency_wait();   // scores and the histogram come from the previous launch
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (static_cast<int>(blockIdx.x) >= nslices(B)) return;
  const Workspace &ws = a.ws;
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int64_t end = min(static_cast<int64_t>(B), begin + kSlice);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
  float sv[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {   // this thread's loads in flight while the layout is worked out
    const int64_t pos = begin + i * kThreads + threadIdx.x;
    sv[i] = pos < end ? __ldcg(row + pos) : 0.f;
  }
  uint32_t T, above;
  row_layout(ws.hist12 + static_cast<int64_t>(r) * kHistBins, B, a.K, off, scratch, &T, &above);
  unsigned long long *win = ws.win + static_cast<int64_t>(r) * a.K;
  unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
  uint32_t *cursor = ws.cursor + static_cast<int64_t>(r) * kHistBins;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int64_t pos = begin + i * kThreads + threadIdx.x;
    const bool in = pos < end;
    const uint32_t key = radix_key(sv[i]);
    const uint32_t bin = key >> 20;
    const unsigned long long c = composite(key, pos);
    if (in && (T == kNoBin || bin > T)) {
      const uint32_t slot = off[bin] + atomicAdd(&cursor[bin], 1u);
      if (slot < static_cast<uint32_t>(a.K)) win[slot] = c;
    }
    warp_append(in && T != kNoBin && bin == T, c, tie, &ws.rowsel[r].tie_count, static_cast<uint32_t>(kTieCap));
  }
}

// ---------------------------------------------------------------------------- finish
// Bitonic sort, descending, of n (a power of two) keys in shared memory.  When
// every pair of a stage lies in the 64-key block of the warp that handles it
// (strides below 32, one pair per thread) the stage needs only __syncwarp.
__device__ void bitonic_sort_desc(unsigned long long *s, int n) {
  const int half = n >> 1;
  const bool one_pair = half <= static_cast<int>(blockDim.x);
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int lg = __ffs(stride) - 1;
      for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const int lo = ((i >> lg) << (lg + 1)) | (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = s[lo], y = s[hi];
        if ((x < y) == desc) {
          s[lo] = y;
          s[hi] = x;
        }
      }
      const int next = stride > 1 ? (stride >> 1) : size;
      if (!one_pair || stride >= 32 || next >= 32) __syncthreads();
      else __syncwarp();
    }
  }
  __syncthreads();
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int p = 1;
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

// Threshold on the low 52 bits such that exactly `need` keys of the threshold
// bin are >= it.  `candidate(i, valid)` yields the i-th key (valid = false to skip).
template <typename Get>
__device__ unsigned long long select_threshold(int64_t n, uint32_t need, Get candidate, uint32_t *h /* 2048 */,
                                               uint32_t *scratch) {
  unsigned long long pre = 0ull;
  for (int d = 0; d < 5; ++d) {
    const int sh = digit_shift(d), wd = digit_width(d);
    const int nb = 1 << wd;
    for (int i = threadIdx.x; i < nb; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      bool valid;
      const unsigned long long v = low52(candidate(i, valid));
      if (!valid || (d > 0 && (v >> (sh + wd)) != (pre >> (sh + wd)))) continue;
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

__global__ void __launch_bounds__(kThreads) finish_kernel(const SelectArgs a) {
  extern __shared__ unsigned long long sm[];
  __shared__ uint32_t off[kHistBins];
  __shared__ uint32_t scratch[36];
  __shared__ uint32_t bounds_s[2];
  __shared__ uint32_t count_s;
  grid_dependency_wait();   // every collect slice has placed its keys
  const int part = blockIdx.x;
  const int r = blockIdx.y;
  const Workspace &ws = a.ws;
  const int32_t B = a.bound[r];
  const int K = a.K;
  const int nout = min(K, max(B, 0));
  uint32_t T, above;
  row_layout(ws.hist12 + static_cast<int64_t>(r) * kHistBins, B, K, off, scratch, &T, &above);
  above = min(above, static_cast<uint32_t>(nout));
  int32_t *out = a.out_idx + static_cast<int64_t>(r) * K;
  unsigned long long *s = sm;

  if (part < kParts) {
    // This part's winner segment: from the first bin starting at or after
    // part * S to the first bin starting at or after (part + 1) * S.
    const uint32_t S = (above + kParts - 1) / kParts;
    const uint32_t lo_cut = part * S, hi_cut = (part + 1) * S;
    if (threadIdx.x == 0) {
      bounds_s[0] = above;
      bounds_s[1] = above;
    }
    __syncthreads();
    for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) {
      if (T != kNoBin && static_cast<uint32_t>(b) <= T) continue;
      const uint32_t o = off[b];
      if (o >= above) continue;
      if (o >= lo_cut) atomicMin(&bounds_s[0], o);
      if (o >= hi_cut) atomicMin(&bounds_s[1], o);
    }
    __syncthreads();
    const uint32_t s0 = bounds_s[0], s1 = max(bounds_s[0], bounds_s[1]);
    const int n = static_cast<int>(s1 - s0);
    if (n == 0) return;
    const unsigned long long *win = ws.win + static_cast<int64_t>(r) * K;
    const int p2 = pow2_at_least(n);
    for (int i = threadIdx.x; i < p2; i += blockDim.x) s[i] = i < n ? __ldcg(&win[s0 + i]) : 0ull;
    __syncthreads();
    bitonic_sort_desc(s, p2);
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      out[s0 + i] = static_cast<int32_t>(~static_cast<uint32_t>(s[i] & 0xFFFFFFFFull));
    return;
  }

  // The threshold bin's part: the `need` best candidates after the winners.
  const uint32_t need = static_cast<uint32_t>(nout) - above;
  for (int j = nout + threadIdx.x; j < K; j += blockDim.x) out[j] = -1;
  if (need == 0) return;
  const uint32_t nt = __ldcg(&ws.rowsel[r].tie_count);
  unsigned long long *cand = sm;
  if (threadIdx.x == 0) count_s = 0;
  unsigned long long th;
  if (nt <= static_cast<uint32_t>(kTieCap)) {
    const unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
    for (uint32_t i = threadIdx.x; i < nt; i += blockDim.x) cand[i] = __ldcg(&tie[i]);
    __syncthreads();
    th = select_threshold(static_cast<int64_t>(nt), need,
                          [&](int64_t i, bool &valid) { valid = true; return cand[i]; }, off, scratch);
    // keep the chosen ones at the front (the threshold pass is done with cand)
    __syncthreads();
    unsigned long long mine[kTieCap / kThreads];
    int nm = 0;
    for (uint32_t i = threadIdx.x; i < nt; i += blockDim.x)
      if (low52(cand[i]) >= th) mine[nm++] = cand[i];
    __syncthreads();
    for (int m = 0; m < nm; ++m) cand[atomicAdd(&count_s, 1u)] = mine[m];
  } else {
    // Too many keys in the threshold bin for the list: the same digits, over the row.
    const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
    th = select_threshold(static_cast<int64_t>(B), need,
                          [&](int64_t pos, bool &valid) {
                            const uint32_t key = radix_key(row[pos]);
                            valid = (key >> 20) == T;
                            return composite(key, pos);
                          },
                          off, scratch);
    __syncthreads();
    for (int64_t pos = threadIdx.x; pos < B; pos += blockDim.x) {
      const uint32_t key = radix_key(row[pos]);
      if ((key >> 20) != T) continue;
      const unsigned long long c = composite(key, pos);
      if (low52(c) >= th) {
        const uint32_t at = atomicAdd(&count_s, 1u);
        if (at < static_cast<uint32_t>(kSortCap)) cand[at] = c;
      }
    }
  }
  __syncthreads();
  const int n = min(static_cast<int>(count_s), static_cast<int>(need));
  const int p2 = pow2_at_least(n);
  for (int i = n + threadIdx.x; i < p2; i += blockDim.x) cand[i] = 0ull;
  __syncthreads();
  bitonic_sort_desc(cand, p2);
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    out[above + i] = static_cast<int32_t>(~static_cast<uint32_t>(cand[i] & 0xFFFFFFFFull));
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

cudaError_t launch_collect(const SelectArgs &a, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFinishSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int ns = max(1, (a.max_bound + kSlice - 1) / kSlice);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ns, a.R);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, collect_kernel, a);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t fcfg = {};
  fcfg.gridDim = dim3(kParts + 1, a.R);
  fcfg.blockDim = dim3(kThreads);
  fcfg.dynamicSmemBytes = kFinishSmem;
  fcfg.stream = stream;
  fcfg.attrs = attr;
  fcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&fcfg, finish_kernel, a);
}

}  // namespace idx
