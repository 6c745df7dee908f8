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
// Data flow (one row; many rows run side by side):
//   hist12   the histogram of the top 12 bits of radix_key (the scoring kernel
//            fuses it; idx_topk on given scores builds it with hist12_kernel,
//            needing only the 64-bin first digit when that is given).
//   collect  (slices of kSlice keys, one CTA each) finds the 12-bit bin T that
//            holds the k-th key, appends every key above T (the winners, fewer
//            than K) and every key in T (the candidates).  The CTA that finishes
//            last for its row (an arrival counter: nothing waits) then
//   finish   picks the K - winners best candidates by a radix select over the
//            remaining 52 composite bits in shared memory, sorts the K keys and
//            writes the positions, -1 past min(K, bound).  A row with more
//            candidates than the buffer holds (thousands of equal scores) is
//            resolved digit by digit over the row's scores instead.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kSlice = 16384;
constexpr int kThreads = 1024;
constexpr int kHistThreads = 512;
constexpr int kSortCap = 2048;            // = IDX_MAX_K, power of two
// dynamic shared memory of the collect/finish kernel
constexpr int kFinishSmem = (kTieCap + kSortCap) * 8;

__device__ __forceinline__ unsigned long long composite(uint32_t key, int64_t pos) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}

__device__ __forceinline__ int nslices(int32_t bound) { return bound > 0 ? (bound + kSlice - 1) / kSlice : 1; }

// Among nbins bins taken in descending bin order, the bin holding the need-th key:
// above < need <= above + hist[bin], above = keys in higher bins.  Block-wide:
// every thread must call it and every thread gets the result.
__device__ void find_bin(const uint32_t *hist, int nbins, uint32_t need, uint32_t *out_bin, uint32_t *out_above,
                         uint32_t *scratch /* >= 34 words of shared memory */) {
  const int per = (nbins + blockDim.x - 1) / blockDim.x;
  const int tid = threadIdx.x;
  if (tid == 0) {
    scratch[32] = 0u;
    scratch[33] = 0u;
  }
  uint32_t sum = 0;
  for (int m = 0; m < per; ++m) {
    const int i = tid * per + m;
    if (i < nbins) sum += hist[nbins - 1 - i];
  }
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t incl = sum;
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
  const uint32_t excl = incl - sum + (warp > 0 ? scratch[warp - 1] : 0u);
  __syncthreads();
  if (excl < need && need <= excl + sum) {
    uint32_t above = excl;
    for (int m = 0; m < per; ++m) {
      const int i = tid * per + m;
      if (i >= nbins) break;
      const uint32_t c = hist[nbins - 1 - i];
      if (above + c >= need) {
        scratch[32] = static_cast<uint32_t>(nbins - 1 - i);
        scratch[33] = above;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
  *out_bin = scratch[32];
  *out_above = scratch[33];
  __syncthreads();
}

// ---------------------------------------------------------------------------- idx_topk front
__global__ void select_clear_kernel(const SelectArgs a, const int32_t *row_bound) {
  const int r = blockIdx.x;
  const Workspace &ws = a.ws;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) ws.hist12[static_cast<int64_t>(r) * kHistBins + i] = 0u;
  if (threadIdx.x < sizeof(RowSelect) / 4) reinterpret_cast<uint32_t *>(&ws.rowsel[r])[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    const int32_t b = row_bound[r];
    const int32_t be = max(0, min(b, a.max_bound));
    if (be != b) flag_status(ws.status, kStatusBadBound);
    ws.bound_eff[r] = be;
  }
}

// The 12-bit histogram of given scores.  With a first-digit histogram `coarse`,
// only the keys of the first digit that holds the k-th key are counted finely;
// every other digit's count goes to that digit's lowest 12-bit bin, which keeps
// every count "above" a bin exact for the threshold search.
__global__ void __launch_bounds__(kHistThreads) hist12_kernel(const SelectArgs a, const uint32_t *coarse) {
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t scratch[34];
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (B <= a.K || static_cast<int>(blockIdx.x) >= nslices(B)) return;   // rows that keep all keys skip it
  const Workspace &ws = a.ws;
  for (int i = threadIdx.x; i < kHistBins; i += kHistThreads) h[i] = 0u;
  uint32_t d1 = 0xFFFFFFFFu;
  if (coarse != nullptr) {
    __syncthreads();
    uint32_t bin, above;
    find_bin(coarse + r * 64, 64, static_cast<uint32_t>(a.K), &bin, &above, scratch);
    d1 = bin;
    if (blockIdx.x == 0 && threadIdx.x < 64 && threadIdx.x != d1 && coarse[r * 64 + threadIdx.x])
      atomicAdd(&ws.hist12[static_cast<int64_t>(r) * kHistBins + threadIdx.x * 64], coarse[r * 64 + threadIdx.x]);
  }
  __syncthreads();
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int64_t end = min(static_cast<int64_t>(B), begin + kSlice);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
  for (int64_t pos = begin + threadIdx.x; pos < end; pos += kHistThreads) {
    const uint32_t key = radix_key(row[pos]);
    if (d1 == 0xFFFFFFFFu || (key >> 26) == d1) atomicAdd(&h[key >> 20], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += kHistThreads)
    if (h[i]) atomicAdd(&ws.hist12[static_cast<int64_t>(r) * kHistBins + i], h[i]);
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

// Bitonic sort, descending, of n (a power of two) keys in shared memory.
// Stages whose pairs stay inside one warp's 64-key block need only __syncwarp.
__device__ void bitonic_sort_desc(unsigned long long *s, int n) {
  const int half = n >> 1;
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
      const int next = stride > 1 ? (stride >> 1) : (size << 1) >> 1;
      if (stride >= 64 || next >= 64 || half > static_cast<int>(blockDim.x)) __syncthreads();
      else __syncwarp();
    }
  }
  __syncthreads();
}

// Digits of the low 52 composite bits, most significant first: six of 8 bits, one of 4.
__device__ __forceinline__ int digit_shift(int d) { return d < 6 ? 44 - 8 * d : 0; }
__device__ __forceinline__ int digit_width(int d) { return d < 6 ? 8 : 4; }

// Low 52 bits of a candidate's composite (the 12 high bits are the shared bin).
__device__ __forceinline__ unsigned long long low52(unsigned long long c) { return c & ((1ull << 52) - 1); }

// Picks the `need` largest of n candidates (composites sharing their top 12 bits)
// by 8-bit digits of the low 52 bits; returns the smallest low-52 value taken.
__device__ unsigned long long select_candidates(const unsigned long long *cand, int n, uint32_t need,
                                                uint32_t *h /* 256 */, uint32_t *scratch) {
  unsigned long long pre = 0ull;
  for (int d = 0; d < 7; ++d) {
    const int sh = digit_shift(d), wd = digit_width(d);
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const unsigned long long v = low52(cand[i]);
      if (d > 0 && (v >> (sh + wd)) != (pre >> (sh + wd))) continue;
      atomicAdd(&h[(v >> sh) & ((1u << wd) - 1u)], 1u);
    }
    __syncthreads();
    uint32_t bin, above;
    find_bin(h, 1 << wd, need, &bin, &above, scratch);
    need -= above;
    pre |= static_cast<unsigned long long>(bin) << sh;
  }
  return pre;
}

__device__ void finish_row(const SelectArgs &a, int r, unsigned long long *sm, uint32_t *h, uint32_t *scratch,
                           uint32_t T12) {
  const Workspace &ws = a.ws;
  const int32_t B = a.bound[r];
  const int K = a.K;
  const int nout = min(K, B);
  unsigned long long *cand = sm;                 // kTieCap
  unsigned long long *fin = sm + kTieCap;        // kSortCap
  __shared__ uint32_t count_s;
  const uint32_t nw = min(__ldcg(&ws.rowsel[r].win_count), static_cast<uint32_t>(kSortCap));
  const uint32_t nt = B > K ? __ldcg(&ws.rowsel[r].tie_count) : 0u;
  const unsigned long long *win = ws.win + static_cast<int64_t>(r) * K;
  const unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
  for (uint32_t i = threadIdx.x; i < nw; i += blockDim.x) fin[i] = __ldcg(&win[i]);
  if (threadIdx.x == 0) count_s = nw;
  __syncthreads();
  if (B > K) {
    const uint32_t need = static_cast<uint32_t>(K) - nw;
    if (nt <= static_cast<uint32_t>(kTieCap)) {
      for (uint32_t i = threadIdx.x; i < nt; i += blockDim.x) cand[i] = __ldcg(&tie[i]);
      __syncthreads();
      const unsigned long long th = select_candidates(cand, static_cast<int>(nt), need, h, scratch);
      for (uint32_t i = threadIdx.x; i < nt; i += blockDim.x) {
        if (low52(cand[i]) >= th) {
          const uint32_t at = atomicAdd(&count_s, 1u);
          if (at < static_cast<uint32_t>(kSortCap)) fin[at] = cand[i];
        }
      }
    } else {
      // Too many keys in the threshold bin: the same digits, over the row's scores.
      const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
      unsigned long long pre = 0ull;
      uint32_t nd = need;
      for (int d = 0; d < 7; ++d) {
        const int sh = digit_shift(d), wd = digit_width(d);
        for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0u;
        __syncthreads();
        for (int64_t pos = threadIdx.x; pos < B; pos += blockDim.x) {
          const uint32_t key = radix_key(row[pos]);
          if ((key >> 20) != T12) continue;
          const unsigned long long v = low52(composite(key, pos));
          if (d > 0 && (v >> (sh + wd)) != (pre >> (sh + wd))) continue;
          atomicAdd(&h[(v >> sh) & ((1u << wd) - 1u)], 1u);
        }
        __syncthreads();
        uint32_t bin, above;
        find_bin(h, 1 << wd, nd, &bin, &above, scratch);
        nd -= above;
        pre |= static_cast<unsigned long long>(bin) << sh;
      }
      for (int64_t pos = threadIdx.x; pos < B; pos += blockDim.x) {
        const uint32_t key = radix_key(row[pos]);
        if ((key >> 20) != T12) continue;
        const unsigned long long c = composite(key, pos);
        if (low52(c) >= pre) {
          const uint32_t at = atomicAdd(&count_s, 1u);
          if (at < static_cast<uint32_t>(kSortCap)) fin[at] = c;
        }
      }
    }
  }
  __syncthreads();
  const int n = min(static_cast<int>(count_s), kSortCap);
  int p2 = 1;
  while (p2 < n) p2 <<= 1;
  for (int i = n + threadIdx.x; i < p2; i += blockDim.x) fin[i] = 0ull;
  __syncthreads();
  bitonic_sort_desc(fin, p2);
  int32_t *out = a.out_idx + static_cast<int64_t>(r) * K;
  for (int j = threadIdx.x; j < K; j += blockDim.x)
    out[j] = (j < nout && j < n) ? static_cast<int32_t>(~static_cast<uint32_t>(fin[j] & 0xFFFFFFFFull)) : -1;
}

__global__ void __launch_bounds__(kThreads) collect_kernel(const SelectArgs a) {
  extern __shared__ unsigned long long sm[];
  __shared__ uint32_t h[256];
  __shared__ uint32_t hist_s[kHistBins];
  __shared__ uint32_t scratch[34];
  __shared__ int is_last;
  grid_dependency_wait();   // scores and the histogram come from the previous launch
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (static_cast<int>(blockIdx.x) >= nslices(B)) return;
  const Workspace &ws = a.ws;
  const bool take_all = B <= a.K;
  uint32_t T12 = 0;
  if (!take_all) {
    for (int i = threadIdx.x; i < kHistBins; i += kThreads)
      hist_s[i] = __ldcg(&ws.hist12[static_cast<int64_t>(r) * kHistBins + i]);
    __syncthreads();
    uint32_t above;
    find_bin(hist_s, kHistBins, static_cast<uint32_t>(a.K), &T12, &above, scratch);
  }
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int64_t end = min(static_cast<int64_t>(B), begin + kSlice);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
  unsigned long long *win = ws.win + static_cast<int64_t>(r) * a.K;
  unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
  for (int64_t base = begin; base < end; base += kThreads) {
    const int64_t pos = base + threadIdx.x;
    const bool in = pos < end;
    const uint32_t key = in ? radix_key(row[pos]) : 0u;
    const uint32_t bin = key >> 20;
    const bool w = in && (take_all || bin > T12);
    const bool t = in && !take_all && bin == T12;
    const unsigned long long c = composite(key, pos);
    warp_append(w, c, win, &ws.rowsel[r].win_count, static_cast<uint32_t>(a.K));
    warp_append(t, c, tie, &ws.rowsel[r].tie_count, static_cast<uint32_t>(kTieCap));
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0)
    is_last = atomicAdd(&ws.rowsel[r].nslices_done, 1u) == static_cast<uint32_t>(nslices(B) - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  finish_row(a, r, sm, h, scratch, T12);
}

}  // namespace

cudaError_t launch_select_clear(const SelectArgs &a, const int32_t *row_bound, cudaStream_t stream) {
  select_clear_kernel<<<a.R, 256, 0, stream>>>(a, row_bound);
  return cudaGetLastError();
}

cudaError_t launch_hist12(const SelectArgs &a, const uint32_t *coarse, cudaStream_t stream) {
  const int ns = max(1, (a.max_bound + kSlice - 1) / kSlice);
  hist12_kernel<<<dim3(ns, a.R), kHistThreads, 0, stream>>>(a, coarse);
  return cudaGetLastError();
}

cudaError_t launch_collect(const SelectArgs &a, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(collect_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFinishSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int ns = max(1, (a.max_bound + kSlice - 1) / kSlice);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ns, a.R);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kFinishSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, collect_kernel, a);
}

}  // namespace idx
