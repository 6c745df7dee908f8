// Exact top-K selection by radix digits.
//
// sglang PR 48224 page (sgl-amd-mono #86): each row's "exact top-2048" (section
// Motivation, first paragraph) is chosen by radix selection over slices of at
// most 8,192 keys whose first digit is radix_key >> 26 in 64 bins (section
// Motivation, fourth bullet; section Modifications, commit 4, where that
// histogram comes from the scoring stage instead of a pass of its own).  The
// later digits, the counts and the placement are the selection's own.
//
// Order of keys: by the 64-bit composite (radix_key(score) << 32) | ~position,
// larger first, i.e. score descending and, among equal scores, position
// ascending; the top K composites are exactly the wanted set, so ties at the
// k-th value go to the lowest positions.
//
// Kernels, each over (slice, row) unless noted:
//   first_hist   only when no histogram is given: 64-bin first-digit histogram;
//   hist2        the 64-bin histogram fixes the first digit d1 holding the k-th
//                key; this pass counts the next 12 bits of the keys in bin d1;
//                the slice that arrives last for its row finds the 18-bit prefix
//                holding the k-th key (no waiting: an arrival counter);
//   collect      appends every key above that prefix (winners, < K of them) and
//                every key on it (threshold candidates);
//   finish (row) sorts winners and candidates and writes the first min(K, bound)
//                positions, -1 after.  When a row has more candidates than the
//                candidate buffer holds (many equal scores), it resolves the
//                remaining 46 composite bits digit by digit over the row itself.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kSlice = 8192;
constexpr int kSelThreads = 256;
constexpr int kFinishThreads = 512;
constexpr int kFinishCap = 8192;   // >= IDX_MAX_K + kTieCap, power of two

__device__ __forceinline__ unsigned long long composite(uint32_t key, int64_t pos) {
  return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}

__device__ __forceinline__ int nslices(int32_t bound) { return (bound + kSlice - 1) / kSlice; }

// Among nbins bins in descending bin order, the bin holding the need-th key:
// above < need <= above + hist[bin], above = keys in higher bins.  Block-wide;
// every thread returns the result.  nbins = 64 uses one warp's worth of work,
// but all threads must call it.
__device__ void find_bin(const uint32_t *hist, int nbins, uint32_t need, uint32_t *out_bin, uint32_t *out_above,
                         uint32_t *scratch /* >= 34 words */) {
  const int per = (nbins + blockDim.x - 1) / blockDim.x;
  const int tid = threadIdx.x;
  uint32_t sum = 0;
  for (int m = 0; m < per; ++m) {
    const int i = tid * per + m;
    if (i < nbins) sum += hist[nbins - 1 - i];
  }
  // exclusive scan of sum over the block
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

// ---------------------------------------------------------------------------- state
__global__ void select_clear_kernel(const SelectArgs a, const int32_t *row_bound, uint32_t *hist1) {
  const int r = blockIdx.x;
  const Workspace &ws = a.ws;
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) ws.hist2[static_cast<int64_t>(r) * 4096 + i] = 0u;
  if (threadIdx.x < sizeof(RowSelect) / 4) reinterpret_cast<uint32_t *>(&ws.rowsel[r])[threadIdx.x] = 0u;
  if (hist1 != nullptr && threadIdx.x < 64) hist1[r * 64 + threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    const int32_t b = row_bound[r];
    const int32_t be = max(0, min(b, a.max_bound));
    if (be != b) flag_status(ws.status, kStatusBadBound);
    ws.bound_eff[r] = be;
  }
}

__global__ void __launch_bounds__(kSelThreads) first_hist_kernel(const SelectArgs a, uint32_t *hist1) {
  __shared__ uint32_t h[64];
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (static_cast<int>(blockIdx.x) >= nslices(B)) return;
  if (threadIdx.x < 64) h[threadIdx.x] = 0u;
  __syncthreads();
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int64_t end = min(static_cast<int64_t>(B), begin + kSlice);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
  for (int64_t base = begin; base < end; base += kSelThreads) {
    const int64_t pos = base + threadIdx.x;
    const uint32_t d = pos < end ? (radix_key(row[pos]) >> 26) : 64u;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    if (d < 64u && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[d], __popc(peers));
  }
  __syncthreads();
  if (threadIdx.x < 64 && h[threadIdx.x]) atomicAdd(&hist1[r * 64 + threadIdx.x], h[threadIdx.x]);
}

// ---------------------------------------------------------------------------- second digit
__global__ void __launch_bounds__(kSelThreads) hist2_kernel(const SelectArgs a) {
  __shared__ uint32_t h[4096];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t d1_s, above1_s;
  __shared__ int is_last;
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (B <= a.K) return;  // the row keeps all its keys
  const int ns = nslices(B);
  if (static_cast<int>(blockIdx.x) >= ns) return;
  const Workspace &ws = a.ws;
  for (int i = threadIdx.x; i < 4096; i += kSelThreads) h[i] = 0u;
  if (threadIdx.x < 64) scratch[threadIdx.x & 31] = 0u;
  __syncthreads();
  {
    uint32_t d1, above1;
    find_bin(a.hist1 + r * 64, 64, static_cast<uint32_t>(a.K), &d1, &above1, scratch);
    if (threadIdx.x == 0) {
      d1_s = d1;
      above1_s = above1;
    }
  }
  __syncthreads();
  const uint32_t d1 = d1_s;
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int64_t end = min(static_cast<int64_t>(B), begin + kSlice);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
#pragma unroll 4
  for (int64_t pos = begin + threadIdx.x; pos < end; pos += kSelThreads) {
    const uint32_t key = radix_key(row[pos]);
    if ((key >> 26) == d1) atomicAdd(&h[(key >> 14) & 4095u], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 4096; i += kSelThreads)
    if (h[i]) atomicAdd(&ws.hist2[static_cast<int64_t>(r) * 4096 + i], h[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(&ws.rowsel[r].nslices_done, 1u) == static_cast<uint32_t>(ns - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < 4096; i += kSelThreads) h[i] = __ldcg(&ws.hist2[static_cast<int64_t>(r) * 4096 + i]);
  __syncthreads();
  uint32_t d2, above2;
  find_bin(h, 4096, static_cast<uint32_t>(a.K) - above1_s, &d2, &above2, scratch);
  if (threadIdx.x == 0) {
    ws.rowsel[r].prefix = (d1 << 12) | d2;
    ws.rowsel[r].above = above1_s + above2;
    ws.rowsel[r].mode = 1u;
  }
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

__global__ void __launch_bounds__(kSelThreads) collect_kernel(const SelectArgs a) {
  const int r = blockIdx.y;
  const int32_t B = a.bound[r];
  if (static_cast<int>(blockIdx.x) >= nslices(B)) return;
  const Workspace &ws = a.ws;
  const bool take_all = B <= a.K;
  const uint32_t prefix = take_all ? 0u : ws.rowsel[r].prefix;
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * kSlice;
  const int64_t end = min(static_cast<int64_t>(B), begin + kSlice);
  const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
  unsigned long long *win = ws.win + static_cast<int64_t>(r) * a.K;
  unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
  for (int64_t base = begin; base < end; base += kSelThreads) {
    const int64_t pos = base + threadIdx.x;
    const bool in = pos < end;
    const uint32_t key = in ? radix_key(row[pos]) : 0u;
    const uint32_t p18 = key >> 14;
    const bool w = in && (take_all || p18 > prefix);
    const bool t = in && !take_all && p18 == prefix;
    const unsigned long long c = composite(key, pos);
    warp_append(w, c, win, &ws.rowsel[r].win_count, static_cast<uint32_t>(a.K));
    warp_append(t, c, tie, &ws.rowsel[r].tie_count, static_cast<uint32_t>(kTieCap));
  }
}

// ---------------------------------------------------------------------------- finish
__device__ void bitonic_sort_desc(unsigned long long *s, int n /* power of two */) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (n >> 1); i += blockDim.x) {
        const int lo = 2 * stride * (i / stride) + (i % stride);
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = s[lo], y = s[hi];
        if ((x < y) == desc) {
          s[lo] = y;
          s[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Remaining composite bits below the 18-bit prefix: 14 score bits, 32 position bits.
__device__ __forceinline__ unsigned long long low46(uint32_t key, int64_t pos) {
  return (static_cast<unsigned long long>(key & 0x3FFFu) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}

__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const SelectArgs a) {
  extern __shared__ unsigned long long sk[];   // kFinishCap entries
  __shared__ uint32_t h[256];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t count_s;
  const int r = blockIdx.x;
  const Workspace &ws = a.ws;
  const int32_t B = a.bound[r];
  const int K = a.K;
  const int nout = min(K, B);
  int32_t *out = a.out_idx + static_cast<int64_t>(r) * K;
  const uint32_t nw = min(ws.rowsel[r].win_count, static_cast<uint32_t>(K));
  const uint32_t nt_all = B > K ? ws.rowsel[r].tie_count : 0u;
  const unsigned long long *win = ws.win + static_cast<int64_t>(r) * K;
  const unsigned long long *tie = ws.tie + static_cast<int64_t>(r) * kTieCap;
  uint32_t n = nw;
  for (uint32_t i = threadIdx.x; i < nw; i += kFinishThreads) sk[i] = win[i];
  if (nt_all <= static_cast<uint32_t>(kTieCap)) {
    for (uint32_t i = threadIdx.x; i < nt_all; i += kFinishThreads) sk[nw + i] = tie[i];
    n = nw + nt_all;
  } else {
    // Many keys on the 18-bit prefix: find the exact composite threshold among them.
    const uint32_t prefix = ws.rowsel[r].prefix;
    uint32_t need = static_cast<uint32_t>(nout) - nw;
    unsigned long long pre = 0ull;
    const float *row = a.scores + static_cast<int64_t>(r) * a.ld;
    const int shifts[6] = {38, 30, 22, 14, 6, 0};
    const int widths[6] = {8, 8, 8, 8, 8, 6};
    for (int d = 0; d < 6; ++d) {
      const int sh = shifts[d], wd = widths[d];
      for (int i = threadIdx.x; i < 256; i += kFinishThreads) h[i] = 0u;
      __syncthreads();
      for (int64_t pos = threadIdx.x; pos < B; pos += kFinishThreads) {
        const uint32_t key = radix_key(row[pos]);
        if ((key >> 14) != prefix) continue;
        const unsigned long long v = low46(key, pos);
        if (d > 0 && (v >> (sh + wd)) != (pre >> (sh + wd))) continue;
        atomicAdd(&h[(v >> sh) & ((1u << wd) - 1u)], 1u);
      }
      __syncthreads();
      uint32_t bin, above;
      find_bin(h, 1 << wd, need, &bin, &above, scratch);
      need -= above;
      pre |= static_cast<unsigned long long>(bin) << sh;
    }
    // pre is now the composite (low 46 bits) of the last key taken from the prefix bin.
    if (threadIdx.x == 0) count_s = nw;
    __syncthreads();
    for (int64_t pos = threadIdx.x; pos < B; pos += kFinishThreads) {
      const uint32_t key = radix_key(row[pos]);
      if ((key >> 14) != prefix) continue;
      if (low46(key, pos) >= pre) {
        const uint32_t idx = atomicAdd(&count_s, 1u);
        if (idx < static_cast<uint32_t>(kFinishCap)) sk[idx] = composite(key, pos);
      }
    }
    __syncthreads();
    n = min(count_s, static_cast<uint32_t>(kFinishCap));
  }
  __syncthreads();
  int p2 = 1;
  while (p2 < static_cast<int>(n)) p2 <<= 1;
  for (int i = static_cast<int>(n) + threadIdx.x; i < p2; i += kFinishThreads) sk[i] = 0ull;
  __syncthreads();
  bitonic_sort_desc(sk, p2);
  for (int j = threadIdx.x; j < K; j += kFinishThreads)
    out[j] = (j < nout && j < static_cast<int>(n)) ? static_cast<int32_t>(~static_cast<uint32_t>(sk[j] & 0xFFFFFFFFull)) : -1;
}

}  // namespace

cudaError_t launch_select_clear(const SelectArgs &a, const int32_t *row_bound, uint32_t *hist1_to_clear,
                                cudaStream_t stream) {
  select_clear_kernel<<<a.R, 256, 0, stream>>>(a, row_bound, hist1_to_clear);
  return cudaGetLastError();
}

cudaError_t launch_first_hist(const SelectArgs &a, uint32_t *hist1, cudaStream_t stream) {
  const int ns = max(1, (a.max_bound + kSlice - 1) / kSlice);
  first_hist_kernel<<<dim3(ns, a.R), kSelThreads, 0, stream>>>(a, hist1);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectArgs &a, cudaStream_t stream) {
  static bool configured = false;
  const int ns = max(1, (a.max_bound + kSlice - 1) / kSlice);
  hist2_kernel<<<dim3(ns, a.R), kSelThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  collect_kernel<<<dim3(ns, a.R), kSelThreads, 0, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int smem = kFinishCap * static_cast<int>(sizeof(unsigned long long));
  if (!configured) {
    e = cudaFuncSetAttribute(finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  finish_kernel<<<a.R, kFinishThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace idx
