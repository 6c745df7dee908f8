// Exact top-K of the union of ranked parts: the merge of a key-sharded indexer.
//
// "Release Test Suite - GLM-5.2-EXL3" page, section Config change: decode
// context parallelism shards a request's KV cache over GPUs and merges the
// indexer's top-k at an owner GPU, by an exchange the page calls exact.  Each shard selects its own top-K of the keys it holds, with their
// scores; the global top-K is a subset of the union of the shards' lists (a key
// that is not in its own shard's top-K has K keys above it), so merging the
// lists by the same order gives the unsharded selection exactly.
//
// Order: the 64-bit composite (radix_key(score) << 32) | ~position, larger
// first: score descending, then position ascending, as idx_launch orders its
// output.  Every part must come in that order (as idx_launch_scored writes it),
// -1 padded.  The grid has one CTA per (part, row).  Each loads all S lists of
// its row into shared memory as composites (padding as 0, below every real key)
// and places the keys of its own part: a key's slot in the merged list is its
// index in its own list plus, for every other list, the number of keys above it
// there (a binary search; among equal keys, which only the padding has, lower
// parts go first).  Keys whose slot reaches K are dropped, and the CTA of part 0
// writes the padding past the lists' total length.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kMergeThreads = 1024;

__device__ __forceinline__ unsigned long long merge_key(float score, int64_t pos) {
  return (static_cast<unsigned long long>(radix_key(score)) << 32) |
         static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}

// Number of keys of the descending list b[0, n) that are > x (strict) or >= x.
__device__ __forceinline__ int count_above(const unsigned long long *b, int n, unsigned long long x, bool strict) {
  int lo = 0, hi = n;   // answer in [lo, hi]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const bool above = strict ? (b[mid] > x) : (b[mid] >= x);
    if (above) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  extern __shared__ unsigned long long msm[];   // [S][Kin]
  __shared__ int nvalid[kMergeMaxParts];
  const int own = blockIdx.x, r = blockIdx.y;
  const int S = a.S, Kin = a.Kin, K = a.K;
  const int tid = threadIdx.x;
  if (tid < S) nvalid[tid] = Kin;
  __syncthreads();
  // a list's entries are its ranked keys, then the padding: its length is the
  // index of its first -1
  // every load of the thread goes out before any is used (one memory round trip)
  constexpr int kPer = kMergeMaxParts * IDX_MAX_K / kMergeThreads;
  int32_t pv[kPer];
  float sv[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = tid + k * kMergeThreads;
    pv[k] = -1;
    sv[k] = 0.0f;
    if (i < S * Kin) {
      const int s = i / Kin, j = i - s * Kin;
      const int64_t at = (static_cast<int64_t>(s) * a.R + r) * Kin + j;
      pv[k] = __ldg(&a.part_idx[at]);
      sv[k] = __ldg(&a.part_score[at]);
    }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = tid + k * kMergeThreads;
    if (i < S * Kin) {
      const int s = i / Kin, j = i - s * Kin;
      msm[i] = pv[k] < 0 ? 0ull : merge_key(sv[k], static_cast<int64_t>(pv[k]) + a.offset[s]);
      if (pv[k] < 0) atomicMin(&nvalid[s], j);
    }
  }
  __syncthreads();
  const unsigned long long *mine = msm + static_cast<int64_t>(own) * Kin;
  for (int j = tid; j < nvalid[own] && j < K; j += kMergeThreads) {
    const unsigned long long x = mine[j];
    int rank = j;
    for (int t = 0; t < S && rank < K; ++t) {
      if (t == own) continue;
      rank += count_above(msm + static_cast<int64_t>(t) * Kin, nvalid[t], x, t > own);
    }
    if (rank < K) {
      const int64_t at = static_cast<int64_t>(r) * K + rank;
      a.out_idx[at] = static_cast<int32_t>(~static_cast<uint32_t>(x & 0xFFFFFFFFull));
      if (a.out_score != nullptr) a.out_score[at] = radix_key_value(static_cast<uint32_t>(x >> 32));
    }
  }
  if (own == 0) {
    int total = 0;
    for (int s = 0; s < S; ++s) total += nvalid[s];
    for (int j = min(total, K) + tid; j < K; j += kMergeThreads) {
      const int64_t at = static_cast<int64_t>(r) * K + j;
      a.out_idx[at] = -1;
      if (a.out_score != nullptr) a.out_score[at] = __uint_as_float(0xFF800000u);
    }
  }
}

}  // namespace

size_t merge_smem_bytes(int S, int Kin, int /*K*/) {
  return static_cast<size_t>(S) * Kin * sizeof(unsigned long long);
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t stream) {
  static std::mutex mu;
  static bool done[128] = {};
  const cudaError_t e = once_per_device(mu, done, [] {
    return cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(merge_smem_bytes(kMergeMaxParts, IDX_MAX_K, IDX_MAX_K)));
  });
  if (e != cudaSuccess) return e;
  merge_kernel<<<dim3(a.S, a.R), kMergeThreads, merge_smem_bytes(a.S, a.Kin, a.K), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace idx
