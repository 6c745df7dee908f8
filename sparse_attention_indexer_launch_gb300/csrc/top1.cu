// Top-1 of each row of logits in one launch.
//
// The sglang PR 48224 page, later commit on the draft top-1 postprocess: the
// page's version made two launches per step (a pass over splits of each row,
// then a finalizing one).  Here a single launch covers both.  Each CTA takes a
// split of a row, finds its best (value, position) pair, and merges it into the
// row's running best with one 64-bit atomicMax.  An arrival counter per row
// tells the CTA that merges last; that CTA writes the row's outputs and zeroes
// the row's state for the next call.  Equal values resolve to the smaller
// position, and a NaN logit counts as -1e30, as on the page.
//
// The packed key is (radix_key(value) << 32) | ~position: the order-preserving
// radix key makes a larger value win, and for equal values (with -0.0 equal to
// +0.0) the complemented position is larger for the smaller position.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kTop1Threads = 256;
constexpr int kTop1Unroll = 4;          // 16-byte loads per thread issued together
constexpr int64_t kTop1MinChunk = 2048;  // values per split, at least

__device__ __forceinline__ unsigned long long top1_key(float x, int64_t j) {
  const float v = isnan(x) ? -1e30f : x;
  return (static_cast<unsigned long long>(radix_key(v)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(j));
}

__global__ void __launch_bounds__(kTop1Threads) top1_kernel(const Top1Args a) {
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float *row = a.logits + static_cast<int64_t>(r) * a.ld;
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * a.chunk;
  const int64_t end = min(a.V, begin + a.chunk);
  unsigned long long best = 0ull;
  if (a.vec4 && begin < end) {
    // chunk and row start are multiples of 4 floats: 16-byte loads, then the tail
    const float4 *r4 = reinterpret_cast<const float4 *>(row + begin);
    const int64_t n4 = (end - begin) >> 2;
    for (int64_t i0 = 0; i0 < n4; i0 += kTop1Threads * kTop1Unroll) {
      float4 x[kTop1Unroll];
#pragma unroll
      for (int u = 0; u < kTop1Unroll; ++u) {   // all of this thread's loads in flight at once
        const int64_t i = i0 + u * kTop1Threads + tid;
        if (i < n4) x[u] = __ldcs(&r4[i]);
      }
#pragma unroll
      for (int u = 0; u < kTop1Unroll; ++u) {
        const int64_t i = i0 + u * kTop1Threads + tid;
        if (i >= n4) continue;
        const int64_t j = begin + 4 * i;
        best = max(best, top1_key(x[u].x, j));
        best = max(best, top1_key(x[u].y, j + 1));
        best = max(best, top1_key(x[u].z, j + 2));
        best = max(best, top1_key(x[u].w, j + 3));
      }
    }
    for (int64_t j = begin + 4 * n4 + tid; j < end; j += kTop1Threads) best = max(best, top1_key(__ldcs(&row[j]), j));
  } else {
    for (int64_t j = begin + tid; j < end; j += kTop1Threads) best = max(best, top1_key(__ldcs(&row[j]), j));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  __shared__ unsigned long long wbest[kTop1Threads / 32];
  if (lane == 0) wbest[warp] = best;
  __syncthreads();
  if (tid != 0) return;
#pragma unroll
  for (int w = 1; w < kTop1Threads / 32; ++w) best = max(best, wbest[w]);
  Top1State &st = a.state[r];
  atomicMax(&st.key, best);
  __threadfence();   // this split's maximum is in before its arrival is counted
  if (atomicAdd(&st.arrived, 1u) != static_cast<uint32_t>(gridDim.x) - 1u) return;
  // last split of the row: read and reset the row's state, write the results
  __threadfence();
  const unsigned long long key = atomicExch(&st.key, 0ull);
  atomicExch(&st.arrived, 0u);
  const int32_t j = static_cast<int32_t>(~static_cast<uint32_t>(key & 0xFFFFFFFFull));
  a.out_idx[r] = j;
  if (a.out_val != nullptr) {   // the value back from its radix key (no second read of the row)
    const uint32_t k = static_cast<uint32_t>(key >> 32);
    a.out_val[r] = __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  }
  if (a.tokens != nullptr) a.tokens[static_cast<int64_t>(r) * a.tokens_ld + a.token_col] = j;
  if (a.positions != nullptr) a.positions[r] += 1;
}

}  // namespace

cudaError_t launch_top1(const Top1Args &a, int num_sms, cudaStream_t stream) {
  // splits of at least kTop1MinChunk values, about four CTAs per SM over all rows
  const int64_t sms = num_sms > 1 ? num_sms : 1;
  int64_t per_row = (4 * sms + a.R - 1) / a.R;
  if (per_row < 1) per_row = 1;
  int64_t splits = (a.V + kTop1MinChunk - 1) / kTop1MinChunk;
  if (splits > per_row) splits = per_row;
  if (splits < 1) splits = 1;
  Top1Args b = a;
  b.chunk = (a.V + splits - 1) / splits;
  b.chunk = (b.chunk + 3) / 4 * 4;
  splits = (a.V + b.chunk - 1) / b.chunk;
  b.vec4 = b.vec4 && (b.chunk % 4 == 0);
  top1_kernel<<<dim3(static_cast<unsigned>(splits), a.R), kTop1Threads, 0, stream>>>(b);
  return cudaGetLastError();
}

}  // namespace idx
