// Launch front: the scoring plan and the query operands.
//
// One launch, R + 1 blocks.  Blocks 0..R-1 each prepare one row's query as the B
// operand of the tensor-core contraction and clear that row's selection state;
// block R plans the scoring layout (row groups and their tiles).  This is the
// GB300 counterpart of the sglang PR 48224 page's "scoring layout ahead"
// (section Modifications, commit 3): the row groups, their requests and each
// row's index bound are worked out once, on the device, before the scan.
#include <cuda_fp8.h>

#include "idx_device.cuh"
#include "launch.h"
#include "plan.cuh"

namespace idx {
namespace {

constexpr int kPrepThreads = 1024;

// Byte offset of (row n, byte k) of a 128-byte-row operand block in the 128-byte
// swizzled layout: the 16-byte chunk index is XORed with the row index mod 8.
__device__ __forceinline__ uint32_t swz128(uint32_t n, uint32_t kbyte) {
  return n * 128u + ((((kbyte >> 4) ^ (n & 7u)) & 7u) << 4) + (kbyte & 15u);
}

// Publishes the plan (plan.cuh) for the scoring launch and the selection, clears
// the status word and flags rows with a bad request or bound.
__device__ void plan_block(const PrepArgs &a) {
  const Workspace &ws = a.ws;
  const int64_t bound_cap = min(static_cast<int64_t>(a.pt_stride) * kPage, static_cast<int64_t>(a.max_bound));
  if (threadIdx.x == 0) *ws.status = 0u;
  __syncthreads();
  const PlanResult pr = plan_rows(a.row_req, a.row_bound, a.R, a.Q, bound_cap, ws.groups, ws.bound_eff);
  if (threadIdx.x == 0) {
    if (pr.bad) atomicOr(ws.status, kStatusBadBound);
    ws.plan->num_groups = pr.num_groups;
    ws.plan->total_tiles = pr.total_tiles;
  }
}

// One row's query as the MMA B operand plus its weights.
//  E4M3 cache: per head, q * 2^e (e a power of two putting the head's largest |q|
//  in [128, 256)) is split exactly into hi + lo, both E4M3; the MMA runs both
//  terms against the E4M3 keys, and w * 2^-e undoes the prescale.  The weights
//  are also halved (exactly): the scoring epilogue forms 2 relu(d) as d + |d|.  A bf16 value
//  has 8 significant bits and an E4M3 value 4: hi takes the top 4 (round to
//  nearest) and the remainder, at most 8 units of the bf16 last place, fits the
//  4 bits of lo, so the split is exact wherever lo is not subnormal.
//  bf16 cache: the bf16 query itself, in two 64-dimension K blocks.
__device__ void prep_row(const PrepArgs &a, int r) {
  const Workspace &ws = a.ws;
  const uint16_t *q = reinterpret_cast<const uint16_t *>(a.q) + static_cast<int64_t>(r) * kHeads * kDim;
  uint8_t *op0 = ws.qop0 + static_cast<int64_t>(r) * kRowOperandBytes;
  uint8_t *op1 = ws.qop1 + static_cast<int64_t>(r) * kRowOperandBytes;
  // 1024 threads: 16 per head, 8 dims each.
  const int h = threadIdx.x >> 4;
  const int d0 = (threadIdx.x & 15) * 8;
  float x[8];
  {
    const uint4 raw = *reinterpret_cast<const uint4 *>(q + h * kDim + d0);
    const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(words[i] << 16);
      x[2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
    }
  }
  if (a.kv_dtype == IDX_KV_E4M3) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    int e = 0;
    if (m > 0.f && m <= 3.0e38f) {
      int E;
      frexpf(m, &E);  // m = f * 2^E, f in [0.5, 1)
      e = 8 - E;
      e = max(-120, min(120, e));
    }
    uint8_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xs = ldexpf(x[i], e);
      const __nv_fp8_e4m3 fh(xs);
      const float rem = xs - static_cast<float>(fh);
      const __nv_fp8_e4m3 fl(rem);
      hi[i] = fh.__x;
      lo[i] = fl.__x;
    }
    // dims d0..d0+7 are bytes d0..d0+7 of head row h: half of one 16-byte chunk.
    const uint32_t off = swz128(h, d0);
    uint2 vh, vl;
    vh.x = hi[0] | (hi[1] << 8) | (hi[2] << 16) | (static_cast<uint32_t>(hi[3]) << 24);
    vh.y = hi[4] | (hi[5] << 8) | (hi[6] << 16) | (static_cast<uint32_t>(hi[7]) << 24);
    vl.x = lo[0] | (lo[1] << 8) | (lo[2] << 16) | (static_cast<uint32_t>(lo[3]) << 24);
    vl.y = lo[4] | (lo[5] << 8) | (lo[6] << 16) | (static_cast<uint32_t>(lo[7]) << 24);
    *reinterpret_cast<uint2 *>(op0 + off) = vh;
    *reinterpret_cast<uint2 *>(op1 + off) = vl;
    if ((threadIdx.x & 15) == 0) ws.wq[r * kHeads + h] = ldexpf(a.w[r * kHeads + h], -e - 1);
  } else {
    // dims d0..d0+7 = 16 bytes: one chunk of K block d0 / 64.
    const int kb = d0 >> 6;
    const uint32_t off = swz128(h, (d0 & 63) * 2);
    const uint4 raw = *reinterpret_cast<const uint4 *>(q + h * kDim + d0);
    *reinterpret_cast<uint4 *>((kb == 0 ? op0 : op1) + off) = raw;
    if ((threadIdx.x & 15) == 0) ws.wq[r * kHeads + h] = ldexpf(a.w[r * kHeads + h], -1);
  }
}

__device__ void clear_row_state(const PrepArgs &a, int r) {
  const Workspace &ws = a.ws;
  if (a.hist_target != nullptr && threadIdx.x < 64) a.hist_target[r * 64 + threadIdx.x] = 0u;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
    ws.hist12[static_cast<int64_t>(r) * kHistBins + i] = 0u;
  }
  if (threadIdx.x < 64) ws.hist64[static_cast<int64_t>(r) * 64 + threadIdx.x] = 0u;
  if (a.clear_select)
    for (int i = threadIdx.x; i < kSubBins; i += blockDim.x) ws.hist_sub[static_cast<int64_t>(r) * kSubBins + i] = 0u;
  if (a.clear_select && threadIdx.x < sizeof(RowSelect) / 4)
    reinterpret_cast<uint32_t *>(&ws.rowsel[r])[threadIdx.x] = 0u;
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const PrepArgs a) {
  // The scoring launch may start its CTAs now: they set up shared memory, barriers
  // and TMEM, then wait for this grid to finish before reading anything it writes.
  grid_dependency_trigger();
  if (blockIdx.x == a.R) {
    plan_block(a);
  } else {
    prep_row(a, blockIdx.x);
    clear_row_state(a, blockIdx.x);
  }
}

}  // namespace

cudaError_t launch_prep(const PrepArgs &a, cudaStream_t stream) {
  prep_kernel<<<a.R + 1, kPrepThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace idx
