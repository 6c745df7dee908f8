// Launch front: the scoring plan and the query operands.
//
// One launch, R + 1 blocks.  Blocks 0..R-1 each prepare one row's query as the B
// operand of the tensor-core contraction and clear that row's selection state;
// block R plans the scoring layout (row groups and their tiles).  This is the
// GB300 counterpart of the sglang PR 48224 page's scoring layout computed in
// advance (section Modifications, commit 3): the row groups, their requests and each
// row's index bound are worked out once, on the device, before the scan.
#include <cuda_fp8.h>

#include "idx_device.cuh"
#include "launch.h"
#include "new_key.cuh"

namespace idx {
namespace {

constexpr int kPrepThreads = 1024;

// Byte offset of (row n, byte k) of a 128-byte-row operand block in the 128-byte
// swizzled layout: the 16-byte chunk index is XORed with the row index mod 8.
__device__ __forceinline__ uint32_t swz128(uint32_t n, uint32_t kbyte) {
  return n * 128u + ((((kbyte >> 4) ^ (n & 7u)) & 7u) << 4) + (kbyte & 15u);
}

template <typename T>
__device__ T block_scan_incl(T v, T *tmp, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = is_max ? (n > v ? n : v) : v + n;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    T x = lane < (int)(blockDim.x >> 5) ? tmp[lane] : (is_max ? T(-2147483647 - 1) : T(0));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x = is_max ? (n > x ? n : x) : x + n;
    }
    tmp[lane] = x;
  }
  __syncthreads();
  if (warp > 0) {
    T p = tmp[warp - 1];
    v = is_max ? (p > v ? p : v) : v + p;
  }
  __syncthreads();
  return v;
}

// Row groups by the join rule of the sglang PR 48224 page (section Reviewer
// notes, "The join rule"): row r joins row r-1's group when both belong to the
// same request and bound[r] == bound[r-1] + 1, and a group holds at most four
// rows (section Modifications, commit 1: rows of one request read and convert
// each key once for all of them).  Every other row starts a new group.
__device__ void plan_block(const PrepArgs &a) {
  __shared__ int32_t tmp[32];
  __shared__ int32_t carry_run, carry_group, carry_tiles;
  // With at most one block of rows the whole plan stays in shared memory until it
  // is written out once: each group's first row and request, each row's bound.
  __shared__ int32_t s_row0[kPrepThreads], s_req[kPrepThreads], s_eff[kPrepThreads];
  const bool one_pass = a.R <= kPrepThreads;
  const int R = a.R;
  const Workspace &ws = a.ws;
  const int64_t bound_cap = min(static_cast<int64_t>(a.pt_stride) * kPage, static_cast<int64_t>(a.max_bound));
  if (threadIdx.x == 0) {
    carry_run = 0;
    carry_group = 0;
    carry_tiles = 0;
    *ws.status = 0u;
  }
  __syncthreads();
  bool bad = false;
  // Pass 1: effective bounds, group starts, group records (req, row0).
  for (int base = 0; base < R; base += kPrepThreads) {
    const int r = base + threadIdx.x;
    bool join = false, gstart = false;
    int32_t rs = -1;
    if (r < R) {
      const int32_t req = a.row_req[r];
      const int32_t braw = a.row_bound[r];
      const bool ok = req >= 0 && req < a.Q && braw >= 0 && braw <= bound_cap;
      if (!ok) bad = true;
      const int32_t eff =
          (req >= 0 && req < a.Q) ? static_cast<int32_t>(max(int64_t{0}, min(static_cast<int64_t>(braw), bound_cap))) : 0;
      ws.bound_eff[r] = eff;
      if (one_pass) s_eff[r] = eff;
      if (ok && r > 0) {
        const int32_t reqp = a.row_req[r - 1];
        const int32_t bp = a.row_bound[r - 1];
        join = reqp == req && bp >= 0 && braw == bp + 1;
      }
      if (!join) rs = r;
    }
    // run start: the last non-joining row at or before r
    rs = block_scan_incl<int32_t>(rs, tmp, true);
    if (rs < 0) rs = carry_run;
    gstart = (r < R) && (!join || ((r - rs) % kMaxGroupRows) == 0);
    int32_t gi = block_scan_incl<int32_t>(gstart ? 1 : 0, tmp, false) + carry_group - 1;
    if (gstart) {
      const int32_t req = a.row_req[r];
      if (one_pass) {
        s_row0[gi] = r;
        s_req[gi] = (req >= 0 && req < a.Q) ? req : -1;
      } else {
        Group g;
        g.req = (req >= 0 && req < a.Q) ? req : -1;
        g.row0 = r;
        g.nrows = 0;
        g.L = 0;
        g.tile_begin = 0;
        g.pad[0] = g.pad[1] = g.pad[2] = 0;
        ws.groups[gi] = g;
      }
    }
    __syncthreads();
    if (threadIdx.x == kPrepThreads - 1) {
      carry_run = rs;
      carry_group = gi + 1;
    }
    __syncthreads();
  }
  const int G = carry_group;
  __syncthreads();
  // Pass 2: rows per group, keys read (largest bound), tiles and their prefix.
  if (one_pass) {   // G <= R <= kPrepThreads: one group per thread, from shared memory
    const int g = threadIdx.x;
    int32_t tiles = 0, r0 = 0, r1 = 0, L = 0;
    if (g < G) {
      r0 = s_row0[g];
      r1 = (g + 1 < G) ? s_row0[g + 1] : R;
      for (int r = r0; r < r1; ++r) L = max(L, s_eff[r]);
      if (s_req[g] < 0) L = 0;
      tiles = (L + kTileKeys - 1) / kTileKeys;
    }
    const int32_t incl = block_scan_incl<int32_t>(tiles, tmp, false);
    if (g < G) {
      Group gr;
      gr.req = s_req[g];
      gr.row0 = r0;
      gr.nrows = r1 - r0;
      gr.L = L;
      gr.tile_begin = incl - tiles;
      gr.pad[0] = gr.pad[1] = gr.pad[2] = 0;
      ws.groups[g] = gr;
    }
    if (threadIdx.x == kPrepThreads - 1) carry_tiles = incl;
    __syncthreads();
  }
  for (int base = 0; !one_pass && base < G; base += kPrepThreads) {
    const int g = base + threadIdx.x;
    int32_t tiles = 0;
    if (g < G) {
      const int32_t r0 = ws.groups[g].row0;
      const int32_t r1 = (g + 1 < G) ? ws.groups[g + 1].row0 : R;
      int32_t L = 0;
      for (int r = r0; r < r1; ++r) L = max(L, ws.bound_eff[r]);
      if (ws.groups[g].req < 0) L = 0;
      ws.groups[g].nrows = r1 - r0;
      ws.groups[g].L = L;
      tiles = (L + kTileKeys - 1) / kTileKeys;
    }
    int32_t incl = block_scan_incl<int32_t>(tiles, tmp, false);
    if (g < G) ws.groups[g].tile_begin = carry_tiles + incl - tiles;
    __syncthreads();
    if (threadIdx.x == kPrepThreads - 1) carry_tiles += incl;
    __syncthreads();
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(ws.status, kStatusBadBound);
  if (threadIdx.x == 0) {
    ws.plan->num_groups = G;
    ws.plan->total_tiles = carry_tiles;
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
    // the row's new key first (the fused new-key launch): the scan that follows
    // this launch reads the cache only after the whole grid has finished
    if (a.patch.k_new != nullptr && threadIdx.x < 32) store_new_key(a.patch, blockIdx.x, threadIdx.x);
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
