// The scoring plan: row groups and their tiles, computed by one whole block.
//
// sglang PR 48224 page (sgl-amd-mono #86), section Reviewer notes, "The join
// rule": row r joins row r-1's group when both belong to the same request and
// bound[r] == bound[r-1] + 1; a group holds at most four rows (section
// Modifications, commit 1: the rows of one request read and convert each key once
// for all of them).  Every other row starts a new group.  A group reads the keys
// below the largest effective bound of its rows, in tiles of kTileKeys keys, and
// the tiles of all groups are numbered in group order (section Modifications,
// commit 3: the scoring layout is worked out once, ahead of the scan).
//
// The prep launch runs this to publish the plan; the scoring launch runs it again
// in each CTA (for up to kLocalPlanRows rows) from the same inputs, so that its
// key loads need not wait for the prep launch.  Both get identical plans.
#pragma once

#include "idx_device.cuh"

namespace idx {

constexpr int kLocalPlanRows = 512;   // rows a scoring CTA plans for itself

// Inclusive block-wide scan (sum, or max when is_max) for any block of whole warps.
template <typename T>
__device__ T plan_block_scan(T v, T *tmp, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = is_max ? (n > v ? n : v) : v + n;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    T x = lane < static_cast<int>(blockDim.x >> 5) ? tmp[lane] : (is_max ? T(-2147483647 - 1) : T(0));
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

// A row's bound after the range check: rows of an unknown request read nothing,
// others are clamped to [0, bound_cap].
__device__ __forceinline__ int32_t plan_effective_bound(int32_t req, int32_t braw, int32_t Q, int64_t bound_cap) {
  if (req < 0 || req >= Q) return 0;
  return static_cast<int32_t>(max(int64_t{0}, min(static_cast<int64_t>(braw), bound_cap)));
}

struct PlanResult {
  int32_t num_groups;
  int32_t total_tiles;
  bool bad;   // some row had an unknown request or a bound outside [0, bound_cap]
};

// Writes the group records to groups[0 .. num_groups) (shared or global memory)
// and, when bound_eff is given, every row's effective bound.  Called by every
// thread of the block; returns the same result to all of them.
__device__ inline PlanResult plan_rows(const int32_t *row_req, const int32_t *row_bound, int R, int Q,
                                       int64_t bound_cap, Group *groups, int32_t *bound_eff) {
  __shared__ int32_t tmp[32];
  __shared__ int32_t carry_run, carry_group, carry_tiles;
  const int nt = static_cast<int>(blockDim.x);
  if (threadIdx.x == 0) {
    carry_run = 0;
    carry_group = 0;
    carry_tiles = 0;
  }
  __syncthreads();
  bool bad = false;
  // Pass 1: group starts and group records (req, row0).
  for (int base = 0; base < R; base += nt) {
    const int r = base + threadIdx.x;
    bool join = false;
    int32_t rs = -1;
    if (r < R) {
      const int32_t req = row_req[r];
      const int32_t braw = row_bound[r];
      const bool ok = req >= 0 && req < Q && braw >= 0 && braw <= bound_cap;
      if (!ok) bad = true;
      if (bound_eff != nullptr) bound_eff[r] = plan_effective_bound(req, braw, Q, bound_cap);
      if (ok && r > 0) {
        const int32_t reqp = row_req[r - 1];
        const int32_t bp = row_bound[r - 1];
        join = reqp == req && bp >= 0 && braw == bp + 1;
      }
      if (!join) rs = r;
    }
    // run start: the last non-joining row at or before r
    rs = plan_block_scan<int32_t>(rs, tmp, true);
    if (rs < 0) rs = carry_run;
    const bool gstart = (r < R) && (!join || ((r - rs) % kMaxGroupRows) == 0);
    const int32_t gi = plan_block_scan<int32_t>(gstart ? 1 : 0, tmp, false) + carry_group - 1;
    if (gstart) {
      const int32_t req = row_req[r];
      Group g;
      g.req = (req >= 0 && req < Q) ? req : -1;
      g.row0 = r;
      g.nrows = 0;
      g.L = 0;
      g.tile_begin = 0;
      g.pad[0] = g.pad[1] = g.pad[2] = 0;
      groups[gi] = g;
    }
    __syncthreads();
    if (threadIdx.x == nt - 1) {
      carry_run = rs;
      carry_group = gi + 1;
    }
    __syncthreads();
  }
  const int G = carry_group;
  __syncthreads();
  // Pass 2: rows per group, keys read (largest effective bound), tiles and their prefix.
  for (int base = 0; base < G; base += nt) {
    const int g = base + threadIdx.x;
    int32_t tiles = 0;
    if (g < G) {
      const int32_t r0 = groups[g].row0;
      const int32_t r1 = (g + 1 < G) ? groups[g + 1].row0 : R;
      int32_t L = 0;
      for (int r = r0; r < r1; ++r) L = max(L, plan_effective_bound(row_req[r], row_bound[r], Q, bound_cap));
      if (groups[g].req < 0) L = 0;
      groups[g].nrows = r1 - r0;
      groups[g].L = L;
      tiles = (L + kTileKeys - 1) / kTileKeys;
    }
    const int32_t incl = plan_block_scan<int32_t>(tiles, tmp, false);
    if (g < G) groups[g].tile_begin = carry_tiles + incl - tiles;
    __syncthreads();
    if (threadIdx.x == nt - 1) carry_tiles += incl;
    __syncthreads();
  }
  PlanResult res;
  res.bad = __syncthreads_or(bad) != 0;
  res.num_groups = G;
  res.total_tiles = carry_tiles;
  __syncthreads();   // the carries may be reused by a later call
  return res;
}

}  // namespace idx
