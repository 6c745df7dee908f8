// A decode row's new key written into the paged cache: used by the standalone
// patch launch (patch.cu) and by the fused launch's prep kernel (prep.cu).
//
// sglang PR 48224 page, section Reviewer notes ("New keys"): a key the launch
// writes is scored for every row of its request in the launch.  Row r's key goes
// to its position, row_bound[r] - 1, through the page table.  E4M3 cache: the
// per-token scale amax / 448 (1 for a zero key); each value divided by it in fp32
// goes to the nearest E4M3 code, saturating at +-448.  bf16 cache: the values as
// given.
#pragma once

#include <cuda_fp8.h>

#include "idx_device.cuh"
#include "launch.h"

namespace idx {

// One warp writes row r's new key (lane l: dims 4l .. 4l+3).  Rows with bound 0,
// a request or bound out of range, or a page id outside [0, P) write nothing
// (the scan reports a bad page itself).
__device__ inline void store_new_key(const PatchArgs &a, int r, int lane) {
  const int32_t b = a.row_bound[r];
  const int32_t req = a.row_req[r];
  if (b <= 0 || req < 0 || req >= a.Q || static_cast<int64_t>(b) > static_cast<int64_t>(a.pt_stride) * kPage) return;
  const int64_t t = b - 1;
  const int32_t page = a.page_table[static_cast<int64_t>(req) * a.pt_stride + t / kPage];
  if (page < 0 || static_cast<int64_t>(page) >= a.P) return;
  const int64_t token = static_cast<int64_t>(page) * kPage + t % kPage;
  const uint2 raw = reinterpret_cast<const uint2 *>(a.k_new + static_cast<int64_t>(r) * kDim)[lane];
  if (a.kv_dtype == IDX_KV_BF16) {
    reinterpret_cast<uint2 *>(static_cast<uint16_t *>(a.k_cache) + token * kDim)[lane] = raw;
    return;
  }
  float x[4];
  x[0] = __uint_as_float(raw.x << 16);
  x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  x[2] = __uint_as_float(raw.y << 16);
  x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint32_t packed = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    packed |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x[i], sc), __NV_SATFINITE, __NV_E4M3)) << (8 * i);
  reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(a.k_cache) + token * kDim)[lane] = packed;
  if (lane == 0) a.k_scale[token] = sc;
}

}  // namespace idx
