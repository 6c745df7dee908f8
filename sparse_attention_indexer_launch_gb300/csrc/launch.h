// Host-side launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "idx_device.cuh"

namespace idx {

struct PrepArgs {
  const void *q;
  const float *w;
  const int32_t *row_req;
  const int32_t *row_bound;
  int32_t R, Q, pt_stride, max_bound, kv_dtype;
  uint32_t *hist_target;   // first-digit histogram the scoring kernel will fill (cleared here), or null
  int32_t clear_select;    // also clear the selection state (rowsel)
  Workspace ws;
};

struct ScoreArgs {
  const int32_t *page_table;
  const float *k_scale;
  int64_t P;
  int32_t pt_stride;
  float *scores;
  int64_t ld;
  uint32_t *hist;          // [R][64] first-digit histogram target, or null
  Workspace ws;
  uint64_t wait_limit_ns;
  int32_t stall_first_handoff;
};

struct SelectArgs {
  const float *scores;
  int64_t ld;
  const int32_t *bound;    // effective bounds [R]
  int32_t R, K, max_bound;
  int32_t *out_idx;        // [R][K]
  Workspace ws;
  int32_t bulk_rows;       // scores and ld allow 16-byte bulk copies of row slices
  uint64_t wait_limit_ns;
  int32_t num_sms;         // SMs of the device (sizes the collect grid)
  int32_t slice;           // keys per collect CTA (set by launch_collect)
};

cudaError_t launch_prep(const PrepArgs &a, cudaStream_t stream);
cudaError_t launch_score(const CUtensorMap &kmap, const ScoreArgs &a, int kv_dtype, int num_ctas,
                         cudaStream_t stream);
// Selection.  idx_topk: clear the state and copy the bounds, build the 12-bit
// histogram of the given scores.  Both paths end in the collect and finish launches.
cudaError_t launch_select_clear(const SelectArgs &a, const int32_t *row_bound, cudaStream_t stream);
cudaError_t launch_hist12(const SelectArgs &a, cudaStream_t stream);
cudaError_t launch_collect(const SelectArgs &a, cudaStream_t stream);

}  // namespace idx
