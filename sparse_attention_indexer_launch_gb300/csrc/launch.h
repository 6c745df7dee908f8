// Host-side launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "idx_device.cuh"

namespace idx {

// Runs setup() once per device (the current one) and remembers that it succeeded;
// safe to call from several host threads.  `done` is a caller-owned flag table.
template <typename F>
inline cudaError_t once_per_device(std::mutex &mu, bool (&done)[128], F setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev]) return cudaSuccess;
  e = setup();
  if (e == cudaSuccess) done[dev] = true;
  else (void)cudaGetLastError();   // a failed setup must not be reported again by a later launch
  return e;
}

struct PatchArgs {
  const uint16_t *k_new;   // bf16 [R][128]
  const int32_t *row_req, *row_bound, *page_table;
  void *k_cache;           // E4M3 bytes or bf16 [P][64][128]
  float *k_scale;          // [P][64] for E4M3
  int32_t R, Q, pt_stride, kv_dtype;
  int64_t P;
};

struct PrepArgs {
  const void *q;
  const float *w;
  const int32_t *row_req;
  const int32_t *row_bound;
  int32_t R, Q, pt_stride, max_bound, kv_dtype;
  uint32_t *hist_target;   // first-digit histogram the scoring kernel will fill (cleared here), or null
  int32_t clear_select;    // also clear the selection state (rowsel)
  Workspace ws;
  PatchArgs patch;         // rows' new keys written into the cache first (patch.k_new null: none)
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
  float *out_score;        // [R][K] scores of the selected positions (-inf past them), or null
  Workspace ws;
  int32_t bulk_rows;       // scores and ld allow 16-byte bulk copies of row slices
  uint64_t wait_limit_ns;
  int32_t num_sms;         // SMs of the device (sizes the collect grid)
  int32_t slice;           // keys per collect CTA (set by launch_collect)
};

struct Top1State {          // per row, zero between calls
  unsigned long long key;  // running maximum of (radix_key(value) << 32) | ~index
  uint32_t arrived;        // splits of the row that have folded in their maximum
  uint32_t pad;
};

struct Top1Args {
  const float *logits;
  int64_t ld, V;
  int32_t R;
  int32_t *out_idx;
  float *out_val;          // or null
  int32_t *tokens;         // or null: tokens[r * tokens_ld + token_col]
  int64_t tokens_ld;
  int32_t token_col;
  int32_t *positions;      // or null: positions[r] += 1
  Top1State *state;        // [R]
  int64_t chunk;           // values per split (set by launch_top1)
  int32_t vec4;            // rows and chunks allow 16-byte loads
};


constexpr int kMergeMaxParts = 8;
struct MergeArgs {
  const int32_t *part_idx;   // [S][R][Kin] positions within each part, descending order, -1 padded
  const float *part_score;   // [S][R][Kin] their scores
  int32_t offset[kMergeMaxParts];   // added to part s's positions
  int32_t S, R, Kin, K;
  int32_t *out_idx;          // [R][K]
  float *out_score;          // [R][K] or null
};

cudaError_t launch_prep(const PrepArgs &a, cudaStream_t stream);
cudaError_t launch_score(const CUtensorMap &kmap, const ScoreArgs &a, int kv_dtype, bool batched, int num_ctas,
                         cudaStream_t stream);
// Selection.  idx_topk: clear the state and copy the bounds, build the 12-bit
// histogram of the given scores.  Both paths end in the collect and finish launches.
cudaError_t launch_select_clear(const SelectArgs &a, const int32_t *row_bound, cudaStream_t stream);
cudaError_t launch_hist12(const SelectArgs &a, cudaStream_t stream);
cudaError_t launch_collect(const SelectArgs &a, cudaStream_t stream);
// Every row's new key into the paged cache at position bound - 1.
cudaError_t launch_patch(const PatchArgs &a, cudaStream_t stream);
// Exact top-K of the union of S ranked parts (the key-sharded selection's merge).
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t stream);
size_t merge_smem_bytes(int S, int Kin, int K);
// Top-1 of each row of logits (one launch: splits and last-arriver finalize).
cudaError_t launch_top1(const Top1Args &a, int num_sms, cudaStream_t stream);

}  // namespace idx
