// New keys as a launch of their own: each decode row's key written into the
// paged cache (new_key.cuh) ahead of a later idx_launch.  idx_launch_new_keys
// does the same inside the fused launch's prep kernel.
#include "new_key.cuh"

namespace idx {
namespace {

constexpr int kPatchWarps = 4;   // rows per CTA, one warp per row

__global__ void __launch_bounds__(kPatchWarps * 32) patch_kernel(const PatchArgs a) {
  const int r = blockIdx.x * kPatchWarps + (threadIdx.x >> 5);
  if (r < a.R) store_new_key(a, r, threadIdx.x & 31);
}

}  // namespace

cudaError_t launch_patch(const PatchArgs &a, cudaStream_t stream) {
  patch_kernel<<<(a.R + kPatchWarps - 1) / kPatchWarps, kPatchWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace idx
