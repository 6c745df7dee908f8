// Device-side building blocks shared by the indexer kernels (sm_103a only):
// mbarrier waits with a time limit, TMA and bulk copies, tcgen05 (UMMA)
// descriptors and instructions, the radix key, and the workspace layout.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "idx.h"

namespace idx {

constexpr int kHeads = IDX_HEADS;
constexpr int kDim = IDX_DIM;
constexpr int kPage = IDX_PAGE;
constexpr int kTileKeys = 128;            // keys per MMA tile (M), two pages
constexpr int kMaxGroupRows = 4;          // rows sharing one key read (N = 64 * rows <= 256)
constexpr int kRowOperandBytes = 8192;    // one row's 64 heads x 128 bytes, one K block

// Device status word bits (first word of every workspace).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBadPage = 2u;
constexpr uint32_t kStatusBadBound = 4u;

// ---------------------------------------------------------------------------- workspace
// Every call carves the caller's workspace the same way (offsets in bytes, each
// 1024-aligned).  The layout is computed on the host (api.cu) and handed to the
// kernels in this struct.
struct Group {
  int32_t req;         // request whose keys the group reads
  int32_t row0;        // first row; the group's rows are row0 .. row0 + nrows - 1
  int32_t nrows;       // 1 .. 4
  int32_t L;           // keys read: the largest bound of the group's rows
  int32_t tile_begin;  // first tile of the group in the launch's tile order
  int32_t pad[3];
};

struct PlanHeader {
  int32_t num_groups;
  int32_t total_tiles;
  int32_t pad[30];
};

struct RowSelect {       // per-row selection state
  uint32_t tie_count;    // keys in the threshold bin, appended by the collect kernel
  uint32_t T;            // 12-bit bin holding the k-th key (0xFFFFFFFF: the row keeps all keys)
  uint32_t win_count;    // keys in higher bins (the winners), appended by the collect kernel
  uint32_t pad[5];
};

// The fused score histogram counts the top kHistBits bits of radix_key(score):
// its 64-bin marginal (top 6 bits) is the first digit radix_key >> 26.
constexpr int kHistBits = 12;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kSubBins = 1024;   // second digit of the threshold bin's keys (the next 10 bits)

struct Workspace {
  uint32_t *status;        // [1]
  PlanHeader *plan;        // [1]
  Group *groups;           // [R]
  int32_t *bound_eff;      // [R]       row bounds after the device-side range check
  uint8_t *qop0;           // [R][8192]  FP8: q_hi; bf16: dims 0..63   (MMA B operand, swizzled)
  uint8_t *qop1;           // [R][8192]  FP8: q_lo; bf16: dims 64..127
  float *wq;               // [R][64]    weights / 2 with the query prescale folded in
  uint32_t *hist12;        // [R][4096]  12-bit histogram of the radix keys
  uint32_t *hist64;        // [R][64]    its 64-bin marginal (the first digit radix_key >> 26)
  uint32_t *hist_sub;      // [R][1024]  second-digit histogram of the threshold bin
  RowSelect *rowsel;       // [R]
  unsigned long long *win; // [R][K]     keys above the threshold bin, in arrival order (composite keys)
  unsigned long long *tie; // [R][kTieCap] keys in the threshold bin
  float *scores;           // [R][ld]    score scratch of idx_launch (else unused)
  int64_t scores_ld;
};

// Threshold-bin keys kept per row for the finish: several times what the threshold
// bin of any benchmark workload holds (at most 2,430, in the bf16 batch); a row
// with more is resolved from its scores instead.
constexpr int kTieCap = 6144;

// ---------------------------------------------------------------------------- timing
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag_status(uint32_t *status, uint32_t bits) {
  atomicOr(status, bits);
}

// ---------------------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware up to `hint_ns` while the
// phase is incomplete, instead of spinning on the issue slots other warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// `limit_ns` nanoseconds, or once *abort is set by another role of the CTA;
// returns false then (the caller records the timeout and unwinds).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                          volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------- copies
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// 2-D tiled TMA load into shared memory, completing on `bar` by byte count.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, int32_t x, int32_t y,
                                            uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk reduction shared -> global: dst[i] += src[i] for `bytes` / 4 u32 words,
// element by element atomically, by the TMA engine (16-byte aligned addresses,
// size a multiple of 16).  One bulk group per call; the generic-proxy writes of
// src must be made visible to the async proxy first (fence_proxy_async_shared).
__device__ __forceinline__ void bulk_reduce_add_u32(uint32_t *gdst, const uint32_t *ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.u32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: wait until the grid this launch depends on has
// completed and its memory is visible (a no-op when launched without the attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the dependent grid be scheduled once every CTA of this grid has called it.
__device__ __forceinline__ void grid_dependency_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor for a K-major operand in the 128-byte swizzled
// canonical layout: rows of 128 bytes, groups of 8 rows 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);        // start address
  d |= static_cast<uint64_t>(1u) << 16;                           // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                   // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                           // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                           // 128-byte swizzle
  return d;
}

// Instruction descriptor: D fp32, A and B K-major, M = 128, N = n.
// a_b_format: kind::f8f6f4 -> 0 = E4M3; kind::f16 -> 1 = BF16.
__device__ __forceinline__ uint32_t umma_idesc(uint32_t a_b_format, uint32_t n) {
  return (1u << 4) | (a_b_format << 7) | (a_b_format << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void umma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrive on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 16 lanes x 256 bits (eight 32-bit columns), four repetitions along the columns.
// Thread i of the warp receives, for repetition k (columns col + 8k .. col + 8k + 7):
//   r[4k + 0], r[4k + 1]: lane (lane field + i / 4),     columns 8k + 2 (i % 4) + {0, 1};
//   r[4k + 2], r[4k + 3]: lane (lane field + i / 4 + 8), the same columns.
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Ties the registers to a point after tcgen05.wait::ld so that no use of them is
// scheduled before the wait.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------- radix key
// Order-preserving unsigned key of an fp32 score; -0.0 is read as +0.0.
__device__ __forceinline__ uint32_t radix_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float whose radix_key is k (inverse of radix_key; the key of -0.0 and +0.0
// gives +0.0).
__device__ __forceinline__ float radix_key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

}  // namespace idx
