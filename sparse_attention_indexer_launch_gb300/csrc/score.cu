// The scoring scan: paged key loads (TMA), the tensor-core contraction
// (tcgen05, accumulator in TMEM), the ReLU-weighted head reduction, the score
// store and the fused first-digit histogram.
//
// sglang PR 48224 page (sgl-amd-mono #86): "scores every cached key of each row"
// (section Motivation, first paragraph); rows of one request read each key once
// (section Modifications, commit 1); the store drops "keys at or past a row's
// bound" (commit 2); each stored score's first radix digit radix_key >> 26 is
// counted in 64 bins per row during the scan, which the selection then uses
// instead of a pass of its own (commit 4, the score_hist mailbox).
//
// GB300 layout of the work.  One persistent CTA per SM walks an even share of
// the launch's tiles; a tile is 128 consecutive key positions (two pages) of one
// row group (up to 4 rows of one request).  For a tile the contraction is
//     D[key][row*64 + head] = <k_key, q_row_head>      (M = 128, N = 64 * rows, K = 128)
// so a TMEM lane holds one key and each epilogue thread reduces its key's 64
// head values per row in registers.
//   warp 0      producer: page ids, TMA of the key pages into an smem ring, and
//               the group's query operand (bulk copy) on group changes;
//   warp 1      MMA issuer (one thread) and TMEM owner;
//   warps 2..9  epilogue, two sets of four; set s handles the tiles whose local
//               index is s mod 2, in TMEM accumulator buffer s.
// E4M3 cache: keys feed tcgen05.mma kind::f8f6f4 straight from the TMA ring; the
// query is split exactly into two E4M3 terms (prep.cu), run as K = 256.
// bf16 cache: keys and query are bf16, kind::f16, K = 128.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kBOperandBytes = 2 * kMaxGroupRows * kRowOperandBytes;  // two K blocks
constexpr int kTmemCols = 512;                                        // two accumulators of 256

template <int KV>
struct Cfg {
  static constexpr int kStageBytes = KV == IDX_KV_E4M3 ? kTileKeys * kDim : kTileKeys * kDim * 2;
  static constexpr int kStages = KV == IDX_KV_E4M3 ? 8 : 4;
  static constexpr int kPageBytes = kStageBytes / 2;
};

struct Barriers {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t bfull;
  uint64_t bfree;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int KV>
constexpr int smem_bytes() {
  return 1024 /* alignment slack */ + kBOperandBytes + Cfg<KV>::kStages * Cfg<KV>::kStageBytes +
         static_cast<int>(sizeof(Barriers)) + kEpiWarps * kMaxGroupRows * 64 * 4;
}

// Walks the groups of a CTA's tile range in order.
struct GroupCursor {
  const Group *groups;
  int num_groups;
  int g;          // current group
  int next_begin; // first tile of the next group
  __device__ void seek(const Group *gs, int ng, int t) {
    groups = gs;
    num_groups = ng;
    int lo = 0, hi = ng - 1;
    while (lo < hi) {  // last group with tile_begin <= t
      const int mid = (lo + hi + 1) >> 1;
      if (gs[mid].tile_begin <= t) lo = mid; else hi = mid - 1;
    }
    g = lo;
    next_begin = (g + 1 < ng) ? gs[g + 1].tile_begin : 0x7fffffff;
  }
  __device__ bool advance(int t) {  // true if the group changed
    bool changed = false;
    while (t >= next_begin) {
      ++g;
      next_begin = (g + 1 < num_groups) ? groups[g + 1].tile_begin : 0x7fffffff;
      changed = true;
    }
    return changed;
  }
};

__device__ __forceinline__ void set_abort(Barriers *bars, uint32_t *status) {
  flag_status(status, kStatusTimeout);
  *reinterpret_cast<volatile int *>(&bars->abort) = 1;
}

template <int KV>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ CUtensorMap kmap,
                                                             const ScoreArgs a) {
  using C = Cfg<KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sB0 = smem;                                   // K block 0 of the group's query operand
  uint8_t *sB1 = smem + kBOperandBytes / 2;              // K block 1
  uint8_t *sA = smem + kBOperandBytes;                   // key ring
  Barriers *bars = reinterpret_cast<Barriers *>(sA + C::kStages * C::kStageBytes);
  uint32_t *shist = reinterpret_cast<uint32_t *>(bars + 1);  // [warp][row][64]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Workspace &ws = a.ws;
  const int total_tiles = ws.plan->total_tiles;
  const int num_groups = ws.plan->num_groups;
  const int64_t t0 = static_cast<int64_t>(total_tiles) * blockIdx.x / gridDim.x;
  const int64_t t1 = static_cast<int64_t>(total_tiles) * (blockIdx.x + 1) / gridDim.x;
  if (t0 >= t1) return;  // uniform for the CTA: nothing allocated yet

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->tfull[s], 1);
      mbar_init(&bars->tempty[s], 4);
    }
    mbar_init(&bars->bfull, 1);
    mbar_init(&bars->bfree, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < kEpiWarps * kMaxGroupRows * 64; i += kThreads) shist[i] = 0u;
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&kmap);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  const uint64_t limit = a.wait_limit_ns;
  volatile int *abort = &bars->abort;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      GroupCursor cur;
      cur.seek(ws.groups, num_groups, static_cast<int>(t0));
      int cur_g = -1, req = 0, L = 0, nswitch = 0;
      int k = 0;
      for (int64_t t = t0; t < t1; ++t, ++k) {
        cur.advance(static_cast<int>(t));
        const Group grp = ws.groups[cur.g];
        if (cur.g != cur_g) {
          if (cur_g >= 0 && !mbar_wait(&bars->bfree, (nswitch - 1) & 1, limit, abort)) {
            set_abort(bars, ws.status);
            break;
          }
          const uint32_t bytes = grp.nrows * kRowOperandBytes;
          mbar_arrive_expect_tx(&bars->bfull, 2 * bytes);
          bulk_load(sB0, ws.qop0 + static_cast<int64_t>(grp.row0) * kRowOperandBytes, bytes, &bars->bfull);
          bulk_load(sB1, ws.qop1 + static_cast<int64_t>(grp.row0) * kRowOperandBytes, bytes, &bars->bfull);
          cur_g = cur.g;
          req = grp.req;
          L = grp.L;
          ++nswitch;
        }
        const int s = k % C::kStages;
        if (!mbar_wait(&bars->empty[s], ((k / C::kStages) & 1) ^ 1, limit, abort)) {
          set_abort(bars, ws.status);
          break;
        }
        const int j = static_cast<int>(t) - grp.tile_begin;
        int32_t pages[2];
        uint32_t bytes = 0;
        for (int h = 0; h < 2; ++h) {
          pages[h] = -1;
          const int64_t first = static_cast<int64_t>(j) * kTileKeys + h * kPage;
          if (first < L) {
            const int32_t p = a.page_table[static_cast<int64_t>(req) * a.pt_stride + first / kPage];
            if (p >= 0 && p < a.P) {
              pages[h] = p;
              bytes += C::kPageBytes;
            } else {
              flag_status(ws.status, kStatusBadPage);
            }
          }
        }
        mbar_arrive_expect_tx(&bars->full[s], bytes);
        uint8_t *dst = sA + s * C::kStageBytes;
        for (int h = 0; h < 2; ++h) {
          if (pages[h] < 0) continue;
          if (KV == IDX_KV_E4M3) {
            tma_load_2d(dst + h * (kPage * kDim), &kmap, 0, pages[h] * kPage, &bars->full[s], policy);
          } else {
            tma_load_2d(dst + h * (kPage * 128), &kmap, 0, pages[h] * kPage, &bars->full[s], policy);
            tma_load_2d(dst + kTileKeys * 128 + h * (kPage * 128), &kmap, 64, pages[h] * kPage, &bars->full[s],
                        policy);
          }
        }
      }
      // Wait for every copy still in flight before the CTA may exit (also after an abort).
      int never = 0;
      const int issued = k;
      for (int s = 0; s < C::kStages && s < issued; ++s) {
        const int last_use = issued - 1 - ((issued - 1 - s) % C::kStages);
        if (!mbar_wait(&bars->full[s], (last_use / C::kStages) & 1, limit, &never))
          flag_status(ws.status, kStatusTimeout);
      }
      if (nswitch > 0 && !mbar_wait(&bars->bfull, (nswitch - 1) & 1, limit, &never))
        flag_status(ws.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      GroupCursor cur;
      cur.seek(ws.groups, num_groups, static_cast<int>(t0));
      int cur_g = -1, nswitch = 0;
      uint32_t idesc = 0;
      const uint32_t fmt = KV == IDX_KV_E4M3 ? 0u : 1u;
      int k = 0;
      for (int64_t t = t0; t < t1; ++t, ++k) {
        cur.advance(static_cast<int>(t));
        if (cur.g != cur_g) {
          if (cur_g >= 0) umma_commit(&bars->bfree);
          if (!mbar_wait(&bars->bfull, nswitch & 1, limit, abort)) {
            set_abort(bars, ws.status);
            break;
          }
          ++nswitch;
          cur_g = cur.g;
          idesc = umma_idesc(fmt, 64u * ws.groups[cur_g].nrows);
        }
        const int s = k % C::kStages;
        const int acc = k & 1;
        if (!mbar_wait(&bars->full[s], (k / C::kStages) & 1, limit, abort) ||
            !mbar_wait(&bars->tempty[acc], ((k >> 1) & 1) ^ 1, limit, abort)) {
          set_abort(bars, ws.status);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        const uint32_t a_base = smem_u32(sA + s * C::kStageBytes);
        const uint32_t b0 = smem_u32(sB0), b1 = smem_u32(sB1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          const uint32_t bbase = (kk < 4 ? b0 : b1) + koff;
          if (KV == IDX_KV_E4M3) {
            umma_f8(d, umma_desc_sw128(a_base + koff), umma_desc_sw128(bbase), idesc, kk > 0);
          } else {
            const uint32_t abase = a_base + (kk < 4 ? 0 : kTileKeys * 128) + koff;
            umma_f16(d, umma_desc_sw128(abase), umma_desc_sw128(bbase), idesc, kk > 0);
          }
        }
        umma_commit(&bars->empty[s]);
        if (!(a.stall_first_handoff && k == 0)) umma_commit(&bars->tfull[acc]);
      }
      // All MMAs issued by this thread complete before TMEM is released.
      umma_commit(&bars->drain);
      int never = 0;
      if (!mbar_wait(&bars->drain, 0, limit, &never)) flag_status(ws.status, kStatusTimeout);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int set = ew >> 2;
    const int quarter = warp & 3;              // TMEM lane quarter this warp may read
    uint32_t *hist = shist + ew * kMaxGroupRows * 64;
    GroupCursor cur;
    cur.seek(ws.groups, num_groups, static_cast<int>(t0));
    int cur_g = -1;
    Group grp;
    grp.nrows = 0;
    int k = 0;
    auto flush = [&]() {
      __syncwarp();
      for (int i = 0; i < grp.nrows; ++i) {
        for (int d = lane; d < 64; d += 32) {
          const uint32_t c = hist[i * 64 + d];
          if (c) {
            atomicAdd(&a.hist[static_cast<int64_t>(grp.row0 + i) * 64 + d], c);
            hist[i * 64 + d] = 0u;
          }
        }
      }
      __syncwarp();
    };
    for (int64_t t = t0; t < t1; ++t, ++k) {
      cur.advance(static_cast<int>(t));
      if (cur.g != cur_g) {
        if (cur_g >= 0) flush();
        cur_g = cur.g;
        grp = ws.groups[cur_g];
      }
      if ((k & 1) != set) continue;
      const int j = static_cast<int>(t) - grp.tile_begin;
      const int64_t pos = static_cast<int64_t>(j) * kTileKeys + quarter * 32 + lane;
      const bool valid = pos < grp.L;
      float scale = 1.0f;
      if (KV == IDX_KV_E4M3 && valid) {
        const int32_t p = a.page_table[static_cast<int64_t>(grp.req) * a.pt_stride + pos / kPage];
        scale = (p >= 0 && p < a.P) ? __ldg(&a.k_scale[static_cast<int64_t>(p) * kPage + (pos % kPage)]) : 0.0f;
      }
      if (!mbar_wait(&bars->tfull[set], (k >> 1) & 1, limit, abort)) {
        set_abort(bars, ws.status);
        break;
      }
      tc_fence_after();
      const bool neg_scale = valid && scale < 0.0f;
      const bool any_neg = __any_sync(0xffffffffu, neg_scale);
      for (int i = 0; i < grp.nrows; ++i) {
        const int row = grp.row0 + i;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + set * 256 + i * 64;
        uint32_t v0[32], v1[32];
        tmem_ld32(taddr, v0);
        tmem_ld32(taddr + 32, v1);
        tmem_wait_ld();
        reg_fence(v0);
        reg_fence(v1);
        const float4 *wrow = reinterpret_cast<const float4 *>(ws.wq + static_cast<int64_t>(row) * kHeads);
        float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
        if (!any_neg) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 wv = __ldg(wrow + c);
            acc0 = fmaf(wv.x, fmaxf(__uint_as_float(v0[4 * c + 0]), 0.f), acc0);
            acc1 = fmaf(wv.y, fmaxf(__uint_as_float(v0[4 * c + 1]), 0.f), acc1);
            acc2 = fmaf(wv.z, fmaxf(__uint_as_float(v0[4 * c + 2]), 0.f), acc2);
            acc3 = fmaf(wv.w, fmaxf(__uint_as_float(v0[4 * c + 3]), 0.f), acc3);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 wv = __ldg(wrow + 8 + c);
            acc0 = fmaf(wv.x, fmaxf(__uint_as_float(v1[4 * c + 0]), 0.f), acc0);
            acc1 = fmaf(wv.y, fmaxf(__uint_as_float(v1[4 * c + 1]), 0.f), acc1);
            acc2 = fmaf(wv.z, fmaxf(__uint_as_float(v1[4 * c + 2]), 0.f), acc2);
            acc3 = fmaf(wv.w, fmaxf(__uint_as_float(v1[4 * c + 3]), 0.f), acc3);
          }
        } else {
          // ReLU(s * d) = s * min(d, 0) when s < 0.
          const bool nz = neg_scale;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float4 wv = __ldg(wrow + c);
            const uint32_t *v = c < 8 ? v0 : v1;
            const int o = (c & 7) * 4;
            const float e0 = __uint_as_float(v[o + 0]), e1 = __uint_as_float(v[o + 1]);
            const float e2 = __uint_as_float(v[o + 2]), e3 = __uint_as_float(v[o + 3]);
            acc0 = fmaf(wv.x, nz ? fminf(e0, 0.f) : fmaxf(e0, 0.f), acc0);
            acc1 = fmaf(wv.y, nz ? fminf(e1, 0.f) : fmaxf(e1, 0.f), acc1);
            acc2 = fmaf(wv.z, nz ? fminf(e2, 0.f) : fmaxf(e2, 0.f), acc2);
            acc3 = fmaf(wv.w, nz ? fminf(e3, 0.f) : fmaxf(e3, 0.f), acc3);
          }
        }
        if (i == grp.nrows - 1) {
          // Accumulator buffer fully read: hand it back to the MMA issuer.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->tempty[set]);
        }
        const float score = ((acc0 + acc1) + (acc2 + acc3)) * scale;
        const bool keep = valid && pos < ws.bound_eff[row];
        if (keep) a.scores[static_cast<int64_t>(row) * a.ld + pos] = score;
        const uint32_t digit = keep ? (radix_key(score) >> 26) : 64u;
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        if (digit < 64u && lane == __ffs(peers) - 1) atomicAdd(&hist[i * 64 + digit], __popc(peers));
      }
    }
    if (cur_g >= 0) flush();
  }

  // Every role is done (or gave up); release TMEM.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int KV>
cudaError_t launch_kv(const CUtensorMap &kmap, const ScoreArgs &a, int num_ctas, cudaStream_t stream) {
  static bool configured = false;
  constexpr int bytes = smem_bytes<KV>();
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(score_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  score_kernel<KV><<<num_ctas, kThreads, bytes, stream>>>(kmap, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(const CUtensorMap &kmap, const ScoreArgs &a, int kv_dtype, int num_ctas,
                         cudaStream_t stream) {
  if (kv_dtype == IDX_KV_E4M3) return launch_kv<IDX_KV_E4M3>(kmap, a, num_ctas, stream);
  return launch_kv<IDX_KV_BF16>(kmap, a, num_ctas, stream);
}

}  // namespace idx
