// The scoring scan: paged key loads (TMA), the tensor-core contraction
// (tcgen05, accumulator in TMEM), the ReLU-weighted head reduction, the score
// store and the fused score histogram.
//
// sglang PR 48224 page (sgl-amd-mono #86): "scores every cached key of each row"
// (section Motivation, first paragraph); rows of one request read each key once
// (section Modifications, commit 1); the store drops "keys at or past a row's
// bound" (commit 2); the first radix digit radix_key >> 26 of every stored score
// is counted in 64 bins per row during the scan, so the selection needs no pass
// of its own for it (commit 4, the score_hist mailbox).  Here the scan counts the
// top 12 bits of the radix key; the first digit's 64 bins are its marginal.
//
// GB300 layout of the work.  One persistent CTA per SM walks an even share of
// the launch's tiles; a tile is 128 consecutive key positions (two pages) of one
// row group (up to 4 rows of one request).  For a tile the contraction is
//     D[key][row*64 + head] = <k_key, q_row_head>      (M = 128, N = 64 * rows)
// so a TMEM lane holds one key and each epilogue thread reduces its key's 64
// head values of a row in registers.
//   warp 0      producer (with warp 18 for an E4M3 cache: even / odd tiles):
//               page ids (32 per lane load, a block ahead), TMA of the
//               key pages into an smem ring, the keys' scales into a second ring
//               (two 256-byte bulk copies per tile), and the group's query operand
//               (bulk copy) on group changes;
//   warp 1      MMA issuer (one thread) and TMEM owner; two accumulators in TMEM,
//               so the MMA of tile k+1 runs while tile k's epilogue reads;
//   warps 2..17 epilogue, two groups of eight taking alternate tiles (group g
//               reads accumulator g), four warps per TMEM lane quarter; each warp
//               reduces two rows of its group's tiles for its quarter, so the
//               per-tile costs (waits, scales, hand-back) are paid once per two
//               rows and the groups work out of step with each other.
// E4M3 cache: keys feed tcgen05.mma kind::f8f6f4 straight from the TMA ring; the
// query is split exactly into two E4M3 terms (prep.cu), run as K = 2 x 128.
// bf16 cache: keys and query are bf16, kind::f16, K = 128.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kProducers = 2;                  // producer warps for an E4M3 cache
constexpr int kProducer2Warp = 2 + kEpiWarps;  // the second one, after the epilogue warps
constexpr int kThreads = 64 + kEpiWarps * 32 + 32;
constexpr int kBOperandBytes = 2 * kMaxGroupRows * kRowOperandBytes;  // two K blocks
constexpr int kTmemCols = 512;                                        // two accumulators of 256
constexpr int kScaleSlots = 8;
constexpr int kHistWords = kHistBins / 2;   // two 16-bit counters per word
constexpr int kFlushTiles = 256;            // 256 tiles x 128 keys < 65536: no counter overflows

template <int KV>
struct Cfg {
  static constexpr int kStageBytes = KV == IDX_KV_E4M3 ? kTileKeys * kDim : kTileKeys * kDim * 2;
  static constexpr int kStages = KV == IDX_KV_E4M3 ? 6 : 3;
  static constexpr int kPageBytes = kStageBytes / 2;
};

struct Barriers {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t sfull[kScaleSlots];
  uint64_t sempty[kScaleSlots];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t bfull;
  uint64_t bfree;
  uint64_t drain;
  uint64_t hdone[1];     // every epilogue warp finished adding to the histograms
  uint64_t hflushed[1];  // every epilogue warp finished flushing them
  uint32_t tmem_base;
  int abort;
};

template <int KV>
struct Smem {
  static constexpr int kB = 0;
  static constexpr int kA = kB + kBOperandBytes;
  static constexpr int kHist = kA + Cfg<KV>::kStages * Cfg<KV>::kStageBytes;
  static constexpr int kScales = kHist + kMaxGroupRows * kHistWords * 4;
  static constexpr int kW = kScales + (KV == IDX_KV_E4M3 ? kScaleSlots * kTileKeys * 4 : 0);
  static constexpr int kBars = kW + kEpiWarps * 2 * kHeads * 4;
  static constexpr int kBytes = kBars + static_cast<int>(sizeof(Barriers));
  static constexpr int kDynamic = kBytes + 1024;  // alignment slack
};
static_assert(Smem<IDX_KV_E4M3>::kDynamic <= 227 * 1024, "shared memory");
static_assert(Smem<IDX_KV_BF16>::kDynamic <= 227 * 1024, "shared memory");

// Walks the groups of a CTA's tile range in order.
struct GroupCursor {
  const Group *groups;
  int num_groups;
  int g;
  int next_begin;
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
  __device__ bool advance(int t) {
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

// sum_h w[h] * relu(v[h]) over 32 heads, with the weights already halved:
// v + |v| = 2 relu(v) exactly, one FADD (the |v| is an operand modifier) on the
// FMA pipe instead of a max on the ALU pipe, then packed FMAs into four
// accumulators so that the FMAs of one row form four short chains.
__device__ __forceinline__ void relu_dot32(const uint32_t (&v)[32], const float4 *w, float2 (&acc)[4]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 wv = w[c];
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float d = __uint_as_float(v[4 * c + i]);
      e[i] = d + fabsf(d);
    }
    acc[(2 * c) & 3] = __ffma2_rn(make_float2(e[0], e[1]), make_float2(wv.x, wv.y), acc[(2 * c) & 3]);
    acc[(2 * c + 1) & 3] = __ffma2_rn(make_float2(e[2], e[3]), make_float2(wv.z, wv.w), acc[(2 * c + 1) & 3]);
  }
}

// ReLU(s * d) = s * min(d, 0) for a negative scale s: the other branch
// (d - |d| = 2 min(d, 0), again with the halved weights).
__device__ __forceinline__ void relu_dot32_signed(const uint32_t (&v)[32], const float4 *w, bool neg,
                                                  float2 (&acc)[4]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 wv = w[c];
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float d = __uint_as_float(v[4 * c + i]);
      e[i] = neg ? d - fabsf(d) : d + fabsf(d);
    }
    acc[0] = __ffma2_rn(make_float2(e[0], e[1]), make_float2(wv.x, wv.y), acc[0]);
    acc[1] = __ffma2_rn(make_float2(e[2], e[3]), make_float2(wv.z, wv.w), acc[1]);
  }
}

template <int KV>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ CUtensorMap kmap,
                                                             const ScoreArgs a) {
  using C = Cfg<KV>;
  using S = Smem<KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sB0 = smem + S::kB;                          // K block 0 of the group's query operand
  uint8_t *sB1 = smem + S::kB + kBOperandBytes / 2;     // K block 1
  uint8_t *sA = smem + S::kA;                           // key ring
  uint32_t *shist = reinterpret_cast<uint32_t *>(smem + S::kHist);   // [row][2048] packed 16-bit counts
  float *sscale = reinterpret_cast<float *>(smem + S::kScales);     // [slot][128]
  float *sw = reinterpret_cast<float *>(smem + S::kW);              // [epilogue warp][64]
  Barriers *bars = reinterpret_cast<Barriers *>(smem + S::kBars);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Workspace &ws = a.ws;

  // Set-up that reads nothing from the prep launch runs before waiting for it.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < kScaleSlots; ++s) {
      mbar_init(&bars->sfull[s], 1);           // the producer's arrival; the copies complete by bytes
      mbar_init(&bars->sempty[s], kEpiWarps / 2);   // the eight warps of the tile's group
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->tfull[s], 1);
      mbar_init(&bars->tempty[s], kEpiWarps / 2);
    }
    mbar_init(&bars->hdone[0], kEpiWarps);
    mbar_init(&bars->hflushed[0], kEpiWarps);
    mbar_init(&bars->bfull, 1);
    mbar_init(&bars->bfree, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < kMaxGroupRows * kHistWords; i += kThreads) shist[i] = 0u;
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&kmap);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_wait();   // the plan and the query operands come from the prep launch
  const int total_tiles = ws.plan->total_tiles;
  const int num_groups = ws.plan->num_groups;
  const int64_t t0 = static_cast<int64_t>(total_tiles) * blockIdx.x / gridDim.x;
  const int64_t t1 = static_cast<int64_t>(total_tiles) * (blockIdx.x + 1) / gridDim.x;
  grid_dependency_trigger();
  if (t0 >= t1) {  // uniform for the CTA: no tiles, give the TMEM back
    if (warp == 1) tmem_dealloc(bars->tmem_base, kTmemCols);
    return;
  }
  const uint32_t tmem_base = bars->tmem_base;
  const uint64_t limit = a.wait_limit_ns;
  volatile int *abort = &bars->abort;

  if (warp == 0 || (KV == IDX_KV_E4M3 && kProducers == 2 && warp == kProducer2Warp)) {
    // ------------------------------------------------------------------ producer
    // E4M3: two producer warps, warp 0 for the even tiles of the CTA's range and
    // warp kProducer2Warp for the odd ones (their key stages and scale slots are
    // disjoint: both ring lengths are even); bf16: warp 0 alone.  In each, the whole
    // warp runs the loop: lanes hold the page ids of the current and next block of
    // 16 tiles (32 pages, one lane each); lane 0 issues the key pages' TMA and the
    // bulk copies of their 128 key scales.  Warp 0 also loads the query
    // operand of every group of the range, in order.
    const int pp = warp == 0 ? 0 : 1;           // this producer's tile parity
    const int np = KV == IDX_KV_E4M3 ? kProducers : 1;
    const uint64_t policy = l2_evict_first_policy();
    GroupCursor cur;
    cur.seek(ws.groups, num_groups, static_cast<int>(t0));
    int cur_g = -1, req = 0, L = 0, tile_begin = 0;
    int32_t blk_ids = -2, nxt_ids = -2;   // this lane's page id in the current / next block
    int blk = -1;                          // current block of 16 tiles within the group
    // Waits are taken by lane 0 and the outcome broadcast, so the lanes never split.
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar, parity, limit, abort);
      return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    auto block_ids = [&](int b) -> int32_t {
      const int64_t page = static_cast<int64_t>(b) * 32 + lane;
      return page * kPage < L ? a.page_table[static_cast<int64_t>(req) * a.pt_stride + page] : -2;
    };
    // warp 0: the query operand of every group with tiles in the range that starts
    // at or before tile `upto`, in order (groups without tiles have none: the MMA
    // issuer never switches to them)
    int nb = 0;                                 // query operands loaded
    int bg = cur.g;                             // next group to consider (seek lands on a group with tiles)
    auto load_b_upto = [&](int64_t upto) -> bool {
      while (bg < num_groups) {
        const int begin = ws.groups[bg].tile_begin;
        if (begin > upto || begin >= t1) break;
        const int end = bg + 1 < num_groups ? ws.groups[bg + 1].tile_begin : total_tiles;
        if (end > begin) {
          if (nb > 0 && !warp_wait(&bars->bfree, (nb - 1) & 1)) return false;
          if (lane == 0) {
            const Group grp = ws.groups[bg];
            const uint32_t bytes = grp.nrows * kRowOperandBytes;
            mbar_arrive_expect_tx(&bars->bfull, 2 * bytes);
            bulk_load(sB0, ws.qop0 + static_cast<int64_t>(grp.row0) * kRowOperandBytes, bytes, &bars->bfull);
            bulk_load(sB1, ws.qop1 + static_cast<int64_t>(grp.row0) * kRowOperandBytes, bytes, &bars->bfull);
          }
          ++nb;
        }
        ++bg;
      }
      return true;
    };
    bool ok = true;
    int last_k = -1;
    int s = pp;                 // this producer's stage of tile k and the phase it waits for
    uint32_t ephase = 1u;
    static_assert(C::kStages % kProducers == 0 || KV != IDX_KV_E4M3, "producers alternate stages");
    for (int64_t t = t0 + pp; t < t1; t += np, s += np) {
      if (s >= C::kStages) {
        s -= C::kStages;
        ephase ^= 1u;
      }
      const int k = static_cast<int>(t - t0);
      if (pp == 0 && !load_b_upto(t)) {
        ok = false;
        break;
      }
      if (cur.advance(static_cast<int>(t)) || cur_g < 0) {
        const Group grp = ws.groups[cur.g];
        cur_g = cur.g;
        req = grp.req;
        L = grp.L;
        tile_begin = grp.tile_begin;
        blk = (static_cast<int>(t) - tile_begin) >> 4;
        blk_ids = block_ids(blk);
        nxt_ids = block_ids(blk + 1);
      }
      const int j = static_cast<int>(t) - tile_begin;
      if ((j >> 4) != blk) {               // next block: its ids were loaded a block ago
        blk = j >> 4;
        blk_ids = nxt_ids;
        nxt_ids = block_ids(blk + 1);
      }
      int32_t pages[2];
      pages[0] = __shfl_sync(0xffffffffu, blk_ids, (j & 15) * 2);
      pages[1] = __shfl_sync(0xffffffffu, blk_ids, (j & 15) * 2 + 1);
      const int ss = k % kScaleSlots;
      if (!warp_wait(&bars->empty[s], ephase) ||
          (KV == IDX_KV_E4M3 && !warp_wait(&bars->sempty[ss], ((k / kScaleSlots) & 1) ^ 1))) {
        ok = false;
        break;
      }
      uint32_t bytes = 0;
      for (int h = 0; h < 2; ++h) {
        if (pages[h] == -2) {
          pages[h] = -1;
        } else if (pages[h] >= 0 && pages[h] < a.P) {
          bytes += C::kPageBytes;
        } else {
          pages[h] = -1;
          if (lane == 0) flag_status(ws.status, kStatusBadPage);
        }
      }
      uint8_t *dst = sA + s * C::kStageBytes;
      if (lane == 0) {
        if (KV == IDX_KV_E4M3) {
          // the two pages' 64 scales each (256 bytes, one bulk copy per page)
          mbar_arrive_expect_tx(&bars->sfull[ss], (pages[0] >= 0 ? 256u : 0u) + (pages[1] >= 0 ? 256u : 0u));
          for (int h = 0; h < 2; ++h)
            if (pages[h] >= 0)
              bulk_load(sscale + ss * kTileKeys + h * kPage, a.k_scale + static_cast<int64_t>(pages[h]) * kPage, 256u,
                        &bars->sfull[ss]);
        }
        mbar_arrive_expect_tx(&bars->full[s], bytes);
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
      last_k = k;
    }
    if (ok && pp == 0) ok = load_b_upto(t1 - 1);   // groups whose tiles all fell to the other producer
    if (!ok && lane == 0) set_abort(bars, ws.status);
    // Wait for every copy this warp still has in flight before the CTA may exit (also
    // after an abort): for each stage and scale slot, its last use by this warp.
    int never = 0;
    auto last_use = [&](int slot, int ring) -> int {   // largest k <= last_k of this warp's parity
      if (last_k < 0) return -1;
      const int back = ((last_k - slot) % ring + ring) % ring;
      const int kk = last_k - back;
      return (kk >= 0 && (kk - pp) % np == 0) ? kk : -1;
    };
    for (int s = 0; s < C::kStages; ++s) {
      const int lu = last_use(s, C::kStages);
      if (lu >= 0 && !mbar_wait(&bars->full[s], (lu / C::kStages) & 1, limit, &never) && lane == 0)
        flag_status(ws.status, kStatusTimeout);
    }
    if (KV == IDX_KV_E4M3) {
      for (int s = 0; s < kScaleSlots; ++s) {
        const int lu = last_use(s, kScaleSlots);
        if (lu >= 0 && !mbar_wait(&bars->sfull[s], (lu / kScaleSlots) & 1, limit, &never) && lane == 0)
          flag_status(ws.status, kStatusTimeout);
      }
    }
    if (pp == 0 && nb > 0 && !mbar_wait(&bars->bfull, (nb - 1) & 1, limit, &never) && lane == 0)
      flag_status(ws.status, kStatusTimeout);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      GroupCursor cur;
      cur.seek(ws.groups, num_groups, static_cast<int>(t0));
      int cur_g = -1, nswitch = 0;
      uint32_t idesc = 0;
      const uint32_t fmt = KV == IDX_KV_E4M3 ? 0u : 1u;
      const uint64_t bdesc0 = umma_desc_sw128(smem_u32(sB0)), bdesc1 = umma_desc_sw128(smem_u32(sB1));
      // stage s of tile k and its phase, kept incrementally (no division per tile);
      // stage s's A descriptor is stage 0's plus s stages of bytes / 16
      const uint64_t adesc0 = umma_desc_sw128(smem_u32(sA));
      int s = 0;
      uint32_t sphase = 0;
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
        const int acc = k & 1;
        if (!mbar_wait(&bars->full[s], sphase, limit, abort) ||
            !mbar_wait(&bars->tempty[acc], ((k >> 1) & 1) ^ 1, limit, abort)) {
          set_abort(bars, ws.status);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * 256;
        // descriptors of the K steps: the base descriptor plus the step's byte offset / 16
        // (the start-address field holds address / 16; no carry out of it in 256 KB)
        const uint64_t adesc = adesc0 + static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          const uint64_t bd = (kk < 4 ? bdesc0 : bdesc1) + (koff >> 4);
          if (KV == IDX_KV_E4M3) {
            umma_f8(d, adesc + (koff >> 4), bd, idesc, kk > 0);
          } else {
            umma_f16(d, adesc + (((kk < 4 ? 0u : static_cast<uint32_t>(kTileKeys) * 128u) + koff) >> 4), bd, idesc,
                     kk > 0);
          }
        }
        umma_commit(&bars->empty[s]);
        if (!(a.stall_first_handoff && k == 0)) umma_commit(&bars->tfull[acc]);
        if (++s == C::kStages) {
          s = 0;
          sphase ^= 1u;
        }
      }
      // All MMAs issued by this thread complete before TMEM is released.
      umma_commit(&bars->drain);
      int never = 0;
      if (!mbar_wait(&bars->drain, 0, limit, &never)) flag_status(ws.status, kStatusTimeout);
    }
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------------ epilogue
    // Two groups of eight warps take alternate tiles (group g reads accumulator g);
    // within a group each warp reduces two rows of the tile for its TMEM lane quarter.
    const int ew = warp - 2;
    const int quarter = warp & 3;            // TMEM lane quarter this warp may read
    const int slot = ew >> 2;                // 0..3 among the quarter's four warps
    const int tg = slot & 1;                 // tile parity this warp handles
    const int r0 = (slot >> 1) * 2;          // first of this warp's two group rows
    float *myw = sw + ew * 2 * kHeads;       // the two rows' weights
    GroupCursor cur;
    cur.seek(ws.groups, num_groups, static_cast<int>(t0));
    int cur_g = -1;
    Group grp;
    grp.nrows = 0;
    grp.row0 = 0;
    bool mine[2] = {false, false};
    int32_t bnd[2] = {0, 0};
    int flushes = 0;
    bool ok = true;

    // Every row's histogram goes to global memory (12-bit counts, the 64-bin first
    // digit, and the caller's copy of the latter when asked) and is cleared; all
    // sixteen warps meet before and after.  The group's nrows x 64 (row, first digit)
    // blocks of 64 bins are dealt round-robin to the warps, four at a time: the four
    // shared-memory reads go out together, and a block with no count (most of them:
    // a CTA's scores fill a few hundred of a row's 4096 bins) costs one vote.
    auto flush = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->hdone[0]);
      if (!mbar_wait(&bars->hdone[0], flushes & 1, limit, abort)) return false;
      const int nblk = grp.nrows * 64;
      for (int b0 = ew; b0 < nblk; b0 += 4 * kEpiWarps) {
        uint32_t wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int b = b0 + i * kEpiWarps;
          wv[i] = b < nblk ? shist[(b >> 6) * kHistWords + (b & 63) * 32 + lane] : 0u;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (__ballot_sync(0xffffffffu, wv[i] != 0u) == 0u) continue;   // uniform for the warp
          const int b = b0 + i * kEpiWarps;
          const int row = b >> 6, d = b & 63;
          const int64_t grow = grp.row0 + row;
          const uint32_t lo = wv[i] & 0xFFFFu, hi = wv[i] >> 16;
          if (wv[i]) {
            shist[row * kHistWords + d * 32 + lane] = 0u;
            if (lo) atomicAdd(&ws.hist12[grow * kHistBins + d * 64 + 2 * lane], lo);
            if (hi) atomicAdd(&ws.hist12[grow * kHistBins + d * 64 + 2 * lane + 1], hi);
          }
          const uint32_t dsum = __reduce_add_sync(0xffffffffu, lo + hi);
          if (lane == 0) {
            atomicAdd(&ws.hist64[grow * 64 + d], dsum);
            if (a.hist != nullptr) atomicAdd(&a.hist[grow * 64 + d], dsum);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->hflushed[0]);
      const bool r = mbar_wait(&bars->hflushed[0], flushes & 1, limit, abort);
      ++flushes;
      return r;
    };

    // The two groups see different tiles, so the flush points (every group start
    // and every kFlushTiles tiles within a group; 16-bit counters) are defined on
    // the CTA's tile sequence and every warp takes each of them, in order.
    auto load_group = [&]() {
      grp = ws.groups[cur.g];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mine[i] = r0 + i < grp.nrows;
        bnd[i] = mine[i] ? ws.bound_eff[grp.row0 + r0 + i] : 0;
        if (mine[i]) {
          const float2 v =
              reinterpret_cast<const float2 *>(ws.wq + static_cast<int64_t>(grp.row0 + r0 + i) * kHeads)[lane];
          reinterpret_cast<float2 *>(myw + i * kHeads)[lane] = v;
        }
      }
      __syncwarp();
    };
    int64_t done = t0;   // flush points at or before this tile are taken
    auto catch_up = [&](int64_t upto) -> bool {   // takes every flush point p in (done, upto]
      for (;;) {
        const int64_t periodic =
            grp.tile_begin + ((done - grp.tile_begin) / kFlushTiles + 1) * static_cast<int64_t>(kFlushTiles);
        const int64_t p = periodic < cur.next_begin ? periodic : static_cast<int64_t>(cur.next_begin);
        if (p > upto) break;
        if (!flush()) return false;
        if (p == cur.next_begin) {
          cur.advance(static_cast<int>(p));
          load_group();
        }
        done = p;
      }
      if (upto > done) done = upto;
      return true;
    };
    load_group();
    cur_g = cur.g;

    for (int64_t t = t0 + tg; t < t1; t += 2) {
      const int k = static_cast<int>(t - t0);
      if (!catch_up(t)) {
        ok = false;
        break;
      }
      const int j = static_cast<int>(t) - grp.tile_begin;
      const int64_t pos = static_cast<int64_t>(j) * kTileKeys + quarter * 32 + lane;
      const int acc = tg;
      const int ss = k % kScaleSlots;
      float scale = 1.0f;
      if (KV == IDX_KV_E4M3) {
        if (!mbar_wait(&bars->sfull[ss], (k / kScaleSlots) & 1, limit, abort)) {
          set_abort(bars, ws.status);
          ok = false;
          break;
        }
        scale = sscale[ss * kTileKeys + quarter * 32 + lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->sempty[ss]);
      }
      if (!mbar_wait(&bars->tfull[acc], (k >> 1) & 1, limit, abort)) {
        set_abort(bars, ws.status);
        ok = false;
        break;
      }
      tc_fence_after();
      float score[2] = {0.f, 0.f};
      const bool valid = pos < grp.L;
      const bool neg = valid && scale < 0.0f;
      const bool any_neg = __any_sync(0xffffffffu, neg);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (!mine[i]) continue;            // uniform for the warp
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * 256 + (r0 + i) * 64;
        const float4 *w4 = reinterpret_cast<const float4 *>(myw + i * kHeads);
        float2 accs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          tmem_ld32(taddr + half * 32, v);
          tmem_wait_ld();
          reg_fence(v);
          if (!any_neg) relu_dot32(v, w4 + half * 8, accs);
          else relu_dot32_signed(v, w4 + half * 8, neg, accs);
        }
        score[i] = (((accs[0].x + accs[0].y) + (accs[1].x + accs[1].y)) + ((accs[2].x + accs[2].y) + (accs[3].x + accs[3].y))) * scale;
      }
      // Accumulator read: hand it back to the MMA issuer.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[acc]);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (!mine[i]) continue;
        const bool keep = valid && pos < bnd[i];
        if (keep) a.scores[static_cast<int64_t>(grp.row0 + r0 + i) * a.ld + pos] = score[i];
        const uint32_t bin = radix_key(score[i]) >> (32 - kHistBits);
        uint32_t *h = shist + (r0 + i) * kHistWords;
        if (keep) atomicAdd(&h[bin >> 1], 1u << ((bin & 1) * 16));   // shared-memory atomics resolve collisions
      }
    }
    if (ok && catch_up(t1 - 1)) flush();
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
  static std::mutex mu;
  static bool done[128] = {};
  constexpr int bytes = Smem<KV>::kDynamic;
  const cudaError_t e = once_per_device(mu, done, [] {
    return cudaFuncSetAttribute(score_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, score_kernel<KV>, kmap, a);
}

}  // namespace

cudaError_t launch_score(const CUtensorMap &kmap, const ScoreArgs &a, int kv_dtype, int num_ctas,
                         cudaStream_t stream) {
  if (kv_dtype == IDX_KV_E4M3) return launch_kv<IDX_KV_E4M3>(kmap, a, num_ctas, stream);
  return launch_kv<IDX_KV_BF16>(kmap, a, num_ctas, stream);
}

}  // namespace idx
