// The scoring scan: paged key loads (TMA), the tensor-core contraction
// (tcgen05, accumulator in TMEM), the ReLU-weighted head reduction, the score
// store and the fused score histogram.
//
// sglang PR 48224 page (sgl-amd-mono #86): each row is scored against every key
// its request has cached (section Motivation, first paragraph); rows of one
// request read each key once (section Modifications, commit 1); positions from a
// row's bound on are not stored (commit 2); the first radix digit radix_key >> 26 of every stored score
// is counted in 64 bins per row during the scan, so the selection needs no pass
// of its own for it (commit 4, the score_hist mailbox).  Here the scan counts the
// top 12 bits of the radix key; the first digit's 64 bins are its marginal.
//
// GB300 layout of the work.  One persistent CTA per SM walks an even share of
// the launch's tiles; a tile is 128 consecutive key positions (two pages) of one
// row group (up to 4 rows of one request).  For a tile the contraction is
//     D[key][row*64 + head] = <k_key, q_row_head>      (M = 128, N = 64 * rows)
// so a TMEM lane holds one key; the 64 head values of a (key, row) are reduced by
// four threads of one warp.
//   warp 0      producer (with warp 18 for an E4M3 cache: even / odd tiles):
//               page ids (32 per lane load, a block ahead), TMA of the
//               key pages into an smem ring, the keys' scales into a second ring
//               (two 256-byte bulk copies per tile), and the group's query operand
//               (bulk copy) on group changes;
//   warp 1      MMA issuer (lane 0) and TMEM owner; two accumulators in TMEM,
//               so the MMA of tile k+1 runs while tile k's epilogue reads; with an
//               E4M3 cache lane 0 of warp 19 issues the odd tiles' MMAs;
//   warps 2..17 epilogue: every warp takes every tile, one row for its TMEM lane
//               quarter (warp % 4), reading the row's 64 columns in the 16x256b
//               shape so that each thread needs only 16 of the row's weights
//               (held in registers), and hands the accumulator back right after
//               its last TMEM read.
// The batched instance (kBatched, for launches whose requests have one or two
// rows: a lone live row and its pad row) fills each accumulator with 4 / rows
// tiles of a group and gives every epilogue warp one (tile, row) of the batch.
// E4M3 cache: keys feed tcgen05.mma kind::f8f6f4 straight from the TMA ring; the
// query is split exactly into two E4M3 terms (prep.cu), run as K = 2 x 128.
// bf16 cache: keys and query are bf16, kind::f16, K = 128.
#include "idx_device.cuh"
#include "launch.h"

namespace idx {
namespace {

constexpr int kEpiWarps = 16;                  // the histogram flush deals its blocks for sixteen
constexpr int kProducers = 2;                  // producer warps for an E4M3 cache
constexpr int kEpiWarp0 = 2;                            // warps 2 .. 17: the epilogue
constexpr int kProducer2Warp = kEpiWarp0 + kEpiWarps;   // the second producer, after the epilogue warps
constexpr int kMma2Warp = kProducer2Warp + 1;           // the second MMA issuer (odd tiles)
constexpr int kThreads = (kMma2Warp + 1) * 32;
template <int KV>
constexpr int kIssuers = KV == IDX_KV_E4M3 ? 2 : 1;   // MMA-issuing threads
constexpr int kBOperandBytes = 2 * kMaxGroupRows * kRowOperandBytes;  // two K blocks
constexpr int kSlots = 2;                    // accumulators in TMEM, used alternately
constexpr int kSlotCols = 256;               // one tile: up to four rows x 64 heads
constexpr int kTmemCols = kSlots * kSlotCols;
constexpr int kScaleSlots = 8;
constexpr int kHistWords = kHistBins / 2;   // two 16-bit counters per word
constexpr int kFlushTiles = 256;            // 256 tiles x 128 keys < 65536: no counter overflows
constexpr int kStageBlocks = 4;             // histogram blocks each epilogue warp has in flight to global

// Groups of one or two rows leave most of an accumulator's 256 columns and most
// epilogue warps idle.  The batched instance of the kernel (chosen by the host
// when the caller says that no request has more than two rows) puts the CTA's
// tiles into the accumulators in batches instead: 4 / rows consecutive tiles of
// one group share one accumulator (N = 64 x rows each) and each epilogue warp
// reduces one (tile, row) of a batch.  Groups of three or four rows still run
// one tile per batch there, so the batched instance is exact for any rows.
__device__ __forceinline__ int batch_tiles(int nrows) { return nrows <= 2 ? 4 / nrows : 1; }

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
  uint64_t tfull[kSlots];
  uint64_t tempty[kSlots];
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
  static constexpr int kFlushStage = kScales + (KV == IDX_KV_E4M3 ? kScaleSlots * kTileKeys * 4 : 0);
  static constexpr int kBars = kFlushStage + kEpiWarps * kStageBlocks * 64 * 4;
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

// One row's 16x256b.x4 fragment pair folded into the four keys' running sums.
// Fragment va holds keys lane/4 (registers 4k, 4k+1) and lane/4 + 8 (4k+2,
// 4k+3), vb the keys 16 lanes further on; repetition k holds heads
// 8k + 2 (lane % 4) + {0, 1} of the half, whose halved weights are w[k].
// v + |v| = 2 relu(v) exactly: one packed add per head pair, then a packed FMA
// per head pair.
__device__ __forceinline__ void relu_frag(const uint32_t (&va)[16], const uint32_t (&vb)[16], const float2 *w,
                                          float2 (&a)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // key j: registers 4k + 2 (j % 2) + {0, 1} of va (j < 2) or vb
      const uint32_t *v = j < 2 ? va : vb;
      const float2 x = make_float2(__uint_as_float(v[4 * k + 2 * (j & 1)]), __uint_as_float(v[4 * k + 2 * (j & 1) + 1]));
      const float2 e = __fadd2_rn(x, make_float2(fabsf(x.x), fabsf(x.y)));
      a[j] = __ffma2_rn(e, w[k], a[j]);
    }
  }
}

// As relu_frag, with ReLU(s d) = s min(d, 0) for the keys whose scale s is
// negative (neg bit m for key m): there the other branch, d - |d| = 2 min(d, 0).
__device__ __forceinline__ void relu_frag_signed(const uint32_t (&va)[16], const uint32_t (&vb)[16],
                                                 const float2 *w, uint32_t neg, float2 (&a)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float e[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float x = __uint_as_float(va[4 * k + i]);
      const float y = __uint_as_float(vb[4 * k + i]);
      e[i] = ((neg >> (i >> 1)) & 1u) ? x - fabsf(x) : x + fabsf(x);
      e[4 + i] = ((neg >> (2 + (i >> 1))) & 1u) ? y - fabsf(y) : y + fabsf(y);
    }
    a[0] = __ffma2_rn(make_float2(e[0], e[1]), w[k], a[0]);
    a[1] = __ffma2_rn(make_float2(e[2], e[3]), w[k], a[1]);
    a[2] = __ffma2_rn(make_float2(e[4], e[5]), w[k], a[2]);
    a[3] = __ffma2_rn(make_float2(e[6], e[7]), w[k], a[3]);
  }
}

// The four threads 4g .. 4g+3 of a warp hold partial sums of the same four keys
// (s[m] for key m); afterwards thread i holds the whole sum of key i % 4.
__device__ __forceinline__ float reduce_quad(const float (&s)[4], int lane) {
  const bool hi2 = (lane & 2) != 0;
  float k0 = hi2 ? s[2] : s[0];
  float k1 = hi2 ? s[3] : s[1];
  k0 += __shfl_xor_sync(0xffffffffu, hi2 ? s[0] : s[2], 2);
  k1 += __shfl_xor_sync(0xffffffffu, hi2 ? s[1] : s[3], 2);
  const bool hi1 = (lane & 1) != 0;
  float k = hi1 ? k1 : k0;
  k += __shfl_xor_sync(0xffffffffu, hi1 ? k0 : k1, 1);
  return k;
}

template <int KV, bool kBatched>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ CUtensorMap kmap,
                                                             const ScoreArgs a) {
  using C = Cfg<KV>;
  using S = Smem<KV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array itself, so that the
  // compiler keeps every pointer below in the shared address space
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *sB0 = smem + S::kB;                          // K block 0 of the group's query operand
  uint8_t *sB1 = smem + S::kB + kBOperandBytes / 2;     // K block 1
  uint8_t *sA = smem + S::kA;                           // key ring
  uint32_t *shist = reinterpret_cast<uint32_t *>(smem + S::kHist);   // [row][2048] packed 16-bit counts
  float *sscale = reinterpret_cast<float *>(smem + S::kScales);     // [slot][128]
  uint32_t *sflush = reinterpret_cast<uint32_t *>(smem + S::kFlushStage);   // [epilogue warp][4][64]
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
      // every epilogue thread passes every tile (batched: every warp, for its share)
      mbar_init(&bars->sempty[s], kBatched ? kEpiWarps : kEpiWarps * 32);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars->tfull[s], kBatched ? kIssuers<KV> : 1);   // batched: every issuer commits every batch
      // every epilogue thread reads every tile (batched: every warp)
      mbar_init(&bars->tempty[s], kBatched ? kEpiWarps : kEpiWarps * 32);
    }
    mbar_init(&bars->hdone[0], kEpiWarps);
    mbar_init(&bars->hflushed[0], kEpiWarps);
    mbar_init(&bars->bfull, 1);
    mbar_init(&bars->bfree, kIssuers<KV>);   // every MMA issuer is done with the group's query operand
    mbar_init(&bars->drain, kIssuers<KV>);
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
  } else if (warp == 1 || warp == kMma2Warp) {
    // ------------------------------------------------------------------ MMA issuers
    // Tile k of the CTA's sequence accumulates into TMEM slot k % 2 (N = 64 x the
    // group's rows); its MMA waits for the epilogue of tile k - 2.  With an E4M3
    // cache two threads issue the MMAs, lane 0 of warp 1 for the even tiles (slot
    // 0, even key stages) and lane 0 of warp kMma2Warp for the odd ones (slot 1,
    // odd stages), so that one thread's per-tile waits and bookkeeping overlap the
    // other's issue; each stage and slot barrier then has one waiter, which the
    // parity waits need.  With a bf16 cache (three stages) warp 1 issues them all.
    // Every issuer walks every group that has tiles in the CTA's range, waiting
    // for its query operand and releasing it afterwards, whether or not it has
    // tiles of its own there.
    constexpr int nis = kIssuers<KV>;
    if (lane == 0 && (warp == 1 || nis == 2)) {
      const int par = warp == 1 ? 0 : 1;
      const uint32_t fmt = KV == IDX_KV_E4M3 ? 0u : 1u;
      const uint64_t bdesc0 = umma_desc_sw128(smem_u32(sB0)), bdesc1 = umma_desc_sw128(smem_u32(sB1));
      // stage s of tile k and its phase, kept incrementally; stage s's A descriptor
      // is stage 0's plus s stages of bytes / 16
      const uint64_t adesc0 = umma_desc_sw128(smem_u32(sA));
      const int T0 = static_cast<int>(t0), T1 = static_cast<int>(t1);
      int s = par;
      uint32_t sphase = 0;
      int t = T0 + par;       // next tile of this issuer
      int nswitch = 0;
      bool ok = true;
      GroupCursor cur;
      cur.seek(ws.groups, num_groups, T0);
      uint32_t bn = 0;        // batched walk: batches of the CTA's sequence so far
      for (int g = cur.g; ok && g < num_groups; ++g) {
        const int gbeg = ws.groups[g].tile_begin;
        if (gbeg >= T1) break;
        const int gend = g + 1 < num_groups ? ws.groups[g + 1].tile_begin : total_tiles;
        if (gend <= gbeg) continue;          // no tiles: its operand is never loaded
        if (!mbar_wait(&bars->bfull, nswitch & 1, limit, abort)) {
          ok = false;
          break;
        }
        ++nswitch;
        if constexpr (kBatched) {
          // Batch b (batch_tiles(rows) consecutive tiles of the group) accumulates
          // into slot b % 2, tile i of the batch at columns i x 64 x rows; both
          // issuers walk every batch, wait for its slot, issue their own tiles of it
          // (possibly none) and commit the slot, whose barrier counts both commits.
          const int nrows = ws.groups[g].nrows;
          const int bt = batch_tiles(nrows);
          const uint32_t idesc_b = umma_idesc(fmt, 64u * static_cast<uint32_t>(nrows));
          const int tbeg = gbeg > T0 ? gbeg : T0, tend = gend < T1 ? gend : T1;
          for (int bs = tbeg; ok && bs < tend; bs += bt, ++bn) {
            const uint32_t slot = bn % kSlots;
            if (!mbar_wait(&bars->tempty[slot], ((bn / kSlots) & 1u) ^ 1u, limit, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int be = bs + bt < tend ? bs + bt : tend;
            for (int tt = bs; tt < be; ++tt) {
              if (nis == 2 && ((tt - T0) & 1) != par) continue;   // the other issuer's tile
              if (!mbar_wait(&bars->full[s], sphase, limit, abort)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t d = tmem_base + slot * kSlotCols + static_cast<uint32_t>((tt - bs) * 64 * nrows);
              const uint64_t adesc = adesc0 + static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t koff = (kk & 3) * 32;
                const uint64_t bd = (kk < 4 ? bdesc0 : bdesc1) + (koff >> 4);
                if (KV == IDX_KV_E4M3) {
                  umma_f8(d, adesc + (koff >> 4), bd, idesc_b, kk > 0);
                } else {
                  umma_f16(d, adesc + (((kk < 4 ? 0u : static_cast<uint32_t>(kTileKeys) * 128u) + koff) >> 4), bd,
                           idesc_b, kk > 0);
                }
              }
              umma_commit(&bars->empty[s]);
              s += nis;
              if (s >= C::kStages) {
                s -= C::kStages;
                sphase ^= 1u;
              }
            }
            if (ok && !(a.stall_first_handoff && bn == 0)) umma_commit(&bars->tfull[slot]);
          }
          if (ok) umma_commit(&bars->bfree);
          continue;
        } else {
          (void)bn;
        }
        const uint32_t idesc = umma_idesc(fmt, 64u * static_cast<uint32_t>(ws.groups[g].nrows));
        const int tend = gend < T1 ? gend : T1;
        for (; t < tend; t += nis) {
          const int k = t - T0;
          const uint32_t slot = static_cast<uint32_t>(k) % kSlots;
          if (!mbar_wait(&bars->full[s], sphase, limit, abort) ||
              !mbar_wait(&bars->tempty[slot], ((static_cast<uint32_t>(k) / kSlots) & 1u) ^ 1u, limit, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + slot * kSlotCols;
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
              umma_f16(d, adesc + (((kk < 4 ? 0u : static_cast<uint32_t>(kTileKeys) * 128u) + koff) >> 4), bd,
                       idesc, kk > 0);
            }
          }
          umma_commit(&bars->empty[s]);
          if (!(a.stall_first_handoff && t == T0)) umma_commit(&bars->tfull[slot]);
          s += nis;
          if (s >= C::kStages) {
            s -= C::kStages;
            sphase ^= 1u;
          }
        }
        if (ok) umma_commit(&bars->bfree);   // this thread's MMAs of the group read the operand
      }
      if (!ok) set_abort(bars, ws.status);
      // All MMAs issued by this thread complete before TMEM is released.
      umma_commit(&bars->drain);
      int never = 0;
      if (!mbar_wait(&bars->drain, 0, limit, &never)) flag_status(ws.status, kStatusTimeout);
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ------------------------------------------------------------------ epilogue
    // Every epilogue warp takes every tile: the four warps of a TMEM lane quarter
    // reduce one row each, so a warp reduces the same row of every tile of a
    // group.  TMEM is read in the 16x256b shape: a thread sees four keys of its
    // quarter and a quarter of the row's heads, so it keeps just those heads'
    // weights in registers; the four threads that share keys add their partial
    // sums by shuffles, after which thread `lane` holds key kl of the quarter.
    // The tile's accumulator goes back to the MMA issuer right after the warp's
    // last TMEM read; in the plain walk each thread arrives on the slot barriers
    // itself (no warp sync before a lane-0 arrival).  Tile and key indices are
    // 32-bit (a launch has fewer than 2^31 of either).
    const int ew = warp - kEpiWarp0;
    const int quarter = warp & 3;            // TMEM lane quarter this warp may read
    const int row = ew >> 2;                 // group row this warp reduces
    const int kl = (lane >> 2) + 8 * (lane & 3);
    const int qk = quarter * 32 + kl;        // this thread's key within a tile
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(row * 64);
    uint32_t *hrow = shist + row * kHistWords;
    const float *sc = sscale + qk;
    const int T0 = static_cast<int>(t0), T1 = static_cast<int>(t1);
    GroupCursor cur;
    cur.seek(ws.groups, num_groups, T0);
    Group grp{};
    bool mine = false;
    int bnd = 0, gbegin = 0, next_fp = 0;
    float *srow = a.scores;
    float2 w2[8];          // halved weights of heads 8k + 2 (lane % 4) + {0, 1}, k = 0..7
    int flushes = 0;
    bool ok = true;

    // Every row's histogram goes to global memory (12-bit counts, the 64-bin first
    // digit, and the caller's copy of the latter when asked) and is cleared; all
    // sixteen warps meet before and after.  The group's nrows x 64 (row, first digit)
    // blocks of 64 bins are dealt to the warps, four per row at a time: the four
    // shared-memory reads go out together, and a block with no count (most of them:
    // a CTA's scores fill a few hundred of a row's 4096 bins) costs one vote.  A
    // block with counts is unpacked into one of the warp's staging slots and added
    // to the row's 12-bit histogram by one bulk reduction (the TMA engine performs
    // the 64 additions); its sum goes to the first digit by one atomic.  The counts
    // sit in a few first digits, the same ones in every row: scores of magnitude
    // near 1 fall in digits 15 and 16 (negative) and 47 and 48 (positive).  So warp
    // w takes the digits d of row r with d + 2 (d >> 5) + 4 r = w (mod 16):
    // consecutive digits of one sign go to consecutive warps, mirrored digits of the
    // two signs apart, and each row is shifted by four, which puts those sixteen
    // blocks on sixteen different warps.
    uint32_t *stage = sflush + ew * (kStageBlocks * 64);
    auto flush = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->hdone[0]);
      if (!mbar_wait(&bars->hdone[0], flushes & 1, limit, abort)) return false;
      int staged = 0;
      for (int hr = 0; hr < grp.nrows; ++hr) {
        const int x = (ew - 4 * hr) & 15, y = (ew - 4 * hr - 2) & 15;
        const int ds[4] = {x, x + 16, 32 + y, 48 + y};
        uint32_t wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wv[i] = shist[hr * kHistWords + ds[i] * 32 + lane];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (__ballot_sync(0xffffffffu, wv[i] != 0u) == 0u) continue;   // uniform for the warp
          const int d = ds[i];
          const int64_t grow = grp.row0 + hr;
          const uint32_t lo = wv[i] & 0xFFFFu, hi = wv[i] >> 16;
          if (staged >= kStageBlocks) {   // the slot's previous block must have been read
            if (lane == 0) bulk_wait_read<kStageBlocks - 1>();
            __syncwarp();
          }
          uint32_t *slot = stage + (staged % kStageBlocks) * 64;
          reinterpret_cast<uint2 *>(slot)[lane] = make_uint2(lo, hi);
          shist[hr * kHistWords + d * 32 + lane] = 0u;
          const uint32_t dsum = __reduce_add_sync(0xffffffffu, lo + hi);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            bulk_reduce_add_u32(&ws.hist12[grow * kHistBins + d * 64], slot, 256u);
            atomicAdd(&ws.hist64[grow * 64 + d], dsum);
            if (a.hist != nullptr) atomicAdd(&a.hist[grow * 64 + d], dsum);
          }
          ++staged;
        }
      }
      if (lane == 0 && staged > 0) bulk_wait_all();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->hflushed[0]);
      const bool r = mbar_wait(&bars->hflushed[0], flushes & 1, limit, abort);
      ++flushes;
      return r;
    };
    // A new group: whether it has this warp's row, that row's bound, score row and
    // weights.
    auto load_group = [&]() {
      grp = ws.groups[cur.g];
      mine = row < grp.nrows;
      const int r = grp.row0 + (mine ? row : 0);
      bnd = mine ? ws.bound_eff[r] : 0;
      gbegin = grp.tile_begin;
      srow = a.scores + static_cast<int64_t>(r) * a.ld;
      const float2 *wr = reinterpret_cast<const float2 *>(ws.wq + static_cast<int64_t>(r) * kHeads);
#pragma unroll
      for (int k = 0; k < 8; ++k) w2[k] = wr[4 * k + (lane & 3)];
    };
    // The histogram flush points: every group start and every kFlushTiles tiles
    // within a group (16-bit counters), on the CTA's tile sequence; every warp
    // takes each of them, in order, before the tile that starts there.
    auto set_next_fp = [&](int t) {
      const int periodic = gbegin + ((t - gbegin) / kFlushTiles + 1) * kFlushTiles;
      next_fp = periodic < cur.next_begin ? periodic : cur.next_begin;
    };
    if constexpr (kBatched) {
      // The batched walk: warp q of a TMEM lane quarter (q = 0..3) reduces one
      // (tile, row) of each batch: tile q with one row, row q % 2 of tile q / 2
      // with two, row q of the batch's one tile with three or four.  The histogram
      // goes to global memory before each group after the first, every
      // kFlushTiles tiles within a group and at the end; every warp takes each of
      // these points, in order.
      const int rq = ew >> 2;   // this warp's rank among its quarter's four
      const uint32_t tqb = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      int brow = 0, bi = 0, bt = 1;
      int cnt = 1;              // this warp's share of the kEpiWarps arrivals on a tile's scale slot
      uint32_t *bhrow = shist;
      uint32_t bn = 0;          // batches of the CTA's sequence so far
      bool first_group = true;
      for (int g = cur.g; ok && g < num_groups; ++g) {
        const int gbeg = ws.groups[g].tile_begin;
        if (gbeg >= T1) break;
        const int gend = g + 1 < num_groups ? ws.groups[g + 1].tile_begin : total_tiles;
        if (gend <= gbeg) continue;
        if (!first_group && !flush()) {
          ok = false;
          break;
        }
        first_group = false;
        grp = ws.groups[g];
        {
          const int n = grp.nrows;
          bt = batch_tiles(n);
          brow = n >= 3 ? rq : (n == 2 ? (rq & 1) : 0);
          bi = n >= 3 ? 0 : (n == 2 ? (rq >> 1) : rq);
          mine = brow < n;
          // readers of a tile per quarter: four (four rows), three (three: the first
          // arrives twice), two (two rows) or one (one row); four arrivals in all
          cnt = n == 4 ? 1 : n == 3 ? (brow == 0 ? 2 : 1) : n == 2 ? 2 : 4;
          const int r = grp.row0 + (mine ? brow : 0);
          bnd = mine ? ws.bound_eff[r] : 0;
          gbegin = grp.tile_begin;
          srow = a.scores + static_cast<int64_t>(r) * a.ld;
          bhrow = shist + brow * kHistWords;
          const float2 *wr = reinterpret_cast<const float2 *>(ws.wq + static_cast<int64_t>(r) * kHeads);
#pragma unroll
          for (int k = 0; k < 8; ++k) w2[k] = wr[4 * k + (lane & 3)];
        }
        const int tbeg = gbeg > T0 ? gbeg : T0, tend = gend < T1 ? gend : T1;
        int since = 0;   // tiles counted since the last flush
        for (int bs = tbeg; bs < tend; bs += bt, ++bn) {
          if (since + bt > kFlushTiles) {
            if (!flush()) {
              ok = false;
              break;
            }
            since = 0;
          }
          since += bt;
          const int t = bs + bi;
          const bool act = mine && t < tend && bi < bt;
          float scale = 1.0f;
          if (KV == IDX_KV_E4M3 && act) {
            const int k = t - T0;
            const int ss = k & (kScaleSlots - 1);
            if (!mbar_wait(&bars->sfull[ss], (k / kScaleSlots) & 1, limit, abort)) {
              set_abort(bars, ws.status);
              ok = false;
              break;
            }
            scale = sc[ss * kTileKeys];
            __syncwarp();
            if (lane == 0) mbar_arrive_cnt(&bars->sempty[ss], static_cast<uint32_t>(cnt));
          }
          const uint32_t slot = bn % kSlots;
          if (!mbar_wait(&bars->tfull[slot], (bn / kSlots) & 1u, limit, abort)) {
            set_abort(bars, ws.status);
            ok = false;
            break;
          }
          tc_fence_after();
          if (!act) {   // nothing of this batch for this warp: hand the accumulator back at once
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[slot]);
            continue;
          }
          const int pos = (t - gbegin) * kTileKeys + qk;
          const bool keep = pos < bnd;
          const uint32_t negmask = __ballot_sync(0xffffffffu, keep && scale < 0.0f);
          const uint32_t taddr = tqb + slot * kSlotCols + static_cast<uint32_t>((bi * grp.nrows + brow) * 64);
          float2 sums[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t va[16], vb[16];
            tmem_ld16x256_x4(taddr + half * 32, va);
            tmem_ld16x256_x4(taddr + (16u << 16) + half * 32, vb);
            tmem_wait_ld();
            reg_fence16(va);
            reg_fence16(vb);
            if (half == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->tempty[slot]);
            }
            if (negmask == 0u) relu_frag(va, vb, &w2[4 * half], sums);
            else relu_frag_signed(va, vb, &w2[4 * half], (negmask >> (lane & ~3)) & 15u, sums);
          }
          const float part[4] = {sums[0].x + sums[0].y, sums[1].x + sums[1].y, sums[2].x + sums[2].y,
                                 sums[3].x + sums[3].y};
          const float score = reduce_quad(part, lane) * scale;
          if (keep) {
            srow[pos] = score;
            const uint32_t bin = radix_key(score) >> (32 - kHistBits);
            atomicAdd(&bhrow[bin >> 1], 1u << ((bin & 1) * 16));
          }
        }
      }
      if (ok) flush();
    } else {
    load_group();
    set_next_fp(T0);

    for (int t = T0; t < T1; ++t) {
      if (t == next_fp) {
        if (!flush()) {
          ok = false;
          break;
        }
        if (t == cur.next_begin) {
          cur.advance(t);
          load_group();
        }
        set_next_fp(t);
      }
      const int k = t - T0;
      float scale = 1.0f;
      if (KV == IDX_KV_E4M3) {
        const int ss = k & (kScaleSlots - 1);
        if (!mbar_wait(&bars->sfull[ss], (k / kScaleSlots) & 1, limit, abort)) {
          set_abort(bars, ws.status);
          ok = false;
          break;
        }
        scale = sc[ss * kTileKeys];
        mbar_arrive(&bars->sempty[ss]);
      }
      const int slot = k & (kSlots - 1);
      if (!mbar_wait(&bars->tfull[slot], (k / kSlots) & 1, limit, abort)) {
        set_abort(bars, ws.status);
        ok = false;
        break;
      }
      tc_fence_after();
      if (!mine) {   // the group has no row for this warp: hand the accumulator back at once
        tc_fence_before();
        mbar_arrive(&bars->tempty[slot]);
        continue;
      }
      const int pos = (t - gbegin) * kTileKeys + qk;
      const bool keep = pos < bnd;   // below the row's bound (so also below the group's L)
      // bit (4g + m) set: key m of threads 4g .. 4g+3 (quarter lane g + 8m) has a negative scale
      const uint32_t negmask = __ballot_sync(0xffffffffu, keep && scale < 0.0f);
      const uint32_t taddr = tq + static_cast<uint32_t>(slot * kSlotCols);
      float2 sums[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t va[16], vb[16];
        tmem_ld16x256_x4(taddr + half * 32, va);
        tmem_ld16x256_x4(taddr + (16u << 16) + half * 32, vb);
        tmem_wait_ld();
        reg_fence16(va);
        reg_fence16(vb);
        if (half == 1) {   // every read of this thread is done: hand the accumulator back
          tc_fence_before();
          mbar_arrive(&bars->tempty[slot]);
        }
        if (negmask == 0u) relu_frag(va, vb, &w2[4 * half], sums);
        else relu_frag_signed(va, vb, &w2[4 * half], (negmask >> (lane & ~3)) & 15u, sums);
      }
      const float part[4] = {sums[0].x + sums[0].y, sums[1].x + sums[1].y, sums[2].x + sums[2].y,
                             sums[3].x + sums[3].y};
      const float score = reduce_quad(part, lane) * scale;
      if (keep) {
        srow[pos] = score;
        const uint32_t bin = radix_key(score) >> (32 - kHistBits);
        atomicAdd(&hrow[bin >> 1], 1u << ((bin & 1) * 16));   // shared-memory atomics resolve collisions
      }
    }
    if (ok) flush();
    }
  }

  // Every role is done (or gave up); release TMEM.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int KV, bool kBatched>
cudaError_t launch_kv(const CUtensorMap &kmap, const ScoreArgs &a, int num_ctas, cudaStream_t stream) {
  static std::mutex mu;
  static bool done[128] = {};
  constexpr int bytes = Smem<KV>::kDynamic;
  const cudaError_t e = once_per_device(mu, done, [] {
    return cudaFuncSetAttribute(score_kernel<KV, kBatched>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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
  return cudaLaunchKernelEx(&cfg, score_kernel<KV, kBatched>, kmap, a);
}

}  // namespace

cudaError_t launch_score(const CUtensorMap &kmap, const ScoreArgs &a, int kv_dtype, bool batched, int num_ctas,
                         cudaStream_t stream) {
  if (kv_dtype == IDX_KV_E4M3) {
    return batched ? launch_kv<IDX_KV_E4M3, true>(kmap, a, num_ctas, stream)
                   : launch_kv<IDX_KV_E4M3, false>(kmap, a, num_ctas, stream);
  }
  return batched ? launch_kv<IDX_KV_BF16, true>(kmap, a, num_ctas, stream)
                 : launch_kv<IDX_KV_BF16, false>(kmap, a, num_ctas, stream);
}

}  // namespace idx
