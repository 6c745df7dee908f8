// The C ABI (include/idx.h): argument checks, workspace carving, the key
// cache's TMA descriptor, and the order of launches on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <climits>
#include <mutex>
#include <vector>

#include "idx.h"
#include "idx_device.cuh"
#include "launch.h"

namespace {

using idx::Workspace;

constexpr size_t kAlign = 1024;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t g_wait_limit_ns = 1000000000LL;
int64_t g_stall_next = 0;
cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;
std::mutex g_mu;

uint64_t wait_limit() {
  std::lock_guard<std::mutex> lk(g_mu);
  return static_cast<uint64_t>(g_wait_limit_ns);
}

struct Layout {
  size_t status, plan, groups, bound_eff, qop0, qop1, wq, hist12, hist64, hist_sub, rowsel, win, tie, scores;
  size_t total;
  int64_t scores_ld;
};

Layout make_layout(int64_t R, int64_t K, int64_t max_bound, bool with_scores) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kAlign);
    return at;
  };
  L.status = take(256);
  L.plan = take(sizeof(idx::PlanHeader));
  L.groups = take(static_cast<size_t>(R) * sizeof(idx::Group));
  L.bound_eff = take(static_cast<size_t>(R) * 4);
  L.qop0 = take(static_cast<size_t>(R) * idx::kRowOperandBytes);
  L.qop1 = take(static_cast<size_t>(R) * idx::kRowOperandBytes);
  L.wq = take(static_cast<size_t>(R) * idx::kHeads * 4);
  L.hist12 = take(static_cast<size_t>(R) * idx::kHistBins * 4);
  L.hist64 = take(static_cast<size_t>(R) * 64 * 4);
  L.hist_sub = take(static_cast<size_t>(R) * idx::kSubBins * 4);
  L.rowsel = take(static_cast<size_t>(R) * sizeof(idx::RowSelect));
  L.win = take(static_cast<size_t>(R) * K * 8);
  L.tie = take(static_cast<size_t>(R) * idx::kTieCap * 8);
  L.scores_ld = static_cast<int64_t>(align_up(static_cast<size_t>(max_bound > 0 ? max_bound : 1), 4));
  L.scores = take(with_scores ? static_cast<size_t>(R) * L.scores_ld * 4 : 0);
  L.total = off;
  return L;
}

Workspace carve(void *base, const Layout &L) {
  uint8_t *b = static_cast<uint8_t *>(base);
  Workspace w{};
  w.status = reinterpret_cast<uint32_t *>(b + L.status);
  w.plan = reinterpret_cast<idx::PlanHeader *>(b + L.plan);
  w.groups = reinterpret_cast<idx::Group *>(b + L.groups);
  w.bound_eff = reinterpret_cast<int32_t *>(b + L.bound_eff);
  w.qop0 = b + L.qop0;
  w.qop1 = b + L.qop1;
  w.wq = reinterpret_cast<float *>(b + L.wq);
  w.hist12 = reinterpret_cast<uint32_t *>(b + L.hist12);
  w.hist64 = reinterpret_cast<uint32_t *>(b + L.hist64);
  w.hist_sub = reinterpret_cast<uint32_t *>(b + L.hist_sub);
  w.rowsel = reinterpret_cast<idx::RowSelect *>(b + L.rowsel);
  w.win = reinterpret_cast<unsigned long long *>(b + L.win);
  w.tie = reinterpret_cast<unsigned long long *>(b + L.tie);
  w.scores = reinterpret_cast<float *>(b + L.scores);
  w.scores_ld = L.scores_ld;
  return w;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

idx_status check_problem(const idx_problem *p) {
  if (p == nullptr) return IDX_EINVAL;
  if (p->q == nullptr || p->w == nullptr || p->k_cache == nullptr || p->page_table == nullptr ||
      p->row_req == nullptr || p->row_bound == nullptr)
    return IDX_EINVAL;
  if (p->R < 1 || p->Q < 1 || p->P < 1 || p->pt_stride < 1 || p->max_bound < 0 || p->rows_hint < 0)
    return IDX_EINVAL;
  if (p->R > IDX_MAX_ROWS) return IDX_EUNSUPPORTED;
  if (static_cast<int64_t>(p->max_bound) > static_cast<int64_t>(p->pt_stride) * IDX_PAGE) return IDX_EINVAL;
  if (p->P > (INT32_MAX / IDX_PAGE)) return IDX_EUNSUPPORTED;  // TMA row coordinate is 32-bit
  if (p->kv_dtype == IDX_KV_E4M3) {
    if (p->k_scale == nullptr || !aligned16(p->k_scale)) return IDX_EINVAL;
  } else if (p->kv_dtype == IDX_KV_BF16) {
    if (p->k_scale != nullptr) return IDX_EINVAL;
  } else {
    return IDX_EINVAL;
  }
  if (!aligned16(p->q) || !aligned16(p->w) || !aligned16(p->k_cache)) return IDX_EINVAL;
  return IDX_OK;
}

// ---------------------------------------------------------------------------- device info
std::atomic<int> g_num_sms[128];   // filled on first use per device (concurrent callers store the same value)

idx_status device_sms(int *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ECUDA;
  if (dev < 0 || dev >= 128) return IDX_EUNSUPPORTED;
  if (g_num_sms[dev].load(std::memory_order_relaxed) == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return IDX_ECUDA;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return IDX_EUNSUPPORTED;  // built for sm_103a only
    g_num_sms[dev].store(n, std::memory_order_relaxed);
  }
  *out = g_num_sms[dev].load(std::memory_order_relaxed);
  return IDX_OK;
}

// ---------------------------------------------------------------------------- TMA descriptor
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

idx_status key_tensor_map(const idx_problem *p, CUtensorMap *map) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return IDX_ECUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const bool f8 = p->kv_dtype == IDX_KV_E4M3;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(IDX_DIM), static_cast<cuuint64_t>(p->P) * IDX_PAGE};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(f8 ? IDX_DIM : IDX_DIM * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(f8 ? 128 : 64), static_cast<cuuint32_t>(IDX_PAGE)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void *>(p->k_cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IDX_OK : IDX_ECUDA;
}

idx_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? IDX_OK : IDX_ECUDA; }

// prep + scoring launches shared by idx_score and idx_launch.
// The new-key writes of a problem's rows (k_new: bf16 [R][128], device).
idx::PatchArgs make_patch(const idx_problem *problem, const void *k_new) {
  idx::PatchArgs pa{};
  pa.k_new = static_cast<const uint16_t *>(k_new);
  pa.row_req = problem->row_req;
  pa.row_bound = problem->row_bound;
  pa.page_table = problem->page_table;
  pa.k_cache = const_cast<void *>(problem->k_cache);
  pa.k_scale = const_cast<float *>(problem->k_scale);
  pa.R = problem->R;
  pa.Q = problem->Q;
  pa.pt_stride = problem->pt_stride;
  pa.kv_dtype = problem->kv_dtype;
  pa.P = problem->P;
  return pa;
}

idx_status run_scoring(const idx_problem *p, const Workspace &w, float *scores, int64_t ld, uint32_t *hist,
                       bool clear_select, const void *k_new, cudaStream_t s) {
  int sms = 0;
  idx_status st = device_sms(&sms);
  if (st != IDX_OK) return st;
  CUtensorMap map;
  st = key_tensor_map(p, &map);
  if (st != IDX_OK) return st;
  idx::PrepArgs pa{};
  pa.q = p->q;
  pa.w = p->w;
  pa.row_req = p->row_req;
  pa.row_bound = p->row_bound;
  pa.R = p->R;
  pa.Q = p->Q;
  pa.pt_stride = p->pt_stride;
  pa.max_bound = p->max_bound;
  pa.kv_dtype = p->kv_dtype;
  pa.hist_target = hist;
  pa.clear_select = clear_select ? 1 : 0;
  pa.ws = w;
  if (k_new != nullptr) pa.patch = make_patch(p, k_new);
  st = cuda_ok(idx::launch_prep(pa, s));
  if (st != IDX_OK) return st;
  idx::ScoreArgs sa{};
  sa.page_table = p->page_table;
  sa.k_scale = p->k_scale;
  sa.P = p->P;
  sa.pt_stride = p->pt_stride;
  sa.scores = scores;
  sa.ld = ld;
  sa.hist = hist;
  sa.ws = w;
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    sa.wait_limit_ns = static_cast<uint64_t>(g_wait_limit_ns);
    sa.stall_first_handoff = g_stall_next > 0 ? 1 : 0;
    if (g_stall_next > 0) --g_stall_next;
    ev0 = g_prof_start;
    ev1 = g_prof_stop;
    g_prof_start = g_prof_stop = nullptr;
  }
  if (ev0 != nullptr && cudaEventRecord(ev0, s) != cudaSuccess) return IDX_ECUDA;
  st = cuda_ok(idx::launch_score(map, sa, p->kv_dtype, p->rows_hint == 1 || p->rows_hint == 2, sms, s));
  if (st != IDX_OK) return st;
  if (ev1 != nullptr && cudaEventRecord(ev1, s) != cudaSuccess) return IDX_ECUDA;
  return IDX_OK;
}


// Scratch of idx_topk_noalloc: a file-scope device array, so that the call takes
// no workspace from the caller and allocates nothing.  Its address is looked up
// once per device; the workspace starts at the first 1024-byte boundary inside
// it (the loaded module guarantees a smaller alignment only), so up to
// IDX_NOALLOC_SCRATCH_BYTES - 1023 bytes are usable.
__device__ __align__(256) unsigned char g_noalloc_scratch[IDX_NOALLOC_SCRATCH_BYTES];
std::mutex g_noalloc_mu;
void *g_noalloc_base[128] = {};

}  // namespace

extern "C" {

size_t idx_workspace_size(const idx_problem *problem, int32_t K) {
  if (check_problem(problem) != IDX_OK || K < 1 || K > IDX_MAX_K) return 0;
  return make_layout(problem->R, K, problem->max_bound, true).total;
}

idx_status idx_score(const idx_problem *problem, float *scores, int64_t ld, uint32_t *hist, void *ws,
                     size_t ws_bytes, void *stream) {
  idx_status st = check_problem(problem);
  if (st != IDX_OK) return st;
  if (scores == nullptr || ws == nullptr || ld < 1 || ld < problem->max_bound) return IDX_EINVAL;
  const Layout L = make_layout(problem->R, 1, problem->max_bound, false);
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return IDX_EINVAL;
  const Workspace w = carve(ws, L);
  return run_scoring(problem, w, scores, ld, hist, false, nullptr, static_cast<cudaStream_t>(stream));
}

idx_status idx_topk(const float *scores, int64_t ld, const int32_t *row_bound, int32_t R, int32_t max_bound,
                    int32_t K, const uint32_t *hist, int32_t *out_idx, void *ws, size_t ws_bytes, void *stream) {
  if (scores == nullptr || row_bound == nullptr || out_idx == nullptr || ws == nullptr) return IDX_EINVAL;
  if (R < 1 || max_bound < 0 || K < 1 || K > IDX_MAX_K || ld < 1 || ld < max_bound) return IDX_EINVAL;
  if (R > IDX_MAX_ROWS) return IDX_EUNSUPPORTED;
  const Layout L = make_layout(R, K, max_bound, false);
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return IDX_EINVAL;
  int sms = 0;
  idx_status st = device_sms(&sms);
  if (st != IDX_OK) return st;
  const Workspace w = carve(ws, L);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = cuda_ok(cudaMemsetAsync(w.status, 0, 4, s));
  if (st != IDX_OK) return st;
  idx::SelectArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.bound = w.bound_eff;
  a.R = R;
  a.K = K;
  a.max_bound = max_bound;
  a.out_idx = out_idx;
  a.ws = w;
  a.bulk_rows = (reinterpret_cast<uintptr_t>(scores) & 15u) == 0 && ld % 4 == 0;
  a.wait_limit_ns = wait_limit();
  a.num_sms = sms;
  st = cuda_ok(idx::launch_select_clear(a, row_bound, s));
  if (st != IDX_OK) return st;
  st = cuda_ok(idx::launch_hist12(a, s));
  if (st != IDX_OK) return st;
  return cuda_ok(idx::launch_collect(a, s));
}

namespace {
idx_status launch_impl(const idx_problem *problem, const void *k_new, int32_t K, int32_t *out_idx, float *out_score,
                       void *ws, size_t ws_bytes, void *stream) {
  idx_status st = check_problem(problem);
  if (st != IDX_OK) return st;
  if (out_idx == nullptr || ws == nullptr || K < 1 || K > IDX_MAX_K) return IDX_EINVAL;
  const Layout L = make_layout(problem->R, K, problem->max_bound, true);
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return IDX_EINVAL;
  const Workspace w = carve(ws, L);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = run_scoring(problem, w, w.scores, w.scores_ld, nullptr, true, k_new, s);
  if (st != IDX_OK) return st;
  idx::SelectArgs a{};
  a.scores = w.scores;
  a.ld = w.scores_ld;
  a.bound = w.bound_eff;
  a.R = problem->R;
  a.K = K;
  a.max_bound = problem->max_bound;
  a.out_idx = out_idx;
  a.out_score = out_score;
  a.ws = w;
  a.bulk_rows = (reinterpret_cast<uintptr_t>(w.scores) & 15u) == 0 && w.scores_ld % 4 == 0;
  a.wait_limit_ns = wait_limit();
  int sms = 0;
  st = device_sms(&sms);
  if (st != IDX_OK) return st;
  a.num_sms = sms;
  return cuda_ok(idx::launch_collect(a, s));
}
}  // namespace

idx_status idx_launch(const idx_problem *problem, int32_t K, int32_t *out_idx, void *ws, size_t ws_bytes,
                      void *stream) {
  return launch_impl(problem, nullptr, K, out_idx, nullptr, ws, ws_bytes, stream);
}

idx_status idx_launch_new_keys(const idx_problem *problem, const void *k_new, int32_t K, int32_t *out_idx, void *ws,
                               size_t ws_bytes, void *stream) {
  if (k_new == nullptr || (reinterpret_cast<uintptr_t>(k_new) & 15u) != 0) return IDX_EINVAL;
  return launch_impl(problem, k_new, K, out_idx, nullptr, ws, ws_bytes, stream);
}

idx_status idx_launch_scored(const idx_problem *problem, int32_t K, int32_t *out_idx, float *out_score, void *ws,
                             size_t ws_bytes, void *stream) {
  if (out_score == nullptr) return IDX_EINVAL;
  return launch_impl(problem, nullptr, K, out_idx, out_score, ws, ws_bytes, stream);
}

idx_status idx_merge_topk(const int32_t *part_idx, const float *part_score, const int32_t *part_offset,
                          int32_t S, int32_t R, int32_t Kin, int32_t K, int32_t *out_idx, float *out_score,
                          void *stream) {
  if (part_idx == nullptr || part_score == nullptr || part_offset == nullptr || out_idx == nullptr)
    return IDX_EINVAL;
  if (S < 1 || R < 1 || Kin < 1 || K < 1 || K > IDX_MAX_K || Kin > IDX_MAX_K) return IDX_EINVAL;
  if (S > IDX_MERGE_MAX_PARTS || R > IDX_MAX_ROWS) return IDX_EUNSUPPORTED;
  if (idx::merge_smem_bytes(S, Kin, K) > idx::merge_smem_bytes(IDX_MERGE_MAX_PARTS, IDX_MAX_K, IDX_MAX_K))
    return IDX_EUNSUPPORTED;
  idx::MergeArgs m{};
  for (int s = 0; s < S; ++s) {
    if (part_offset[s] < 0) return IDX_EINVAL;
    m.offset[s] = part_offset[s];
  }
  m.part_idx = part_idx;
  m.part_score = part_score;
  m.S = S;
  m.R = R;
  m.Kin = Kin;
  m.K = K;
  m.out_idx = out_idx;
  m.out_score = out_score;
  return cuda_ok(idx::launch_merge(m, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------- host inputs
namespace {
struct HostArena {
  size_t q, w, kc, ks, pt, rr, rb, out, ws, total;
};

HostArena host_arena(const idx_problem *p, int32_t K) {
  HostArena A{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kAlign);
    return at;
  };
  const size_t key_bytes = static_cast<size_t>(p->P) * IDX_PAGE * IDX_DIM * (p->kv_dtype == IDX_KV_E4M3 ? 1 : 2);
  A.q = take(static_cast<size_t>(p->R) * IDX_HEADS * IDX_DIM * 2);
  A.w = take(static_cast<size_t>(p->R) * IDX_HEADS * 4);
  A.kc = take(key_bytes);
  A.ks = take(p->kv_dtype == IDX_KV_E4M3 ? static_cast<size_t>(p->P) * IDX_PAGE * 4 : 0);
  A.pt = take(static_cast<size_t>(p->Q) * p->pt_stride * 4);
  A.rr = take(static_cast<size_t>(p->R) * 4);
  A.rb = take(static_cast<size_t>(p->R) * 4);
  A.out = take(static_cast<size_t>(p->R) * K * 4);
  A.ws = take(make_layout(p->R, K, p->max_bound, true).total);
  A.total = off;
  return A;
}
}  // namespace

size_t idx_host_arena_size(const idx_problem *host_problem, int32_t K) {
  if (check_problem(host_problem) != IDX_OK || K < 1 || K > IDX_MAX_K) return 0;
  return host_arena(host_problem, K).total;
}

idx_status idx_launch_host(const idx_problem *hp, int32_t K, int32_t *host_out, void *arena, size_t arena_bytes,
                           void *stream) {
  idx_status st = check_problem(hp);
  if (st != IDX_OK) return st;
  if (host_out == nullptr || arena == nullptr || K < 1 || K > IDX_MAX_K) return IDX_EINVAL;
  const HostArena A = host_arena(hp, K);
  if (arena_bytes < A.total || (reinterpret_cast<uintptr_t>(arena) & (kAlign - 1)) != 0) return IDX_EINVAL;
  uint8_t *b = static_cast<uint8_t *>(arena);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f8 = hp->kv_dtype == IDX_KV_E4M3;
  struct Copy {
    size_t off;
    const void *src;
    size_t bytes;
  } copies[] = {
      {A.q, hp->q, static_cast<size_t>(hp->R) * IDX_HEADS * IDX_DIM * 2},
      {A.w, hp->w, static_cast<size_t>(hp->R) * IDX_HEADS * 4},
      {A.kc, hp->k_cache, static_cast<size_t>(hp->P) * IDX_PAGE * IDX_DIM * (f8 ? 1 : 2)},
      {A.ks, hp->k_scale, f8 ? static_cast<size_t>(hp->P) * IDX_PAGE * 4 : 0},
      {A.pt, hp->page_table, static_cast<size_t>(hp->Q) * hp->pt_stride * 4},
      {A.rr, hp->row_req, static_cast<size_t>(hp->R) * 4},
      {A.rb, hp->row_bound, static_cast<size_t>(hp->R) * 4},
  };
  for (const Copy &c : copies) {
    if (c.bytes == 0) continue;
    st = cuda_ok(cudaMemcpyAsync(b + c.off, c.src, c.bytes, cudaMemcpyHostToDevice, s));
    if (st != IDX_OK) return st;
  }
  idx_problem dp = *hp;
  if (dp.rows_hint == 0) {   // the row map is host memory here: count each request's rows
    std::vector<int32_t> rows(static_cast<size_t>(hp->Q), 0);
    int32_t most = 0;
    for (int32_t r = 0; r < hp->R; ++r) {
      const int32_t q = hp->row_req[r];
      if (q >= 0 && q < hp->Q) most = std::max(most, ++rows[static_cast<size_t>(q)]);
    }
    dp.rows_hint = most;
  }
  dp.q = b + A.q;
  dp.w = reinterpret_cast<const float *>(b + A.w);
  dp.k_cache = b + A.kc;
  dp.k_scale = f8 ? reinterpret_cast<const float *>(b + A.ks) : nullptr;
  dp.page_table = reinterpret_cast<const int32_t *>(b + A.pt);
  dp.row_req = reinterpret_cast<const int32_t *>(b + A.rr);
  dp.row_bound = reinterpret_cast<const int32_t *>(b + A.rb);
  int32_t *dout = reinterpret_cast<int32_t *>(b + A.out);
  st = idx_launch(&dp, K, dout, b + A.ws, A.total - A.ws, stream);
  if (st != IDX_OK) return st;
  return cuda_ok(cudaMemcpyAsync(host_out, dout, static_cast<size_t>(hp->R) * K * 4, cudaMemcpyDeviceToHost, s));
}

idx_status idx_last_device_status(void *ws, void *stream) {
  if (ws == nullptr) return IDX_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return IDX_ECUDA;
  uint32_t word = 0;
  uint32_t *status = static_cast<uint32_t *>(ws);  // the status word is the workspace's first word
  if (cudaMemcpy(&word, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return IDX_ECUDA;
  if (cudaMemset(status, 0, 4) != cudaSuccess) return IDX_ECUDA;
  if (word & idx::kStatusTimeout) return IDX_ETIMEOUT;
  if (word & (idx::kStatusBadPage | idx::kStatusBadBound)) return IDX_EDEVICE;
  return IDX_OK;
}

const char *idx_status_string(idx_status status) {
  switch (status) {
    case IDX_OK: return "ok";
    case IDX_EINVAL: return "invalid argument";
    case IDX_EUNSUPPORTED: return "unsupported shape or device";
    case IDX_ECUDA: return "CUDA error";
    case IDX_ETIMEOUT: return "a device-side wait ran out of time";
    case IDX_EDEVICE: return "out-of-range page id or row bound seen on the device";
  }
  return "unknown status";
}

int32_t idx_version(void) { return 100; }

void idx_profile_events(void *start, void *stop) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof_start = static_cast<cudaEvent_t>(start);
  g_prof_stop = static_cast<cudaEvent_t>(stop);
}

int64_t idx_debug_set(int32_t what, int64_t value) {
  std::lock_guard<std::mutex> lk(g_mu);
  int64_t prev = 0;
  if (what == IDX_DEBUG_WAIT_LIMIT_NS) {
    prev = g_wait_limit_ns;
    g_wait_limit_ns = value > 0 ? value : 1000000000LL;
  } else if (what == IDX_DEBUG_STALL_SCORE_MMA) {
    prev = g_stall_next;
    g_stall_next = value > 0 ? value : 0;
  }
  return prev;
}

idx_status idx_patch_new_keys(const idx_problem *problem, const void *k_new, void *stream) {
  idx_status st = check_problem(problem);
  if (st != IDX_OK) return st;
  if (k_new == nullptr || (reinterpret_cast<uintptr_t>(k_new) & 15u) != 0) return IDX_EINVAL;
  return cuda_ok(idx::launch_patch(make_patch(problem, k_new), static_cast<cudaStream_t>(stream)));
}

size_t idx_top1_state_size(int32_t R) {
  return R < 1 ? 0 : static_cast<size_t>(R) * sizeof(idx::Top1State);
}

idx_status idx_top1(const float *logits, int64_t ld, int32_t R, int64_t V, int32_t *out_idx, float *out_val,
                    int32_t *tokens, int64_t tokens_ld, int32_t token_col, int32_t *positions, void *state,
                    size_t state_bytes, void *stream) {
  if (logits == nullptr || out_idx == nullptr || state == nullptr) return IDX_EINVAL;
  if (R < 1 || V < 1 || ld < V) return IDX_EINVAL;
  if (V > INT32_MAX || R > IDX_MAX_ROWS) return IDX_EUNSUPPORTED;
  if (tokens != nullptr && (tokens_ld < 1 || token_col < 0 || token_col >= tokens_ld)) return IDX_EINVAL;
  if (state_bytes < idx_top1_state_size(R) || (reinterpret_cast<uintptr_t>(state) & 15u) != 0) return IDX_EINVAL;
  int sms = 0;
  idx_status st = device_sms(&sms);
  if (st != IDX_OK) return st;
  idx::Top1Args t{};
  t.logits = logits;
  t.ld = ld;
  t.V = V;
  t.R = R;
  t.out_idx = out_idx;
  t.out_val = out_val;
  t.tokens = tokens;
  t.tokens_ld = tokens_ld;
  t.token_col = token_col;
  t.positions = positions;
  t.state = static_cast<idx::Top1State *>(state);
  t.vec4 = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && ld % 4 == 0;
  return cuda_ok(idx::launch_top1(t, sms, static_cast<cudaStream_t>(stream)));
}

idx_status idx_topk_noalloc(const float *scores, int64_t ld, const int32_t *row_bound, int32_t R,
                            int32_t max_bound, int32_t K, int32_t *out_idx, void *stream) {
  if (R > IDX_NOALLOC_MAX_ROWS) return IDX_EUNSUPPORTED;
  if (R < 1 || K < 1 || K > IDX_MAX_K || max_bound < 0) return IDX_EINVAL;
  const Layout L = make_layout(R, K, max_bound, false);
  if (L.total > IDX_NOALLOC_SCRATCH_BYTES - (kAlign - 1)) return IDX_EUNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ECUDA;
  if (dev < 0 || dev >= 128) return IDX_EUNSUPPORTED;
  void *base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_base[dev] == nullptr) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return IDX_ECUDA;
      g_noalloc_base[dev] = p;
    }
    base = g_noalloc_base[dev];
  }
  const uintptr_t raw = reinterpret_cast<uintptr_t>(base);
  const uintptr_t aligned = (raw + kAlign - 1) & ~static_cast<uintptr_t>(kAlign - 1);
  return idx_topk(scores, ld, row_bound, R, max_bound, K, nullptr, out_idx, reinterpret_cast<void *>(aligned),
                  IDX_NOALLOC_SCRATCH_BYTES - (aligned - raw), stream);
}

}  // extern "C"
