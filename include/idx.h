/*
 * idx.h - C ABI of the GB300 decode indexer library (libidx.so).
 *
 * The indexer of the sglang PR 48224 page (sgl-amd-mono #86): every decode row is
 * scored against every key its request has cached, and the row's exact top-2048
 * is selected (section Motivation, first paragraph).  It reads an FP8 E4M3 or
 * bf16 paged key cache (section Accuracy Tests), leaves out positions from a
 * row's bound on (section Modifications, commit 2), and selects by radix digits whose first digit is radix_key >> 26
 * over 64 bins (section Modifications, commit 4).  The score of the key at
 * logical position t for row r is
 *
 *     score[r][t] = sum_{h<64} w[r][h] * ReLU(scale_t * <q[r][h][:], k_t>)
 *
 * with 64 heads of 128 dimensions; scale_t is the key's fp32 scale (E4M3 cache)
 * or 1 (bf16 cache).
 *
 * Conventions for every call below:
 *   - Pointers named "device" are caller-owned device memory; the library never
 *     allocates, frees or keeps them.  Pointers named "host" are host memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     is asynchronous on it unless its comment says otherwise.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns IDX_EINVAL (or IDX_EUNSUPPORTED for a shape the library
 *     does not handle) and launches nothing.  A failed launch returns IDX_ECUDA.
 *   - Errors found on the device (a page id outside [0, P), a row bound above
 *     max_bound or pt_stride * 64, a request id outside [0, Q), a pipeline wait
 *     that ran out of time) never trap: the kernel records them in a status word
 *     inside the workspace, clamps the bound or skips the page or the row, and
 *     finishes; read the word with idx_last_device_status().
 *   - Key positions are logical positions within the row's request: position t
 *     lives in physical page page_table[req * pt_stride + t / 64], slot t % 64.
 *   - Host threads: any call may be made from several host threads at once, on
 *     the same or different devices, as long as concurrent calls use different
 *     workspaces (the library's one-time per-device setup is serialised inside
 *     it).  idx_topk_noalloc is the exception: its scratch is one per device.
 *     idx_debug_set and idx_profile_events change process-wide state that the
 *     next call from any thread picks up.
 */
#ifndef IDX_H
#define IDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IDX_HEADS 64      /* query heads per row */
#define IDX_DIM 128       /* dimensions per head and per key */
#define IDX_PAGE 64       /* tokens per cache page */
#define IDX_MAX_K 2048    /* largest top-k */
#define IDX_MAX_ROWS 65535

typedef enum {
    IDX_OK = 0,
    IDX_EINVAL = 1,       /* bad argument (null pointer, negative size, small workspace ...) */
    IDX_EUNSUPPORTED = 2, /* valid but outside what this build handles */
    IDX_ECUDA = 3,        /* a CUDA runtime call or launch failed */
    IDX_ETIMEOUT = 4,     /* a device-side wait ran out of time (device status only) */
    IDX_EDEVICE = 5       /* bad data seen on the device: page id, bound or request id out of range */
} idx_status;

typedef enum {
    IDX_KV_E4M3 = 0,      /* keys are OCP E4M3 bytes with one fp32 scale per token */
    IDX_KV_BF16 = 1       /* keys are bf16, scale 1 */
} idx_kv_dtype;

/* One indexer problem.  All array pointers are device memory owned by the caller. */
typedef struct {
    const void *q;             /* bf16 [R][64][128], contiguous, 16-byte aligned */
    const float *w;            /* fp32 [R][64], contiguous, 16-byte aligned */
    const void *k_cache;       /* [P][64][128]: E4M3 bytes or bf16, contiguous, 16-byte aligned */
    const float *k_scale;      /* fp32 [P][64] for IDX_KV_E4M3, 16-byte aligned, every value >= 0;
                                  must be NULL for IDX_KV_BF16 */
    const int32_t *page_table; /* int32 [Q][pt_stride]: page ids in [0, P) for every page a row reads */
    const int32_t *row_req;    /* int32 [R]: request of each row, in [0, Q) */
    const int32_t *row_bound;  /* int32 [R]: row r scores positions 0 .. row_bound[r]-1 */
    int32_t R;                 /* rows, 1 .. IDX_MAX_ROWS */
    int32_t Q;                 /* requests, >= 1 */
    int64_t P;                 /* pages in the cache, >= 1 */
    int32_t pt_stride;         /* page-table row length, >= 1 */
    int32_t max_bound;         /* host upper bound on every row_bound[r]; sizes scratch, so no
                                  device-to-host read is needed; 0 <= max_bound <= pt_stride*64 */
    int32_t kv_dtype;          /* idx_kv_dtype */
    int32_t rows_hint;         /* host hint, like max_bound: 0 if unknown, else an upper bound on the
                                  rows of any one request in this problem.  1 or 2 (a lone live row,
                                  or a row and its pad row) lets the scan batch 4 / rows tiles into
                                  one accumulator so that every epilogue warp has work.  The result
                                  never depends on it: a hint below the true count only costs
                                  speed.  Negative: IDX_EINVAL. */
} idx_problem;

/* Bytes of device workspace that idx_score / idx_topk / idx_launch need for this
 * problem and top-k (the largest of the three; every call accepts more).  The
 * workspace is caller-owned, needs no initialisation and may be reused by later
 * calls on the same stream; two calls that overlap in time need two workspaces.
 * Returns 0 if the problem is invalid. */
size_t idx_workspace_size(const idx_problem *problem, int32_t K);

/* Scores only (the scan and contraction; section Motivation, first paragraph).
 *   scores  device fp32 [R][ld], ld >= max_bound: scores[r][t] written for t < row_bound[r],
 *           other entries untouched.
 *   hist    device uint32 [R][64] or NULL: when given, hist[r][d] = number of t < row_bound[r]
 *           with radix_key(scores[r][t]) >> 26 == d (the fused first-digit histogram of
 *           section Modifications, commit 4).  radix_key maps the fp32 bits to an unsigned key
 *           that orders like the value, with -0.0 read as +0.0.
 *   ws      device workspace of ws_bytes >= idx_workspace_size(problem, 1). */
idx_status idx_score(const idx_problem *problem, float *scores, int64_t ld, uint32_t *hist,
                     void *ws, size_t ws_bytes, void *stream);

/* Exact top-K of given scores (section Motivation: exact top-2048; section
 * Modifications, commit 4: radix selection with a 64-bin first digit).
 *   scores     device fp32 [R][ld]; only t < row_bound[r] is read; values must not be NaN.
 *   row_bound  device int32 [R]; max_bound (host) >= every row_bound[r], ld >= max_bound.
 *   K          1 .. IDX_MAX_K.
 *   hist       device uint32 [R][64] first-digit histogram of these scores (as idx_score
 *              writes it) or NULL.  Accepted for callers that hold one; this build
 *              counts the finer 12-bit prefix of the radix keys in one pass over the
 *              scores and does not need it.
 *   out_idx    device int32 [R][K]: positions ordered by score descending, then position
 *              ascending; entries past min(K, row_bound[r]) are -1.  Scores compare by value
 *              (-0.0 == +0.0).
 *   ws         device workspace of ws_bytes >= idx_workspace_size() of a problem with these
 *              R and max_bound. */
idx_status idx_topk(const float *scores, int64_t ld, const int32_t *row_bound, int32_t R,
                    int32_t max_bound, int32_t K, const uint32_t *hist, int32_t *out_idx,
                    void *ws, size_t ws_bytes, void *stream);

/* The fused indexer launch: idx_score into workspace scratch, the fused first-digit
 * histogram, then idx_topk; out_idx as for idx_topk. */
idx_status idx_launch(const idx_problem *problem, int32_t K, int32_t *out_idx, void *ws,
                      size_t ws_bytes, void *stream);

/* idx_launch that also returns the selected keys' scores (the first half of a
 * key-sharded indexer: each shard ranks the keys it holds; see idx_merge_topk).
 *   out_score  device fp32 [R][K]: out_score[r][j] is the score of position
 *              out_idx[r][j] (-0.0 comes back as +0.0); -inf where out_idx is -1.
 * Other arguments and errors as for idx_launch; a NULL out_score is IDX_EINVAL. */
idx_status idx_launch_scored(const idx_problem *problem, int32_t K, int32_t *out_idx, float *out_score,
                             void *ws, size_t ws_bytes, void *stream);

/* Exact top-K of the union of S ranked parts: the merge of a key-sharded indexer.
 * The "Release Test Suite - GLM-5.2-EXL3" page (section Config change) runs decode
 * context parallelism with a top-k owner merge: every GPU ranks the keys of its
 * shard of the cache and one owner merges the lists.  The union of the shards'
 * top-K lists holds the global top-K, so the merge reproduces the unsharded
 * selection exactly.
 *   part_idx     device int32 [S][R][Kin]: part s's positions in its own numbering,
 *                ordered by score descending then position ascending, -1 padded
 *                (as idx_launch_scored writes them).
 *   part_score   device fp32 [S][R][Kin]: their scores (no NaN).
 *   part_offset  HOST int32 [S], >= 0: added to part s's positions; the parts must
 *                cover disjoint position ranges (a position of the request is in
 *                exactly one part).
 *   S            1 .. IDX_MERGE_MAX_PARTS; Kin, K in 1 .. IDX_MAX_K.
 *   out_idx      device int32 [R][K]: the merged positions, same order, -1 padded.
 *   out_score    device fp32 [R][K] or NULL: their scores, -inf where out_idx is -1.
 * Returns IDX_EINVAL for a bad argument and IDX_EUNSUPPORTED for S or R above the
 * limits; launches nothing then.
 * Asynchronous on `stream`; allocates nothing. */
#define IDX_MERGE_MAX_PARTS 8
idx_status idx_merge_topk(const int32_t *part_idx, const float *part_score, const int32_t *part_offset,
                          int32_t S, int32_t R, int32_t Kin, int32_t K, int32_t *out_idx, float *out_score,
                          void *stream);

/* Bytes of device arena idx_launch_host needs: the inputs' device copies, the
 * output and the workspace. */
size_t idx_host_arena_size(const idx_problem *host_problem, int32_t K);

/* idx_launch on HOST inputs.  host_problem's array pointers are host memory (pinned
 * memory makes the copies asynchronous; pageable memory makes them synchronous).
 * A rows_hint of 0 is replaced by the most rows of any request, counted from the
 * host row map.
 * Copies every input into `arena` (device, arena_bytes >= idx_host_arena_size()),
 * runs idx_launch and copies the [R][K] result back into host_out (host).  All
 * copies are issued on `stream`; the caller synchronises the stream before reading
 * host_out. */
idx_status idx_launch_host(const idx_problem *host_problem, int32_t K, int32_t *host_out,
                           void *arena, size_t arena_bytes, void *stream);

/* Synchronises `stream`, then reads and clears the device status word of workspace
 * `ws` (of the last call that used it): IDX_OK, IDX_ETIMEOUT or IDX_EDEVICE, or
 * IDX_ECUDA if the stream reports an error. */
idx_status idx_last_device_status(void *ws, void *stream);

/* Static description of a status code. */
const char *idx_status_string(idx_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t idx_version(void);

/* Test hooks.  IDX_DEBUG_WAIT_LIMIT_NS sets the time limit of every device-side wait
 * (default 1e9 ns); IDX_DEBUG_STALL_SCORE_MMA > 0 makes the next scoring launch hold
 * back its first accumulator hand-off, so that its waits run out and it reports
 * IDX_ETIMEOUT.  Process-wide; returns the previous value.  Not for production use. */
#define IDX_DEBUG_WAIT_LIMIT_NS 1
#define IDX_DEBUG_STALL_SCORE_MMA 2
int64_t idx_debug_set(int32_t what, int64_t value);

/* Measurement hook.  When `start` and `stop` (cudaEvent_t) are non-NULL, the next
 * idx_score or idx_launch records `start` on its stream just before the scoring
 * kernel and `stop` just after it, so the scoring kernel alone can be timed with
 * cudaEventElapsedTime.  Applies to one call, then clears itself.  Process-wide. */
void idx_profile_events(void *start, void *stop);

/* Writes every row's new key into the paged cache, ahead of idx_launch (the sglang
 * PR 48224 page, section Reviewer notes, "New keys": a key the launch writes is
 * scored for every row of its request in the launch).  Row r's key goes to logical
 * position row_bound[r] - 1 of request row_req[r], so the scan that follows reads it
 * for every row whose bound covers it.
 *   problem  as for idx_launch; problem->k_cache and problem->k_scale are WRITTEN
 *            (device memory the caller owns and may write).
 *   k_new    device bf16 [R][128], 16-byte aligned: each row's new key.
 * E4M3 cache: scale = amax / 448 in fp32 (1 for a zero key) goes to k_scale, and
 * each value divided by it in fp32 goes to the nearest E4M3 code (ties to even),
 * saturating at +-448.  bf16 cache: the values as given.  Rows with bound 0 write
 * nothing; a row whose page id is outside [0, P) writes nothing (idx_launch then
 * reports the page).  Rows of one request must have different bounds (each writes
 * its own position).  Asynchronous on `stream`; allocates nothing. */
idx_status idx_patch_new_keys(const idx_problem *problem, const void *k_new, void *stream);

/* idx_launch with the rows' new keys written first, inside the launch (the same
 * page section, "New keys": a key the launch writes is scored by every row of its
 * request whose bound covers it).  The launch's first kernel writes row r's key
 * at position row_bound[r] - 1 exactly as idx_patch_new_keys does, before the
 * scan reads the cache; the result equals idx_patch_new_keys followed by
 * idx_launch, in one launch sequence instead of two.
 *   problem  as for idx_launch; problem->k_cache and problem->k_scale are WRITTEN.
 *   k_new    device bf16 [R][128], 16-byte aligned (NULL or misaligned: IDX_EINVAL).
 * Other arguments, outputs and errors as for idx_launch; rows of one request must
 * have different bounds. */
idx_status idx_launch_new_keys(const idx_problem *problem, const void *k_new, int32_t K, int32_t *out_idx,
                               void *ws, size_t ws_bytes, void *stream);

/* Top-1 of each row of logits in one launch: the later "draft_topk1_postprocess"
 * commit on the sglang PR 48224 page.  Each split of a row folds its (value,
 * lowest index) into a per-row 64-bit key with an atomic maximum; the split that
 * arrives last writes the row's results and resets the row's state.  Ties go to
 * the lowest index; a NaN reads as -1e30; -0.0 and +0.0 compare equal.
 *   logits     device fp32 [R][ld], columns 0 .. V-1 read; ld >= V >= 1.
 *   out_idx    device int32 [R]: the index of each row's largest value.
 *   out_val    device fp32 [R] or NULL: that value (after the NaN reading; a zero
 *              maximum is written as +0.0).
 *   tokens     device int32 [R][tokens_ld] or NULL: tokens[r * tokens_ld + token_col]
 *              gets out_idx[r] (the draft token column); 0 <= token_col < tokens_ld.
 *   positions  device int32 [R] or NULL: positions[r] += 1.
 *   state      device buffer of state_bytes >= idx_top1_state_size(R), 16-byte
 *              aligned, all zero before its first use; every call leaves it zero
 *              again.  Calls that share a state must not overlap in time.
 * Returns IDX_EINVAL for a bad argument and IDX_EUNSUPPORTED for V > INT32_MAX, in
 * both cases launching nothing. */
size_t idx_top1_state_size(int32_t R);
idx_status idx_top1(const float *logits, int64_t ld, int32_t R, int64_t V, int32_t *out_idx,
                    float *out_val, int32_t *tokens, int64_t tokens_ld, int32_t token_col,
                    int32_t *positions, void *state, size_t state_bytes, void *stream);

/* Exact top-K of given scores with no caller workspace.  The page has no
 * counterpart: this is idx_topk run on scratch that lives in the library itself,
 * a file-scope device array of IDX_NOALLOC_SCRATCH_BYTES (enough for up to
 * IDX_NOALLOC_MAX_ROWS rows at any K up to IDX_MAX_K and any max_bound).  It is
 * for callers that cannot allocate device memory on their decode path: a host
 * program that links only this library and has no device allocator of its own,
 * or a serving loop that reserves all its memory up front because an allocation
 * between steps can synchronise the device or fail under memory pressure.  The
 * call allocates nothing.
 *   scores, ld, row_bound, R, max_bound, K, out_idx: as for idx_topk (no hist).
 *   R > IDX_NOALLOC_MAX_ROWS returns IDX_EUNSUPPORTED and launches nothing; the
 *   other argument checks are those of idx_topk (IDX_EINVAL).
 *   Setup: the first call on a device looks up the scratch's device address
 *   (cudaGetSymbolAddress) and keeps it for later calls; make that first call on
 *   each device before any stream capture begins.  A failed lookup returns
 *   IDX_ECUDA.  The kept address belongs to the device's context as it was at
 *   that first call: after a cudaDeviceReset (or anything else that destroys and
 *   recreates the device's primary context) the process must be restarted before
 *   this call is used on that device again.
 *   Nothing in the scratch has to start at zero: every call clears the selection
 *   state it uses before its kernels read it.
 *   The scratch is one per device and process: two calls whose work can overlap
 *   in time (different streams, or different host threads) race on it, and the
 *   caller must order them (e.g. one stream).  Device-detected errors (a row bound
 *   outside [0, max_bound], clamped as idx_topk does) have no readback here. */
#define IDX_NOALLOC_MAX_ROWS 8
#define IDX_NOALLOC_SCRATCH_BYTES (1280 * 1024)
idx_status idx_topk_noalloc(const float *scores, int64_t ld, const int32_t *row_bound, int32_t R,
                            int32_t max_bound, int32_t K, int32_t *out_idx, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H */
