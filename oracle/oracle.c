/*
 * Reference oracle for the long-context decode indexer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct CPU
 * statement of what the indexer computes.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant with the CUDA library; neither side includes the other.
 *
 * Source of the method: the sglang PR 48224 page (squashed sgl-amd-mono #86):
 *   - each row scored against every key its request has cached, then the row's
 *     exact top-2048 selected                          (section Motivation, first paragraph)
 *   - FP8 E4M3 and bf16 key caches                    (section Accuracy Tests)
 *   - positions from a row's bound on are not scored  (section Modifications, commit 2)
 *   - first radix digit is radix_key >> 26, 64 bins   (section Modifications, commit 4)
 * The score formula itself, score(s) = sum_h w_h * ReLU(scale_s * <q_h, k_s>) over
 * 64 heads of 128 dims, is the indexer statement the build is scoped by; the page
 * only names a reduction over halves of the heads (section Motivation, first bullet).
 *
 * All arithmetic is in IEEE double.  Each function is the definition written out;
 * nothing is blocked or fused beyond what the definition states.
 *
 * Readings of points the page leaves open (each also listed in the design notes):
 *   - bound semantics: row r sees logical key positions 0 .. bound_r - 1;
 *   - a logical position t of request q lives in physical page
 *     page_table[q * pt_stride + t / 64], slot t % 64 (page size 64);
 *   - the returned indices are logical positions, ordered by score descending and
 *     then position ascending, padded with -1 past min(K, bound_r);
 *   - scores compare by value (so -0.0 == +0.0) and ties go to the lower position;
 *   - radix_key is the order-preserving map of the fp32 bit pattern, with -0.0
 *     read as +0.0 so that equal values share one key.
 *
 * Parity of the score values is pinned by hand-derived exact cases, an
 * exhaustive E4M3 decode check and brute-force selection in the test suite.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORACLE_HEADS 64
#define ORACLE_DIM 128
#define ORACLE_PAGE 64

/* OCP 8-bit floating point, E4M3 "fn" variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits, subnormals when the exponent field is 0, no infinity,
 * NaN only for the exponent and mantissa fields all ones.  The page stores its
 * index keys as "FP8 E4M3" (section Speed Tests, "FP8 E4M3 KV"). */
double oracle_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int exp_field = (code >> 3) & 0xF;
    int man_field = code & 0x7;
    double magnitude;
    if (exp_field == 0xF && man_field == 0x7) return NAN;
    if (exp_field == 0) {
        magnitude = ldexp((double)man_field / 8.0, 1 - 7);
    } else {
        magnitude = ldexp(1.0 + (double)man_field / 8.0, exp_field - 7);
    }
    return sign ? -magnitude : magnitude;
}

double oracle_bf16_to_double(uint16_t bits);

/* The E4M3 code nearest to x (ties to an even mantissa), from the format above:
 * |x| is first clamped to the largest finite value 448; below 2^-6 the step is the
 * subnormal one, 2^-9.  Every step is exact in double. */
uint8_t oracle_e4m3_encode(float x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a > 448.0) a = 448.0;
    if (a < ldexp(1.0, -6)) {                       /* subnormal range: m * 2^-9, m in 0..8 */
        const double m = rint(ldexp(a, 9));         /* m == 8 is the smallest normal, 2^-6 */
        return (uint8_t)(sign | (uint8_t)m);
    }
    int e = ilogb(a);                               /* a = f * 2^e, 1 <= f < 2 */
    double m = rint(ldexp(a, 3 - e));               /* 8 .. 16 */
    if (m == 16.0) {
        m = 8.0;
        e += 1;
    }
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)((int)m - 8));
}

/* The new key of a decode row, as the launch writes it into the paged cache (the
 * page's Reviewer notes, "New keys": a key that the launch writes is scored for
 * every row of its request).  E4M3 cache: scale = amax / 448 in fp32
 * (1 for a zero key), each value x / scale in fp32, clamped to +-448, encoded to
 * the nearest E4M3 code.  bf16 cache: the values as given.  key_bf16 [128]. */
void oracle_quantize_key(const uint16_t *key_bf16, uint8_t *codes, float *scale) {
    float amax = 0.0f;
    for (int i = 0; i < ORACLE_DIM; ++i) {
        const float v = fabsf((float)oracle_bf16_to_double(key_bf16[i]));
        if (v > amax) amax = v;
    }
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int i = 0; i < ORACLE_DIM; ++i) codes[i] = oracle_e4m3_encode((float)oracle_bf16_to_double(key_bf16[i]) / sc);
    *scale = sc;
}

/* Where row r's new key goes: logical position t = row_bound[r] - 1 of its
 * request, i.e. page id *page at slot *slot.  Returns 0 for a row with bound 0
 * (it adds no key), 1 otherwise. */
static int new_key_target(const int32_t *row_req, const int32_t *row_bound, const int32_t *page_table,
                          int64_t pt_stride, int r, int64_t *page, int64_t *slot) {
    if (row_bound[r] == 0) return 0;
    const int64_t t = (int64_t)row_bound[r] - 1;
    *page = page_table[(int64_t)row_req[r] * pt_stride + t / ORACLE_PAGE];
    *slot = t % ORACLE_PAGE;
    return 1;
}

/* Writes every row's new key into the paged cache (the page's Reviewer notes,
 * "New keys": the key a decode row adds sits at the row's last visible position,
 * bound - 1, and is scored by every row of its request whose bound covers it).
 * Row r's key goes to logical position t = row_bound[r] - 1 of request
 * row_req[r]: physical page page_table[req * pt_stride + t / 64], slot t % 64.
 * Rows with bound 0 add no key.  E4M3 cache (kv_dtype 0): oracle_quantize_key's
 * codes and scale; bf16 cache (kv_dtype 1): the bf16 values as given.
 *   k_new [R][128] bf16 bit patterns; k_cache / k_scale are written in place.
 * Returns 0, or -1 (nothing written) if a row's request, bound or page id is out
 * of range. */
int oracle_patch_new_keys(const uint16_t *k_new, const int32_t *row_req, const int32_t *row_bound, int R,
                          const int32_t *page_table, int64_t pt_stride, int Q, void *k_cache, float *k_scale,
                          int kv_dtype, int64_t P) {
    int64_t page, slot;
    for (int r = 0; r < R; ++r) {
        if (row_req[r] < 0 || row_req[r] >= Q || row_bound[r] < 0 ||
            (int64_t)row_bound[r] > pt_stride * ORACLE_PAGE)
            return -1;
        if (new_key_target(row_req, row_bound, page_table, pt_stride, r, &page, &slot) &&
            (page < 0 || page >= P))
            return -1;
    }
    for (int r = 0; r < R; ++r) {
        if (!new_key_target(row_req, row_bound, page_table, pt_stride, r, &page, &slot)) continue;
        const uint16_t *key = k_new + (int64_t)r * ORACLE_DIM;
        if (kv_dtype == 0) {
            oracle_quantize_key(key, (uint8_t *)k_cache + (page * ORACLE_PAGE + slot) * ORACLE_DIM,
                                &k_scale[page * ORACLE_PAGE + slot]);
        } else {
            memcpy((uint16_t *)k_cache + (page * ORACLE_PAGE + slot) * ORACLE_DIM, key,
                   ORACLE_DIM * sizeof(uint16_t));
        }
    }
    return 0;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t wide = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &wide, sizeof f);
    return (double)f;
}

/* The key at logical position t of request req, dequantised into kd[0..127],
 * and its per-token scale.  kv_dtype 0 = E4M3 bytes with an fp32 scale per token,
 * kv_dtype 1 = bf16 values with scale 1. */
static double load_key(const void *k_cache, int kv_dtype, const float *k_scale,
                       const int32_t *page_table, int64_t pt_stride, int req, int64_t t,
                       double *kd) {
    int64_t page = page_table[(int64_t)req * pt_stride + t / ORACLE_PAGE];
    int64_t slot = t % ORACLE_PAGE;
    int64_t base = (page * ORACLE_PAGE + slot) * ORACLE_DIM;
    if (kv_dtype == 0) {
        const uint8_t *k8 = (const uint8_t *)k_cache;
        for (int i = 0; i < ORACLE_DIM; ++i) kd[i] = oracle_e4m3_to_double(k8[base + i]);
        return (double)k_scale[page * ORACLE_PAGE + slot];
    }
    const uint16_t *kb = (const uint16_t *)k_cache;
    for (int i = 0; i < ORACLE_DIM; ++i) kd[i] = oracle_bf16_to_double(kb[base + i]);
    return 1.0;
}

/* score(t) = sum_h w_h * max(0, scale_t * <q_h, k_t>) for one row, written out.
 * qt holds the row's query transposed to [dim][head] in double so that the 64
 * independent dot products advance together; each dot product still sums its
 * 128 terms in dimension order 0..127. */
static double score_one(const double *qt, const double *w, const double *kd, double scale) {
    double dot[ORACLE_HEADS];
    for (int h = 0; h < ORACLE_HEADS; ++h) dot[h] = 0.0;
    for (int i = 0; i < ORACLE_DIM; ++i) {
        double k = kd[i];
        const double *qrow = qt + (int64_t)i * ORACLE_HEADS;
        for (int h = 0; h < ORACLE_HEADS; ++h) dot[h] += qrow[h] * k;
    }
    double s = 0.0;
    for (int h = 0; h < ORACLE_HEADS; ++h) {
        double a = scale * dot[h];
        double relu = a > 0.0 ? a : 0.0;
        s += w[h] * relu;
    }
    return s;
}

static void row_query(const uint16_t *q_bf16, const float *w, int r, double *qt, double *wd) {
    const uint16_t *qr = q_bf16 + (int64_t)r * ORACLE_HEADS * ORACLE_DIM;
    for (int h = 0; h < ORACLE_HEADS; ++h)
        for (int i = 0; i < ORACLE_DIM; ++i)
            qt[(int64_t)i * ORACLE_HEADS + h] = oracle_bf16_to_double(qr[h * ORACLE_DIM + i]);
    for (int h = 0; h < ORACLE_HEADS; ++h) wd[h] = (double)w[(int64_t)r * ORACLE_HEADS + h];
}

/* Scores of every row over its visible keys.
 *   q_bf16     [R][64][128] bf16 bit patterns
 *   w          [R][64] fp32
 *   k_cache    [P][64][128] E4M3 bytes (kv_dtype 0) or bf16 (kv_dtype 1)
 *   k_scale    [P][64] fp32 (kv_dtype 0; ignored for kv_dtype 1)
 *   page_table [Q][pt_stride] page ids
 *   row_req    [R] request of each row; row_bound [R] keys visible to each row
 *   out        [R][ld] doubles; positions t >= row_bound[r] are left untouched.
 * Returns 0, or -1 if an argument is out of range (nothing is computed then). */
int oracle_score(const uint16_t *q_bf16, const float *w, const void *k_cache, int kv_dtype,
                 const float *k_scale, const int32_t *page_table, int64_t pt_stride,
                 const int32_t *row_req, const int32_t *row_bound, int R, int64_t P,
                 double *out, int64_t ld) {
    for (int r = 0; r < R; ++r) {
        if (row_bound[r] < 0 || row_bound[r] > ld || row_bound[r] > pt_stride * ORACLE_PAGE) return -1;
        if (row_req[r] < 0) return -1;
        for (int64_t p = 0; p < (row_bound[r] + ORACLE_PAGE - 1) / ORACLE_PAGE; ++p) {
            int32_t page = page_table[(int64_t)row_req[r] * pt_stride + p];
            if (page < 0 || page >= P) return -1;
        }
    }
    const int64_t block = 256;
    int64_t nblocks_max = 0;
    for (int r = 0; r < R; ++r) {
        int64_t nb = (row_bound[r] + block - 1) / block;
        if (nb > nblocks_max) nblocks_max = nb;
    }
    int64_t work = (int64_t)R * nblocks_max;
#pragma omp parallel
    {
        double *qt = (double *)malloc(sizeof(double) * ORACLE_HEADS * ORACLE_DIM);
        double wd[ORACLE_HEADS];
        double kd[ORACLE_DIM];
        int cur_row = -1;
#pragma omp for schedule(dynamic, 1)
        for (int64_t item = 0; item < work; ++item) {
            int r = (int)(item / nblocks_max);
            int64_t b = item % nblocks_max;
            int64_t t0 = b * block;
            int64_t t1 = t0 + block;
            if (t1 > row_bound[r]) t1 = row_bound[r];
            if (t0 >= t1) continue;
            if (r != cur_row) {
                row_query(q_bf16, w, r, qt, wd);
                cur_row = r;
            }
            for (int64_t t = t0; t < t1; ++t) {
                double sc = load_key(k_cache, kv_dtype, k_scale, page_table, pt_stride, row_req[r], t, kd);
                out[(int64_t)r * ld + t] = score_one(qt, wd, kd, sc);
            }
        }
        free(qt);
    }
    return 0;
}

/* Scores at n chosen (row, position) points, for checks on inputs too large to
 * score whole.  Same definition as oracle_score.  Returns 0, or -1 if a point is
 * outside its row's bound or reaches a page id outside [0, P). */
int oracle_score_points(const uint16_t *q_bf16, const float *w, const void *k_cache, int kv_dtype,
                        const float *k_scale, const int32_t *page_table, int64_t pt_stride,
                        const int32_t *row_req, const int32_t *row_bound, int64_t P,
                        const int32_t *pt_rows, const int64_t *pt_pos, int64_t n, double *out) {
    for (int64_t j = 0; j < n; ++j) {
        int r = pt_rows[j];
        if (pt_pos[j] < 0 || pt_pos[j] >= row_bound[r]) return -1;
        int32_t page = page_table[(int64_t)row_req[r] * pt_stride + pt_pos[j] / ORACLE_PAGE];
        if (page < 0 || page >= P) return -1;
    }
#pragma omp parallel
    {
        double *qt = (double *)malloc(sizeof(double) * ORACLE_HEADS * ORACLE_DIM);
        double wd[ORACLE_HEADS];
        double kd[ORACLE_DIM];
        int cur_row = -1;
#pragma omp for schedule(static)
        for (int64_t j = 0; j < n; ++j) {
            int r = pt_rows[j];
            if (r != cur_row) {
                row_query(q_bf16, w, r, qt, wd);
                cur_row = r;
            }
            double sc = load_key(k_cache, kv_dtype, k_scale, page_table, pt_stride, row_req[r], pt_pos[j], kd);
            out[j] = score_one(qt, wd, kd, sc);
        }
        free(qt);
    }
    return 0;
}

/* ---- selection ---------------------------------------------------------------- */

typedef struct {
    float score;
    int32_t pos;
} scored_key;

/* Score descending, then position ascending.  Comparison by value: -0.0 == +0.0. */
static int by_score_then_pos(const void *a, const void *b) {
    const scored_key *x = (const scored_key *)a;
    const scored_key *y = (const scored_key *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    if (x->pos < y->pos) return -1;
    if (x->pos > y->pos) return 1;
    return 0;
}

/* Exact top-K of each row by definition: order all bound_r (score, position)
 * pairs, keep the first min(K, bound_r) positions, pad the row of out_idx [R][K]
 * with -1.  Scores are fp32 as the indexer stores them.  Returns 0, or -1 if a
 * score within a bound is NaN (the order is then undefined). */
int oracle_topk(const float *scores, int64_t ld, const int32_t *row_bound, int R, int K,
                int32_t *out_idx) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < R; ++r) {
        int64_t n = row_bound[r];
        scored_key *v = (scored_key *)malloc(sizeof(scored_key) * (size_t)(n > 0 ? n : 1));
        for (int64_t t = 0; t < n; ++t) {
            v[t].score = scores[(int64_t)r * ld + t];
            v[t].pos = (int32_t)t;
            if (isnan(v[t].score)) bad = 1;
        }
        qsort(v, (size_t)n, sizeof(scored_key), by_score_then_pos);
        for (int j = 0; j < K; ++j) out_idx[(int64_t)r * K + j] = (j < n) ? v[j].pos : -1;
        free(v);
    }
    return bad ? -1 : 0;
}

/* Order-preserving unsigned key of an fp32 value: a larger key means a larger
 * value.  Non-negative values get the sign bit set; negative values are bitwise
 * inverted.  -0.0 is first read as +0.0.  The page's first radix digit is this
 * key's top 6 bits, radix_key >> 26 (section Modifications, commit 4). */
/* Merge of a key-sharded selection, by definition: the exact top-K of the union
 * of S parts.  The "Release Test Suite - GLM-5.2-EXL3" page (section Config
 * change) merges each GPU's indexer top-k at an owner under decode context
 * parallelism.  Part s holds, for each row, up to Kin (score, position) pairs with
 * positions in its own numbering (-1 marks an empty entry); global position =
 * position + offset[s].  Every pair of every part is put in one list, ordered as
 * oracle_topk orders (score descending by value, then position ascending), and
 * the first K global positions are kept, -1 padded.
 *   part_idx / part_score [S][R][Kin]; offset [S]; out_idx [R][K].
 * Returns 0, or -1 if a listed score is NaN. */
int oracle_merge_topk(const int32_t *part_idx, const float *part_score, const int32_t *offset, int S, int R,
                      int Kin, int K, int32_t *out_idx) {
    int bad = 0;
    for (int r = 0; r < R; ++r) {
        scored_key *v = (scored_key *)malloc(sizeof(scored_key) * (size_t)S * (size_t)Kin + 1);
        int64_t n = 0;
        for (int s = 0; s < S; ++s) {
            for (int j = 0; j < Kin; ++j) {
                const int64_t at = ((int64_t)s * R + r) * Kin + j;
                if (part_idx[at] < 0) continue;
                v[n].score = part_score[at];
                v[n].pos = part_idx[at] + offset[s];
                if (isnan(v[n].score)) bad = 1;
                ++n;
            }
        }
        qsort(v, (size_t)n, sizeof(scored_key), by_score_then_pos);
        for (int j = 0; j < K; ++j) out_idx[(int64_t)r * K + j] = j < n ? v[j].pos : -1;
        free(v);
    }
    return bad ? -1 : 0;
}

uint32_t oracle_radix_key(float x) {
    uint32_t u;
    if (x == 0.0f) x = 0.0f;
    memcpy(&u, &x, sizeof u);
    return (u >> 31) ? ~u : (u | 0x80000000u);
}

/* hist [R][64]: for each row, the count of first digits radix_key(score) >> 26
 * over positions t < bound_r. */
void oracle_first_digit_hist(const float *scores, int64_t ld, const int32_t *row_bound, int R,
                             uint32_t *hist) {
    for (int r = 0; r < R; ++r) {
        for (int b = 0; b < 64; ++b) hist[r * 64 + b] = 0;
        for (int64_t t = 0; t < row_bound[r]; ++t)
            hist[r * 64 + (oracle_radix_key(scores[(int64_t)r * ld + t]) >> 26)] += 1;
    }
}

/* Top-1 of each row of logits (the sglang PR 48224 page, later commit
 * "draft_topk1_postprocess"): the largest value, ties to the lowest index, a NaN
 * read as -1e30.  out_idx [R] gets the index, out_val [R] the value as read.
 * Values compare as floats, so -0.0 and +0.0 tie.  V >= 1. */
void oracle_top1(const float *logits, int64_t ld, int R, int64_t V, int32_t *out_idx, float *out_val) {
    for (int r = 0; r < R; ++r) {
        const float *row = logits + (int64_t)r * ld;
        int64_t best = 0;
        float bv = isnan(row[0]) ? -1e30f : row[0];
        for (int64_t j = 1; j < V; ++j) {
            const float v = isnan(row[j]) ? -1e30f : row[j];
            if (v > bv) {
                bv = v;
                best = j;
            }
        }
        out_idx[r] = (int32_t)best;
        out_val[r] = bv;
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
