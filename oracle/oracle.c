/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the sparse-attention indexer
 * computes, in float64.  It exists to check the CUDA library, never to stand in for it:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (web pages; each function names the passage it restates):
 *   [scores]  "flashinfer.attn_scores" -- fp8_paged_mqa_logits: the formula block, the Note on
 *             per-slot extents, and the Parameters list (q, kv_fused, weights, block_tables,
 *             seq_lens, out).
 *   [fp4]     "flashinfer.attn_scores" -- fp4_paged_mqa_logits: the formula block and the
 *             Parameters list (q, q_sf, kv_fused with its byte-offset drawing, sf_vec_size).
 *   [select]  "flashinfer.sdsa.indexer_threshold_select" -- the description (candidate / tie
 *             classification, fit rule, repair) and the Parameters list (row_ends,
 *             thresholds, counters, candidates, arrivals, ranges).
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py against values
 * the pages print, library routines and brute force (see each function's comment).
 *
 * Arithmetic: float64 throughout.  An e4m3 value has at most 4 significant bits, so each
 * product q_d * k_d has at most 8 and lies in [2^-18, 448^2]; a sum of 128 such products
 * needs fewer than 53 bits, so every per-head score s_h below is EXACT.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Error codes returned by the oracle (never by the CUDA library). */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_BAD_PAGE -2    /* a block-table entry the definition needs is outside the pool */
#define ORACLE_BAD_COLUMN -3  /* a position the definition needs is outside the output row */
#define ORACLE_NO_MEMORY -4

/* ------------------------------------------------------------------------------------------ */
/* Number formats                                                                              */
/* ------------------------------------------------------------------------------------------ */

/*
 * OCP 8-bit floating point, E4M3 "fn" variant (the float8_e4m3fn dtype the q parameter and the
 * kv_fused value region carry, [scores] Parameters): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 encodes subnormals 2^-6 * m/8; there are no infinities and
 * only S.1111.111 is NaN.
 */
double oracle_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int exponent = (code >> 3) & 0xF;
    int mantissa = code & 0x7;
    double magnitude;
    if (exponent == 0xF && mantissa == 0x7) return NAN;
    if (exponent == 0)
        magnitude = ldexp((double)mantissa / 8.0, -6);
    else
        magnitude = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);
    return sign ? -magnitude : magnitude;
}

/* A little-endian IEEE binary32 stored at p ([scores] Parameters: kv_fused, region 2). */
double oracle_f32_le(const uint8_t *p) {
    uint32_t bits = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
                    ((uint32_t)p[3] << 24);
    float value;
    memcpy(&value, &bits, sizeof value);
    return (double)value;
}

/* ------------------------------------------------------------------------------------------ */
/* Helpers named on [scores] "Scheduling and Setup"                                            */
/* ------------------------------------------------------------------------------------------ */

/* min_block_table_width(seq_len, block_size) = ceil(seq_len / block_size)
 * ([scores] Example comment "ceil(8000/32) = 250" and Parameters: block_tables). */
int64_t oracle_min_block_table_width(int64_t seq_len, int64_t block_size) {
    if (seq_len < 0 || block_size <= 0) return -1;
    return (seq_len + block_size - 1) / block_size;
}

/* padded_seq_len(max_seq_len): the pages print only the example 8000 -> 8192 and say the
 * column count is padded to "an internal store granularity".  Reading used here: round up to a
 * multiple of 256 columns (the smallest power-of-two granularity that maps 8000 to 8192). */
int64_t oracle_padded_seq_len(int64_t max_seq_len) {
    if (max_seq_len < 0) return -1;
    return (max_seq_len + 255) / 256 * 256;
}

/* The per-slot extent ([scores] Note and Returns): row b*next_n+t is meaningful for KV positions
 * 0 .. seq_lens[b] - next_n + t inclusive, i.e. the first seq_lens[b] - next_n + t + 1 of them
 * (none when that count is not positive). */
int64_t oracle_row_end(int64_t seq_len, int64_t next_n, int64_t t) {
    int64_t count = seq_len - next_n + t + 1;
    return count > 0 ? count : 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Paged MQA logits                                                                            */
/* ------------------------------------------------------------------------------------------ */

/*
 * logits[b*next_n + t, p] = scale[p] * sum_h w[b*next_n + t, h] * relu(q[b,t,h,:] . k[p,:])
 * ([scores] fp8_paged_mqa_logits formula block), for every request b with seq_lens[b] > 0,
 * every draft slot t < next_n and every position p inside the slot's extent.
 *
 * Where k[p,:] and scale[p] live ([scores] Parameters: kv_fused and block_tables): position p
 * of request b sits in physical block pg = block_tables[b, p / block_size] at in-block token
 * i = p % block_size.  The block is block_size*(head_dim+4) bytes: bytes [0, block_size*head_dim)
 * hold the e4m3 values token-major (token i at i*head_dim), bytes [block_size*head_dim, end)
 * hold block_size little-endian float32 scales (token i's at block_size*head_dim + 4*i).
 *
 * Layouts: q is [batch, next_n, num_heads, head_dim] e4m3 bytes, contiguous; weights is
 * [batch*next_n, num_heads] float32, contiguous; block_tables[b, j] is at
 * block_tables[b*bt_row_stride + j]; seq_lens[b] is at seq_lens[b*seq_lens_stride].
 *
 * Outputs (float64): out[r*out_row_stride + p] = the logit, and, if tol is not NULL,
 * tol[r*out_row_stride + p] = |scale[p]| * sum_h |w[r,h] * relu(s_h)|, the magnitude against
 * which a float32 implementation's rounding is judged.  Entries outside every row's extent, and
 * every entry of a request with seq_lens[b] == 0, are left untouched ([scores] Note: such rows
 * "are never written").
 *
 * Returns ORACLE_OK, or ORACLE_BAD_PAGE if a block-table entry the definition needs is outside
 * [0, num_blocks) (the oracle never reads an entry past ceil(seq_lens[b] / block_size)), or
 * ORACLE_BAD_COLUMN if an extent runs past out_cols.
 */
int oracle_paged_logits(const uint8_t *q, const uint8_t *kv_fused, int64_t num_blocks,
                        int block_size, const float *weights, const int32_t *block_tables,
                        int64_t bt_row_stride, int64_t bt_width, const int32_t *seq_lens,
                        int64_t seq_lens_stride, int batch, int next_n, int num_heads,
                        int head_dim, double *out, int64_t out_row_stride, int64_t out_cols,
                        double *tol, int nthreads) {
    if (!q || !kv_fused || !weights || !block_tables || !seq_lens || !out) return ORACLE_BAD_ARG;
    if (block_size <= 0 || batch < 0 || next_n <= 0 || num_heads <= 0 || head_dim <= 0)
        return ORACLE_BAD_ARG;

    const int64_t block_bytes = (int64_t)block_size * (head_dim + 4);
    const int64_t scale_region = (int64_t)block_size * head_dim;
    const int64_t rows = (int64_t)batch * next_n;
    /* Work items: (row, chunk of 256 positions), so long rows spread over threads. */
    const int64_t chunk = 256;
    int64_t max_len = 0;
    for (int b = 0; b < batch; ++b)
        if (seq_lens[(int64_t)b * seq_lens_stride] > max_len)
            max_len = seq_lens[(int64_t)b * seq_lens_stride];
    const int64_t chunks_per_row = (max_len + chunk - 1) / chunk;
    int status = ORACLE_OK;

    double *qd = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * num_heads *
                                  head_dim);
    if (!qd) return ORACLE_NO_MEMORY;
    for (int64_t i = 0; i < rows * num_heads * head_dim; ++i) qd[i] = oracle_e4m3_to_double(q[i]);

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double *kd = (double *)malloc(sizeof(double) * (size_t)head_dim);
        int64_t item;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (item = 0; item < rows * chunks_per_row; ++item) {
            const int64_t r = item / chunks_per_row;
            const int64_t b = r / next_n;
            const int64_t t = r % next_n;
            const int64_t seq_len = seq_lens[b * seq_lens_stride];
            const int64_t row_end = oracle_row_end(seq_len, next_n, t);
            const int64_t p_begin = (item % chunks_per_row) * chunk;
            int64_t p_end = p_begin + chunk;
            if (p_end > row_end) p_end = row_end;
            if (!kd) {
                status = ORACLE_NO_MEMORY;
                continue;
            }
            if (seq_len == 0) continue;
            for (int64_t p = p_begin; p < p_end; ++p) {
                const int64_t j = p / block_size;
                const int64_t i = p % block_size;
                if (j >= bt_width) {
                    status = ORACLE_BAD_PAGE;
                    break;
                }
                const int64_t pg = block_tables[b * bt_row_stride + j];
                if (pg < 0 || pg >= num_blocks) {
                    status = ORACLE_BAD_PAGE;
                    break;
                }
                if (p >= out_cols) {
                    status = ORACLE_BAD_COLUMN;
                    break;
                }
                const uint8_t *block = kv_fused + pg * block_bytes;
                for (int d = 0; d < head_dim; ++d)
                    kd[d] = oracle_e4m3_to_double(block[i * head_dim + d]);
                const double scale = oracle_f32_le(block + scale_region + 4 * i);
                double weighted = 0.0, magnitude = 0.0;
                for (int h = 0; h < num_heads; ++h) {
                    const double *qh = qd + (r * num_heads + h) * head_dim;
                    double s = 0.0;
                    for (int d = 0; d < head_dim; ++d) s += qh[d] * kd[d];
                    /* ReLU per head, before the weighted sum ([scores] formula notes). */
                    const double relu = s > 0.0 ? s : 0.0;
                    const double wh = (double)weights[r * num_heads + h];
                    weighted += wh * relu;
                    magnitude += fabs(wh * relu);
                }
                out[r * out_row_stride + p] = scale * weighted;
                if (tol) tol[r * out_row_stride + p] = fabs(scale) * magnitude;
            }
        }
        free(kd);
    }
    free(qd);
    return status;
}

/* ------------------------------------------------------------------------------------------ */
/* MXFP4 paged MQA logits                                                                      */
/* ------------------------------------------------------------------------------------------ */

/*
 * OCP microscaling FP4 element, E2M1 ([fp4] Parameters: q, "Two FP4 (E2M1) values packed per
 * byte"): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent field 0 encodes the
 * subnormal m/2; there are no infinities and no NaN.  Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 */
double oracle_e2m1_to_double(uint8_t nibble) {
    const int sign = (nibble >> 3) & 1;
    const int exponent = (nibble >> 1) & 3;
    const int mantissa = nibble & 1;
    const double magnitude = exponent == 0 ? 0.5 * mantissa
                                           : ldexp(1.0 + 0.5 * mantissa, exponent - 1);
    return sign ? -magnitude : magnitude;
}

/* A UE8M0 scale factor ([fp4] Parameters: q_sf, "the raw float32 exponent byte"): 2^(e - 127);
 * the all-ones byte is NaN in the OCP microscaling formats. */
double oracle_ue8m0_to_double(uint8_t e) { return e == 0xFF ? NAN : ldexp(1.0, (int)e - 127); }

/*
 * logits[b*next_n + t, p] = sum_h w[b*next_n + t, h] * relu(q[b,t,h,:] . k[p,:])
 * ([fp4] formula block), with every element dequantized: element d of a head_dim-long row is
 * e2m1(its nibble) * ue8m0(the row's scale byte d / 32) (sf_vec_size = 32).  There is no
 * per-position factor: the block scales are part of the values ([fp4] description).
 *
 * Layouts ([fp4] Parameters): a row of head_dim elements is head_dim/2 bytes, byte j holding
 * element 2j in its low nibble and element 2j+1 in its high nibble; q is [batch, next_n,
 * num_heads, head_dim/2] bytes; q_sf is [batch, next_n, num_heads, head_dim/32] bytes (the
 * little-endian bytes of the pages' int32 view: byte k scales elements [32k, 32k + 32)); a
 * kv_fused block is block_size*(head_dim/2 + head_dim/32) bytes: the packed rows token-major
 * (token i at i*head_dim/2), then head_dim/32 scale bytes per token (token i's at
 * block_size*head_dim/2 + (head_dim/32)*i).  Extents, paging and the untouched entries are as
 * in oracle_paged_logits; tol = sum_h |w relu(s_h)|.
 *
 * Each product is exact in float64 (2 significant bits times 2 times a power of two); the
 * head sums are exact unless a row's scales span more than ~45 binades.
 */
int oracle_paged_logits_mxfp4(const uint8_t *q, const uint8_t *q_sf, const uint8_t *kv_fused,
                              int64_t num_blocks, int block_size, const float *weights,
                              const int32_t *block_tables, int64_t bt_row_stride,
                              int64_t bt_width, const int32_t *seq_lens, int64_t seq_lens_stride,
                              int batch, int next_n, int num_heads, int head_dim, double *out,
                              int64_t out_row_stride, int64_t out_cols, double *tol,
                              int nthreads) {
    if (!q || !q_sf || !kv_fused || !weights || !block_tables || !seq_lens || !out)
        return ORACLE_BAD_ARG;
    if (block_size <= 0 || batch < 0 || next_n <= 0 || num_heads <= 0 || head_dim <= 0 ||
        head_dim % 32 != 0)
        return ORACLE_BAD_ARG;
    const int row_bytes = head_dim / 2, groups = head_dim / 32;
    const int64_t block_bytes = (int64_t)block_size * (row_bytes + groups);
    const int64_t scale_region = (int64_t)block_size * row_bytes;
    const int64_t rows = (int64_t)batch * next_n;
    const int64_t chunk = 256;
    int64_t max_len = 0;
    for (int b = 0; b < batch; ++b)
        if (seq_lens[(int64_t)b * seq_lens_stride] > max_len)
            max_len = seq_lens[(int64_t)b * seq_lens_stride];
    const int64_t chunks_per_row = (max_len + chunk - 1) / chunk;
    int status = ORACLE_OK;

    /* q dequantized once: row (r, h) element d. */
    double *qd = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * num_heads *
                                  head_dim);
    if (!qd) return ORACLE_NO_MEMORY;
    for (int64_t rh = 0; rh < rows * num_heads; ++rh)
        for (int d = 0; d < head_dim; ++d) {
            const uint8_t byte = q[rh * row_bytes + d / 2];
            const uint8_t nibble = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            qd[rh * head_dim + d] =
                oracle_e2m1_to_double(nibble) * oracle_ue8m0_to_double(q_sf[rh * groups + d / 32]);
        }

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double *kd = (double *)malloc(sizeof(double) * (size_t)head_dim);
        int64_t item;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (item = 0; item < rows * chunks_per_row; ++item) {
            const int64_t r = item / chunks_per_row;
            const int64_t b = r / next_n;
            const int64_t t = r % next_n;
            const int64_t seq_len = seq_lens[b * seq_lens_stride];
            const int64_t row_end = oracle_row_end(seq_len, next_n, t);
            const int64_t p_begin = (item % chunks_per_row) * chunk;
            int64_t p_end = p_begin + chunk;
            if (p_end > row_end) p_end = row_end;
            if (!kd) {
                status = ORACLE_NO_MEMORY;
                continue;
            }
            if (seq_len == 0) continue;
            for (int64_t p = p_begin; p < p_end; ++p) {
                const int64_t j = p / block_size;
                const int64_t i = p % block_size;
                if (j >= bt_width) {
                    status = ORACLE_BAD_PAGE;
                    break;
                }
                const int64_t pg = block_tables[b * bt_row_stride + j];
                if (pg < 0 || pg >= num_blocks) {
                    status = ORACLE_BAD_PAGE;
                    break;
                }
                if (p >= out_cols) {
                    status = ORACLE_BAD_COLUMN;
                    break;
                }
                const uint8_t *block = kv_fused + pg * block_bytes;
                for (int d = 0; d < head_dim; ++d) {
                    const uint8_t byte = block[i * row_bytes + d / 2];
                    const uint8_t nibble = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
                    kd[d] = oracle_e2m1_to_double(nibble) *
                            oracle_ue8m0_to_double(block[scale_region + i * groups + d / 32]);
                }
                double weighted = 0.0, magnitude = 0.0;
                for (int h = 0; h < num_heads; ++h) {
                    const double *qh = qd + (r * num_heads + h) * head_dim;
                    double s = 0.0;
                    for (int d = 0; d < head_dim; ++d) s += qh[d] * kd[d];
                    const double relu = s > 0.0 ? s : 0.0;
                    const double wh = (double)weights[r * num_heads + h];
                    weighted += wh * relu;
                    magnitude += fabs(wh * relu);
                }
                out[r * out_row_stride + p] = weighted;
                if (tol) tol[r * out_row_stride + p] = magnitude;
            }
        }
        free(kd);
    }
    free(qd);
    return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Top-k                                                                                       */
/* ------------------------------------------------------------------------------------------ */

/*
 * IEEE 754-2008 totalOrder on binary32 (section 5.10): numerically ordered, with -0 below +0,
 * NaNs with the sign bit clear above +inf (larger payload higher) and NaNs with the sign bit set
 * below -inf (larger payload lower).  Returns <0, 0, >0.
 */
int oracle_total_order_cmp(float a, float b) {
    uint32_t ba, bb;
    memcpy(&ba, &a, 4);
    memcpy(&bb, &b, 4);
    const int na = isnan(a), nb = isnan(b);
    const int sa = (ba >> 31) != 0, sb = (bb >> 31) != 0;
    if (na || nb) {
        if (na && nb) {
            if (sa != sb) return sa ? -1 : 1;
            const uint32_t pa = ba & 0x7FFFFFFFu, pb = bb & 0x7FFFFFFFu;
            if (pa == pb) return 0;
            if (!sa) return pa < pb ? -1 : 1;
            return pa < pb ? 1 : -1;
        }
        if (na) return sa ? -1 : 1;
        return sb ? 1 : -1;
    }
    if (a < b) return -1;
    if (a > b) return 1;
    if (sa != sb) return sa ? -1 : 1; /* -0 < +0 */
    return 0;
}

typedef struct {
    float value;
    int32_t index;
} oracle_scored_key;

/* Descending value (totalOrder), then ascending index: the order in which the top-k is taken
 * (ties broken by the lowest key index). */
static int oracle_rank_cmp(const void *x, const void *y) {
    const oracle_scored_key *a = (const oracle_scored_key *)x;
    const oracle_scored_key *b = (const oracle_scored_key *)y;
    const int c = oracle_total_order_cmp(a->value, b->value);
    if (c != 0) return -c;
    return (a->index > b->index) - (a->index < b->index);
}

/*
 * The exact top-k of each row: row r's keys are positions 0 .. row_ends[r]-1 of
 * logits[r*row_stride + .] ([select] Parameters: row_ends); K' = min(row_ends[r], top_k) of them
 * are taken, ordered by descending value and ascending index, by a full sort of the row.
 * idx_out[r*top_k + i] (i < K') receives them in that order, count_out[r] = K'.
 */
int oracle_topk(const float *logits, int64_t row_stride, const int32_t *row_ends, int rows,
                int top_k, int32_t *idx_out, int32_t *count_out, int nthreads) {
    if (!logits || !row_ends || !idx_out || !count_out || top_k < 0 || rows < 0)
        return ORACLE_BAD_ARG;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int r = 0; r < rows; ++r) {
        const int64_t n = row_ends[r] > 0 ? row_ends[r] : 0;
        const int64_t keep = n < top_k ? n : top_k;
        count_out[r] = (int32_t)keep;
        if (n == 0) continue;
        oracle_scored_key *keys = (oracle_scored_key *)malloc(sizeof(oracle_scored_key) * (size_t)n);
        if (!keys) {
            status = ORACLE_NO_MEMORY;
            continue;
        }
        for (int64_t i = 0; i < n; ++i) {
            keys[i].value = logits[(int64_t)r * row_stride + i];
            keys[i].index = (int32_t)i;
        }
        qsort(keys, (size_t)n, sizeof(oracle_scored_key), oracle_rank_cmp);
        for (int64_t i = 0; i < keep; ++i) idx_out[(int64_t)r * top_k + i] = keys[i].index;
        free(keys);
    }
    return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Threshold select: classification and fit                                                    */
/* ------------------------------------------------------------------------------------------ */

/*
 * [select] description: a key scoring above its row's threshold is a candidate; one scoring
 * neither above nor below it (equal, or NaN) is a tie.  Per row r this counts both over keys
 * 0 .. row_ends[r]-1 and decides whether the row fits:
 *   K' = min(row_ends[r], top_k);
 *   fits  iff  candidates <= capacity  and  (candidates >= K'  or
 *                                            (ties <= top_k  and  candidates + ties >= K')).
 * The pages' wording ("with at most top_k ties, reach K'") is read so that a fitting row holds
 * every tie it needs: when the candidates alone fall short, all ties must have a slot, so the
 * row's exact top-K' (ties broken by the lowest index) is determined by its slots.
 * Outputs: n_cand[r], n_tie[r] (true counts, whether or not they fit their slots), fits[r].
 */
int oracle_select_classify(const float *logits, int64_t row_stride, const int32_t *row_ends,
                           int rows, const float *thresholds, int top_k, int capacity,
                           int32_t *n_cand, int32_t *n_tie, int32_t *fits) {
    if (!logits || !row_ends || !thresholds || !n_cand || !n_tie || !fits) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        const int64_t n = row_ends[r] > 0 ? row_ends[r] : 0;
        const float thr = thresholds[r];
        int64_t cand = 0, tie = 0;
        for (int64_t i = 0; i < n; ++i) {
            const float s = logits[(int64_t)r * row_stride + i];
            if (s > thr)
                ++cand;
            else if (!(s < thr))
                ++tie;
        }
        const int64_t need = n < top_k ? n : top_k;
        n_cand[r] = (int32_t)cand;
        n_tie[r] = (int32_t)tie;
        fits[r] = cand <= capacity && (cand >= need || (tie <= top_k && cand + tie >= need));
    }
    return ORACLE_OK;
}

/*
 * Slot positions ([select] Parameters: candidates): the n-th candidate of a row goes to slot
 * top_k + n when n < capacity, the n-th tie to slot top_k - 1 - n when n < top_k; otherwise it
 * is counted but not stored.  Returns the slot, or -1 when the item is not stored.
 */
int64_t oracle_slot_of(int is_candidate, int64_t n, int top_k, int capacity) {
    if (is_candidate) return n < capacity ? top_k + n : -1;
    return n < top_k ? top_k - 1 - n : -1;
}

/* ------------------------------------------------------------------------------------------ */
/* Work split of the persistent logits kernel                                                  */
/* ------------------------------------------------------------------------------------------ */

/*
 * The [num_ctas + 1, 2] int32 schedule ([scores] Parameters: schedule_meta, opaque there) as
 * this build defines it: request b contributes ceil(seq_lens[b] / tile_tokens) work units (its
 * KV tiles, in order), U units in all, flattened request by request.  CTA c takes the flat units
 * [floor(c*U/num_ctas), floor((c+1)*U/num_ctas)).  Entry c is the (request, tile) pair of flat
 * unit floor(c*U/num_ctas): the request is the first b whose units extend past that flat index;
 * flat index U maps to (batch, 0).
 */
int oracle_schedule(const int32_t *seq_lens, int64_t seq_lens_stride, int batch, int tile_tokens,
                    int num_ctas, int32_t *out) {
    if (!seq_lens || !out || batch < 0 || tile_tokens <= 0 || num_ctas <= 0) return ORACLE_BAD_ARG;
    int64_t total = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t len = seq_lens[(int64_t)b * seq_lens_stride];
        total += (len + tile_tokens - 1) / tile_tokens;
    }
    for (int c = 0; c <= num_ctas; ++c) {
        const int64_t flat = (int64_t)c * total / num_ctas;
        int64_t before = 0;
        int request = batch, tile = 0;
        for (int b = 0; b < batch; ++b) {
            const int64_t len = seq_lens[(int64_t)b * seq_lens_stride];
            const int64_t units = (len + tile_tokens - 1) / tile_tokens;
            if (before + units > flat) {
                request = b;
                tile = (int)(flat - before);
                break;
            }
            before += units;
        }
        out[2 * c] = request;
        out[2 * c + 1] = tile;
    }
    return ORACLE_OK;
}

/* Threads the oracle's OpenMP loops use (1 when built without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
