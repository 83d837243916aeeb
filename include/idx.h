/*
 * idx.h -- C ABI of libidx.so, the GB300 (sm_103a) sparse-attention indexer.
 *
 * Two stages, each one asynchronous launch on the caller's stream:
 *   1. paged FP8 MQA logits   ("flashinfer.attn_scores", fp8_paged_mqa_logits)
 *   2. threshold top-k select  ("flashinfer.sdsa.indexer_threshold_select"), reading stage 1's
 *      logits
 * and both fused into one pass that writes no logits (idx_indexer_threshold_select), the MXFP4
 * variant of stage 1 (idx_logits_mxfp4), plus the
 * persistent work split of stage 1 ("flashinfer.attn_scores", Scheduling and Setup) and the two
 * integer helpers named there.
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are caller-owned device memory; the library never allocates,
 *     frees or synchronises, so every call can be captured in a CUDA graph once it has run
 *     eagerly one time (that first call loads the kernels); this header makes no statement
 *     either way about capturing idx_threshold_select_static.  `stream` is a cudaStream_t
 *     (NULL = the legacy default stream).
 *   - Return value: IDX_OK, or an error code; idx_last_error() then describes it.  On any
 *     error other than IDX_CUDA nothing has been launched.
 *   - Content preconditions (table width, seq_lens <= max_seq_len, page ids inside the pool)
 *     are the caller's, as on the pages; the kernels never read or write outside the buffers
 *     the arguments describe, even when they are violated (out-of-pool page ids are skipped
 *     and flagged, see idx_device_status).  With the environment variable IDX_VALIDATE=1 the
 *     logits call also copies seq_lens and block_tables to the host and checks them, returning
 *     IDX_CONTRACT on a violation (skipped while the stream is being captured, where such a
 *     copy is illegal).
 */
#ifndef IDX_H
#define IDX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IDX_OK 0
#define IDX_INVALID_ARG 1 /* null pointer, bad size/stride/alignment, inconsistent shapes */
#define IDX_UNSUPPORTED 2 /* a shape this build has no kernel for (see idx_logits_fp8) */
#define IDX_CUDA 3        /* a CUDA runtime/driver call or launch failed */
#define IDX_CONTRACT 4    /* IDX_VALIDATE=1 found a violated content precondition */

/* Element types of idx_logits_fp8's output (the pages' output_dtype). */
#define IDX_DTYPE_F32 0 /* float32 (the default on the pages) */
#define IDX_DTYPE_F16 1 /* IEEE binary16 */
#define IDX_DTYPE_BF16 2 /* bfloat16 (idx_logits_mxfp4 with head_dim 128 only; its pages' default) */

/* Device-side status bits (idx_device_status). */
#define IDX_DEV_WAIT_TIMEOUT 1 /* a pipeline wait gave up after its time limit */
#define IDX_DEV_BAD_PAGE 2     /* a needed block-table entry was outside [0, num_blocks) */
#define IDX_DEV_INEXACT_SCALE 4 /* (MXFP4) a row's block scales span more than 8 binades, or a
                                   scale byte is the NaN code 0xFF: its staging rounded */

/* Description of the most recent error on the calling thread ("" if none). */
const char *idx_last_error(void);

/*
 * padded_seq_len ("flashinfer.attn_scores", Scheduling and Setup; Example: 8000 -> 8192): the
 * minimum column count of a logits output row.  The pages give no granularity; this build
 * rounds up to a multiple of 256 (see idx_logits_fp8 for why any row stride >= this value
 * works).  Returns -1 for a negative argument.  Host-only arithmetic.
 */
int64_t idx_padded_seq_len(int64_t max_seq_len);

/*
 * min_block_table_width ("flashinfer.attn_scores", Scheduling and Setup; Parameters:
 * block_tables; Example: ceil(8000/32) = 250): ceil(seq_len / block_size), the fewest
 * block-table columns a request of seq_len tokens needs.  Returns -1 on a negative seq_len or
 * a non-positive block_size.  Host-only arithmetic.
 */
int64_t idx_min_block_table_width(int64_t seq_len, int32_t block_size);

/* The SM count of the current device (the default persistent grid).  Needs a GPU. */
int idx_num_sms(int32_t *num_sms_out);

/*
 * idx_schedule ("flashinfer.attn_scores", Parameters: schedule_meta; Scheduling and Setup):
 * the persistent logits kernel's work split, computed on the device from seq_lens' current
 * contents, so it can be captured and re-derives itself on every replay.
 *
 *   seq_lens         device int32, element b at seq_lens[b * seq_lens_stride] (stride >= 1, so
 *                    a view like seq_lens[::next_n] is taken without a copy)
 *   batch            number of requests, 0 .. 4096
 *   next_n           draft depth 1..4 (the split does not depend on it; checked for symmetry
 *                    with the logits call)
 *   num_sms          CTAs of the persistent grid, 1 .. 1024; 0 = this device's SM count
 *   schedule         device int32 [num_sms + 1][2], written: entry c is the (request, tile)
 *                    at which CTA c starts, where request b owns ceil(seq_lens[b] / 128) tiles
 *                    of 128 positions and CTA c takes the flat tiles
 *                    [floor(c*U/num_sms), floor((c+1)*U/num_sms)) of the U in all; the last
 *                    entry is (batch, 0).  Valid only while seq_lens' contents and num_sms are
 *                    unchanged; a stale one gives wrong coverage but never a hang.
 */
int idx_schedule(const int32_t *seq_lens, int64_t seq_lens_stride, int32_t batch, int32_t next_n,
                 int32_t num_sms, int32_t *schedule, void *stream);

/*
 * idx_logits_fp8 ("flashinfer.attn_scores", fp8_paged_mqa_logits: formula block, Note,
 * Parameters, Returns):
 *
 *   out[(b*next_n + t) * out_row_stride + p] =
 *       scale[p] * sum_h weights[b*next_n + t, h] * relu(q[b, t, h, :] . k[p, :])
 *
 * for every request b with seq_lens[b] > 0, slot t < next_n and position p < seq_lens[b].
 * Only p <= seq_lens[b] - next_n + t is meaningful for slot t (the pages' per-slot extent);
 * positions in [that + 1, seq_lens[b]) hold the same formula's value, columns >= seq_lens[b]
 * are not written, and rows of a request with seq_lens[b] == 0 are never written.
 *
 *   q               device e4m3 bytes [batch, next_n, num_heads, head_dim], contiguous,
 *                   16-byte aligned
 *   kv_fused        device uint8 [num_blocks][block_size*(head_dim+4)], 16-byte aligned: per
 *                   block, all e4m3 values token-major (token i at i*head_dim), then
 *                   block_size little-endian float32 scales (token i's at
 *                   block_size*head_dim + 4*i)
 *   num_blocks      blocks in the pool (>= 1; num_blocks * (block_size*(head_dim+4)/128) must
 *                   stay below 2^31)
 *   weights         device float32 [batch*next_n, num_heads], contiguous, 16-byte aligned
 *   block_tables    device int32; request b's j-th block id at block_tables[b*bt_row_stride+j];
 *                   only j < ceil(seq_lens[b]/block_size) is ever read
 *   bt_row_stride   >= bt_width (a row-strided view like block_tables[::next_n] is fine)
 *   bt_width        columns per row, >= ceil(max(seq_lens)/block_size) (caller's contract); the
 *                   first bt_width entries of every row must be mapped memory: the kernel may
 *                   prefetch them into L2 (it reads only the live ones)
 *   seq_lens        device int32, seq_lens[b * seq_lens_stride], each 0 .. max_seq_len
 *   batch           0 .. 4096
 *   next_n          1 .. 4 (draft depth; slot t = next_n - 1 is the newest and sees the whole
 *                   sequence)
 *   num_heads, head_dim   this build supports 8, 16, 32 or 64 heads of 64 or 128
 *                   (IDX_UNSUPPORTED else; the pages' restrictions num_heads % 4 == 0 and
 *                   next_n * num_heads in [8, 256] hold for all of them); kv_fused blocks are
 *                   then block_size*(head_dim+4) bytes
 *   block_size      32, 64 or 128 tokens per block (IDX_UNSUPPORTED else)
 *   max_seq_len     >= every seq_lens[b]
 *   schedule        device int32 [num_sms+1][2] from idx_schedule with the same seq_lens and
 *                   num_sms, or NULL to derive the split inside the kernel (recommended)
 *   num_sms         CTAs of the persistent grid (0 = this device's SM count)
 *   output_dtype    IDX_DTYPE_F32 or IDX_DTYPE_F16 (Parameters: output_dtype): the float32
 *                   result is converted on store, to nearest even, so a float16 output holds
 *                   +-inf where |logit| exceeds the half range; bfloat16 is not offered (as on
 *                   the pages); anything else is IDX_UNSUPPORTED
 *   out             device, output_dtype elements, rows of out_row_stride elements, 16-byte
 *                   aligned
 *   out_row_stride  >= idx_padded_seq_len(max_seq_len) and a multiple of 4 (elements)
 *   row_ends_out    NULL, or device int32 [batch*next_n] receiving
 *                   max(0, seq_lens[b] - next_n + t + 1) for every row (zero-length requests
 *                   included), ready for idx_threshold_select
 */
int idx_logits_fp8(const uint8_t *q, const uint8_t *kv_fused, int64_t num_blocks,
                   int32_t block_size, const float *weights, const int32_t *block_tables,
                   int64_t bt_row_stride, int32_t bt_width, const int32_t *seq_lens,
                   int64_t seq_lens_stride, int32_t batch, int32_t next_n, int32_t num_heads,
                   int32_t head_dim, int32_t max_seq_len, const int32_t *schedule,
                   int32_t num_sms, int32_t output_dtype, void *out, int64_t out_row_stride,
                   int32_t *row_ends_out, void *stream);

/*
 * idx_logits_mxfp4 ("flashinfer.attn_scores", fp4_paged_mqa_logits: formula block, Parameters
 * q, q_sf, kv_fused, sf_vec_size = 32):
 *
 *   out[(b*next_n + t) * out_row_stride + p] = sum_h weights[b*next_n + t, h] * relu(q . k)
 *
 * with every element of q[b,t,h,:] and k[p,:] an E2M1 value times its 32-element group's UE8M0
 * scale 2^(e - 127), and no per-position factor.  Extents, zero-length requests, block_tables,
 * seq_lens, batch, next_n, num_heads, head_dim, block_size, max_seq_len, num_sms,
 * output_dtype, out, out_row_stride and row_ends_out are as for idx_logits_fp8 (output_dtype:
 * IDX_DTYPE_F32, IDX_DTYPE_F16, or IDX_DTYPE_BF16 -- the pages' default for this variant -- with
 * head_dim 128 and 32 or 64 heads).
 *
 *   q            device uint8 [batch, next_n, num_heads, head_dim/2], 16-byte aligned: two
 *                E2M1 codes per byte, element 2j in the low nibble of byte j
 *   q_sf         device uint8 [batch, next_n, num_heads, head_dim/32]: byte k scales elements
 *                [32k, 32k + 32) (the little-endian bytes of the pages' int32 view)
 *   kv_fused     device uint8 [num_blocks][block_size*(head_dim/2 + head_dim/32)], 16-byte
 *                aligned: per block the packed rows token-major (token i at i*head_dim/2), then
 *                head_dim/32 scale bytes per token (token i's at block_size*head_dim/2 +
 *                (head_dim/32)*i)
 *   weights      device float32 [batch*next_n, num_heads]
 *   workspace    device, 256-byte aligned, at least idx_mxfp4_workspace_bytes(...) bytes
 *
 * Each row's largest block scale 2^(E - 127) leaves the row (exact: a positive power of two
 * commutes with the ReLU): a q head's multiplies the head's weight, a K token's becomes the
 * token's float32 scale, and what remains of each element is an e4m3 value.  With head_dim 128
 * and 32 or 64 heads, two launches: q and the weights are staged in the FP8 layout inside the
 * workspace, then the logits kernel loads the MXFP4 pages themselves and converts each tile to
 * e4m3 in shared memory (no staged KV pool).  Otherwise three: every KV page the batch
 * references is also staged in the workspace and idx_logits_fp8 runs on the staged tensors.
 * Either way the conversion is exact while a row's block scales span at most 8 binades; a row
 * that spans more (or holds the NaN scale byte 0xFF), or a q row whose weight times 2^(E - 127)
 * leaves float32's normal range, is rounded and raises IDX_DEV_INEXACT_SCALE.
 */
int64_t idx_mxfp4_workspace_bytes(int64_t num_blocks, int32_t block_size, int32_t batch,
                                  int32_t next_n, int32_t num_heads, int32_t head_dim);
int idx_logits_mxfp4(const uint8_t *q, const uint8_t *q_sf, const uint8_t *kv_fused,
                     int64_t num_blocks, int32_t block_size, const float *weights,
                     const int32_t *block_tables, int64_t bt_row_stride, int32_t bt_width,
                     const int32_t *seq_lens, int64_t seq_lens_stride, int32_t batch,
                     int32_t next_n, int32_t num_heads, int32_t head_dim, int32_t max_seq_len,
                     int32_t num_sms, int32_t output_dtype, void *out, int64_t out_row_stride,
                     int32_t *row_ends_out, void *workspace, int64_t workspace_bytes,
                     void *stream);

/*
 * idx_threshold_select ("flashinfer.sdsa.indexer_threshold_select": description; Parameters
 * row_ends, thresholds, counters, candidates, max_context, top_k, arrivals, ranges), over
 * logits already written by idx_logits_fp8.  One launch (two with arrivals), no host
 * synchronisation.
 *
 * For row r, key i < row_ends[r] with score s = logits[r*logits_row_stride + i] and
 * thr = thresholds[r]: s > thr makes a candidate, "neither above nor below" (s == thr or NaN)
 * a tie.  The n-th candidate is stored at slot top_k + n when n < capacity, the n-th tie at
 * slot top_k - 1 - n when n < top_k; a slot holds the pair (key index, raw float32 bits of s).
 * counters[r] counts both, stored or not; the order of stored items is unspecified.
 *
 * With K' = min(row_ends[r], top_k) a row fits when candidates <= capacity and either
 * candidates >= K' or (ties <= top_k and candidates + ties >= K'): then every item of its
 * exact top-K' (descending value, ties to the lowest index) is in its slots.
 *
 * With arrivals (and ranges), a second launch, which starts once every row's counts are final,
 * repairs each row that does not fit: it finds the row's K'-th largest score v by radix select
 * over totalOrder keys, stores the keys above v as candidates and the lowest-index keys equal
 * to v as ties (exactly K' items), and sets counters[r] to those counts and thresholds[r] = v.
 * Every row then holds its exact top-K' and ranges[0*rows + r] .. ranges[1*rows + r] (half
 * open) is the slot range holding its candidates and ties.  arrivals (as on the pages) asks for
 * the repair; no CTA counts arrivals, so its contents are never read, and the second launch sets
 * arrivals[r] = 0 for every row.
 *
 *   logits            device float32, 16-byte aligned, row stride a multiple of 4
 *   row_ends          device int32 [rows], 0 .. max_context
 *   rows              1 .. 65535
 *   thresholds        device float32 [rows], read, and written for repaired rows
 *   counters          device int32 [rows][2] (candidates, ties), ZEROED BY THE CALLER
 *   candidates        device int32 [rows][top_k + capacity][2]
 *   top_k             >= 1 (the number of tie slots)
 *   capacity          >= 0 candidate slots; >= top_k - 1 when arrivals is given
 *   max_context       the most keys a row sees, at most IDX_SELECT_MAX_CONTEXT; sizes the grid
 *                     (one CTA per 8192 keys)
 *   arrivals          NULL (no repair), or device int32 [rows] (any contents); every call
 *                     leaves it zeroed
 *   ranges            device int32 [2][rows]; required when arrivals is given, else ignored
 */
#define IDX_SELECT_MAX_CONTEXT (65535 * 8192)
int idx_threshold_select(const float *logits, int64_t logits_row_stride, const int32_t *row_ends,
                         int32_t rows, float *thresholds, int32_t *counters, int32_t *candidates,
                         int32_t top_k, int32_t capacity, int32_t max_context, int32_t *arrivals,
                         int32_t *ranges, void *stream);

/*
 * idx_threshold_select_static -- the pages have no counterpart to this entry point; it exists
 * for callers that cannot allocate device memory.
 *
 * idx_threshold_select with repair takes an `arrivals` array of one int32 per row.  Some
 * callers cannot provide one: a serving runtime that plans all of its device memory up front
 * and forbids allocation inside a step, or a plugin that has no handle on its host
 * framework's allocator and may not call cudaMalloc itself.  This entry point takes the same
 * arguments minus `arrivals` and always repairs (so `ranges` is required and capacity must be
 * >= top_k - 1); the arrival counters live in a static device array inside the library, of
 * IDX_STATIC_SELECT_MAX_ROWS int32 (64 KiB), which every GPU that loads the library holds until
 * the process exits.  It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *
 *   rows   1 .. IDX_STATIC_SELECT_MAX_ROWS; more returns IDX_INVALID_ARG with nothing launched
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current) and caches it.  Each call clears the counters it uses (an asynchronous
 * memset on `stream`) before its launches.
 * Every call, on every stream, shares the one array: calls whose work overlaps on the GPU race
 * on it and must be serialised by the caller (one stream, or events).
 */
#define IDX_STATIC_SELECT_MAX_ROWS 16384
int idx_threshold_select_static(const float *logits, int64_t logits_row_stride,
                                const int32_t *row_ends, int32_t rows, float *thresholds,
                                int32_t *counters, int32_t *candidates, int32_t top_k,
                                int32_t capacity, int32_t max_context, int32_t *ranges,
                                void *stream);

/*
 * idx_indexer_threshold_select ("flashinfer.sdsa.indexer_threshold_select": description;
 * Parameters thresholds, counters, candidates, top_k, arrivals, ranges): the logits of
 * idx_logits_fp8 and the selection of idx_threshold_select in one pass over each request's
 * paged keys, without writing the scores.  The rows are those of idx_logits_fp8 (row
 * b*next_n + t sees keys p < max(0, seq_lens[b] - next_n + t + 1)), and every output --
 * counters, the slot contents (as sets), ranges, repaired thresholds -- equals what
 * idx_logits_fp8 (float32) followed by idx_threshold_select with those row ends would give:
 * each score is computed by the same arithmetic, then classified instead of stored.
 *
 * The pages' query "tile" is here one request: its next_n * 64 query-head rows are the tensor
 * core's N side.
 *
 * Without arrivals: one launch; the rows' counts and slots only (rows that do not fit are not
 * repaired, and ranges is not written).
 * With arrivals: every row fits on return.  Three launches on `stream`, no host
 * synchronisation (capturable once run eagerly):
 *   1. the fused pass: every score classified into its row's slots;
 *   2. the logits of every request with a row that does not fit (the fit rule applied to the
 *      counts of launch 1) recomputed into `scratch` (float32, by the same kernel; every other
 *      request counts as empty, so nothing else is read or written);
 *   3. per row: the slot range of a row that fits, else the radix repair of
 *      idx_threshold_select from its scratch row.
 * When no row needs a repair, launch 2 reads only seq_lens and counters.  The follow-up
 * launches start after the fused pass has finished, so no arrival counting is needed: arrivals
 * is the switch that asks for the repair (as on the pages), and is neither read nor written.
 *
 * q, kv_fused, num_blocks, block_size, weights, block_tables, bt_row_stride, bt_width,
 * seq_lens, seq_lens_stride, batch, next_n, num_heads, head_dim, max_seq_len, num_sms
 *                     as for idx_logits_fp8 (the work split is always derived in the kernel)
 *   thresholds        device float32 [batch*next_n], read, and written for repaired rows
 *   counters          device int32 [batch*next_n][2] (candidates, ties), ZEROED BY THE CALLER,
 *                     8-byte aligned
 *   candidates        device int32 [batch*next_n][top_k + capacity][2], 8-byte aligned
 *   top_k, capacity   as for idx_threshold_select (capacity >= top_k - 1 with arrivals)
 *   arrivals          NULL (no repair), or any non-NULL device pointer (repair); untouched
 *   ranges            device int32 [2][batch*next_n]; required with arrivals
 *   scratch           device float32, 16-byte aligned, rows of scratch_row_stride elements
 *                     (>= idx_padded_seq_len(max_seq_len), a multiple of 4); required with
 *                     arrivals; only rows of requests that need a repair are written
 */
int idx_indexer_threshold_select(const uint8_t *q, const uint8_t *kv_fused, int64_t num_blocks,
                                 int32_t block_size, const float *weights,
                                 const int32_t *block_tables, int64_t bt_row_stride,
                                 int32_t bt_width, const int32_t *seq_lens,
                                 int64_t seq_lens_stride, int32_t batch, int32_t next_n,
                                 int32_t num_heads, int32_t head_dim, int32_t max_seq_len,
                                 int32_t num_sms, float *thresholds, int32_t *counters,
                                 int32_t *candidates, int32_t top_k, int32_t capacity,
                                 int32_t *arrivals, int32_t *ranges, float *scratch,
                                 int64_t scratch_row_stride, void *stream);

/*
 * idx_debug_withhold_first_tile -- fault injection for testing the time-limited pipeline waits
 * (the pages have no counterpart).  From the next logits launch on (idx_logits_fp8,
 * idx_logits_mxfp4, and the scoring passes of idx_indexer_threshold_select), the CTA of index
 * `cta` of the persistent grid issues none of the copies of the first tile of its run, so the
 * waits on that tile run out after their limit (one second): that CTA's roles give up, it drains
 * every copy it did issue, frees its tensor memory and exits, and IDX_DEV_WAIT_TIMEOUT is raised
 * (idx_device_status).  The launch's output is then incomplete.  `cta` = -1 switches it off (the
 * default).  Synchronous; for tests only, never for production use.
 * Returns IDX_INVALID_ARG for cta outside -1 .. 1023.
 */
int idx_debug_withhold_first_tile(int32_t cta);

/*
 * Reads (and, if clear != 0, resets) the OR of the device-side status bits (IDX_DEV_*) that
 * every kernel of this library has raised on the current device since the last reset.
 * Synchronous (it copies from the device); a debugging aid, not for the hot path.
 */
int idx_device_status(int32_t *status_out, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H */
