// abi.cu -- the extern "C" entry points declared in include/idx.h: argument checks, status
// codes, TMA tensor-map encoding and launches.  No allocation, no synchronisation (except in the
// opt-in IDX_VALIDATE mode and the debugging call idx_device_status).

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/idx.h"
#include "internal.h"
#include "mxfp4.h"

#define IDX_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_error;

int fail(int code, const std::string &msg) {
  g_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char *what) {
  g_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return IDX_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, resolved through the runtime so the library needs no libcuda link.
EncodeTiled encode_tiled() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// A 2-D uint8 tensor of `rows` rows of `row_bytes` = 128 or 64 bytes (one e4m3 row of head_dim
// elements), read in boxes of `box_rows` rows with the 128- or 64-byte swizzle: the layout the
// tensor core's descriptors expect.
int encode_rows(CUtensorMap *map, const void *base, uint64_t rows, uint32_t row_bytes,
                uint32_t box_rows) {
  EncodeTiled fn = encode_tiled();
  if (fn == nullptr) return fail(IDX_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {row_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(IDX_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return IDX_OK;
}

// head_dim 192: the pool as [num_blocks][block_size tokens][3 K blocks][64 bytes] (page stride
// block_size * 196 bytes: the tokens' values, then their scales) and q as [rows][3][64], each read
// one K block at a time ([tokens or rows] x 64 bytes) with the 64-byte swizzle.
int encode_kblocks_kv(CUtensorMap *map, const void *base, uint64_t num_blocks,
                      uint32_t block_size) {
  EncodeTiled fn = encode_tiled();
  if (fn == nullptr) return fail(IDX_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[4] = {64, 3, block_size, num_blocks};
  const cuuint64_t strides[3] = {64, 192, static_cast<cuuint64_t>(block_size) * 196};
  const cuuint32_t box[4] = {64, 1, block_size, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(IDX_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return IDX_OK;
}

int encode_kblocks_q(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
  EncodeTiled fn = encode_tiled();
  if (fn == nullptr) return fail(IDX_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {64, 3, rows};
  const cuuint64_t strides[2] = {64, 192};
  const cuuint32_t box[3] = {64, 1, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(IDX_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return IDX_OK;
}

int resolve_sms(int32_t requested, int32_t *out) {
  if (requested < 0 || requested > 1024) return fail(IDX_INVALID_ARG, "num_sms must be 0..1024");
  if (requested > 0) {
    *out = requested;
    return IDX_OK;
  }
  int dev = 0, n = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  *out = n;
  return IDX_OK;
}

bool validate_requested() {
  const char *v = std::getenv("IDX_VALIDATE");
  return v != nullptr && v[0] == '1';
}

// IDX_VALIDATE=1: the content preconditions of the logits call, checked on host copies.
int validate_logits_contents(const int32_t *block_tables, int64_t bt_row_stride, int32_t bt_width,
                             const int32_t *seq_lens, int64_t seq_lens_stride, int32_t batch,
                             int32_t max_seq_len, int64_t num_blocks, int32_t block_size,
                             cudaStream_t stream) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone) return IDX_OK;  // a D2H copy is illegal under capture
  std::vector<int32_t> lens(batch);
  std::vector<int32_t> table(static_cast<size_t>(batch) * bt_width);
  e = cudaMemcpy2DAsync(lens.data(), 4, seq_lens, static_cast<size_t>(seq_lens_stride) * 4, 4,
                        batch, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess && bt_width > 0)
    e = cudaMemcpy2DAsync(table.data(), static_cast<size_t>(bt_width) * 4, block_tables,
                          static_cast<size_t>(bt_row_stride) * 4,
                          static_cast<size_t>(bt_width) * 4, batch, cudaMemcpyDeviceToHost,
                          stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "IDX_VALIDATE copy");
  for (int b = 0; b < batch; ++b) {
    const int64_t len = lens[b];
    if (len < 0 || len > max_seq_len)
      return fail(IDX_CONTRACT, "seq_lens[" + std::to_string(b) + "] = " + std::to_string(len) +
                                    " is outside [0, max_seq_len]");
    const int64_t pages = (len + block_size - 1) / block_size;
    if (pages > bt_width)
      return fail(IDX_CONTRACT, "block table width " + std::to_string(bt_width) +
                                    " < ceil(seq_lens[" + std::to_string(b) + "] / " +
                                    std::to_string(block_size) + ")");
    for (int64_t j = 0; j < pages; ++j) {
      const int32_t id = table[static_cast<size_t>(b) * bt_width + j];
      if (id < 0 || id >= num_blocks)
        return fail(IDX_CONTRACT, "block_tables[" + std::to_string(b) + ", " +
                                      std::to_string(j) + "] = " + std::to_string(id) +
                                      " is outside the pool");
    }
  }
  return IDX_OK;
}

}  // namespace

IDX_EXPORT const char *idx_last_error(void) { return g_error.c_str(); }

IDX_EXPORT int64_t idx_padded_seq_len(int64_t max_seq_len) {
  if (max_seq_len < 0) return -1;
  return (max_seq_len + 255) / 256 * 256;
}

IDX_EXPORT int64_t idx_min_block_table_width(int64_t seq_len, int32_t block_size) {
  if (seq_len < 0 || block_size <= 0) return -1;
  return seq_len / block_size + (seq_len % block_size != 0 ? 1 : 0);
}

IDX_EXPORT int idx_num_sms(int32_t *num_sms_out) {
  if (num_sms_out == nullptr) return fail(IDX_INVALID_ARG, "num_sms_out is NULL");
  g_error.clear();
  return resolve_sms(0, num_sms_out);
}

IDX_EXPORT int idx_schedule(const int32_t *seq_lens, int64_t seq_lens_stride, int32_t batch,
                            int32_t next_n, int32_t num_sms, int32_t *schedule, void *stream) {
  g_error.clear();
  if (seq_lens == nullptr || schedule == nullptr)
    return fail(IDX_INVALID_ARG, "seq_lens and schedule must not be NULL");
  if (seq_lens_stride < 1) return fail(IDX_INVALID_ARG, "seq_lens_stride must be >= 1");
  if (batch < 0) return fail(IDX_INVALID_ARG, "batch must be >= 0");
  if (next_n < 1 || next_n > 4) return fail(IDX_UNSUPPORTED, "next_n must be 1..4");
  if (batch > idx::kMaxBatch) return fail(IDX_UNSUPPORTED, "batch above 4096");
  int32_t ctas = 0;
  int st = resolve_sms(num_sms, &ctas);
  if (st != IDX_OK) return st;
  const cudaError_t e = idx::launch_schedule(seq_lens, seq_lens_stride, batch, ctas, schedule,
                                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "schedule launch");
  return IDX_OK;
}

IDX_EXPORT int idx_logits_fp8(const uint8_t *q, const uint8_t *kv_fused, int64_t num_blocks,
                              int32_t block_size, const float *weights,
                              const int32_t *block_tables, int64_t bt_row_stride,
                              int32_t bt_width, const int32_t *seq_lens, int64_t seq_lens_stride,
                              int32_t batch, int32_t next_n, int32_t num_heads, int32_t head_dim,
                              int32_t max_seq_len, const int32_t *schedule, int32_t num_sms,
                              int32_t output_dtype, void *out, int64_t out_row_stride,
                              int32_t *row_ends_out, void *stream) {
  g_error.clear();
  if (q == nullptr || kv_fused == nullptr || weights == nullptr || block_tables == nullptr ||
      seq_lens == nullptr || out == nullptr)
    return fail(IDX_INVALID_ARG, "q, kv_fused, weights, block_tables, seq_lens, out: NULL");
  if (batch < 0 || max_seq_len < 0 || num_blocks < 1 || bt_width < 0 || seq_lens_stride < 1 ||
      bt_row_stride < bt_width || block_size <= 0 || num_heads <= 0 || head_dim <= 0 ||
      next_n <= 0)
    return fail(IDX_INVALID_ARG, "negative or inconsistent size or stride");
  if ((num_heads != 8 && num_heads != 16 && num_heads != 32 && num_heads != 64) ||
      (head_dim != 64 && head_dim != 128 && head_dim != 192) ||
      (block_size != 32 && block_size != 64 && block_size != 128) ||
      (head_dim == 192 && num_heads != 32 && num_heads != 64))
    return fail(IDX_UNSUPPORTED, "this build supports num_heads 8, 16, 32 or 64 with head_dim 64 "
                                 "or 128, and 32 or 64 heads with head_dim 192; block_size 32, 64 "
                                 "or 128");
  if (next_n > 4) return fail(IDX_UNSUPPORTED, "next_n must be 1..4");
  if (output_dtype != IDX_DTYPE_F32 && output_dtype != IDX_DTYPE_F16)
    return fail(IDX_UNSUPPORTED, "output_dtype must be IDX_DTYPE_F32 or IDX_DTYPE_F16");
  if (batch > idx::kMaxBatch) return fail(IDX_UNSUPPORTED, "batch above 4096");
  if (out_row_stride < idx_padded_seq_len(max_seq_len) || out_row_stride % 4 != 0)
    return fail(IDX_INVALID_ARG,
                "out_row_stride must be >= idx_padded_seq_len(max_seq_len) and a multiple of 4");
  const int64_t page_bytes = static_cast<int64_t>(block_size) * (head_dim + 4);
  if (head_dim != 192 && num_blocks > (INT64_C(1) << 31) / (page_bytes / head_dim) - 1)
    return fail(IDX_INVALID_ARG, "num_blocks too large for 32-bit TMA row coordinates");
  if (head_dim == 192 && num_blocks >= (INT64_C(1) << 31))
    return fail(IDX_INVALID_ARG, "num_blocks too large for 32-bit TMA coordinates");
  if (!aligned(q, 16) || !aligned(kv_fused, 16) || !aligned(weights, 16) || !aligned(out, 16))
    return fail(IDX_INVALID_ARG, "q, kv_fused, weights and out must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
      (row_ends_out != nullptr && !aligned(row_ends_out, 4)) ||
      (schedule != nullptr && !aligned(schedule, 4)))
    return fail(IDX_INVALID_ARG, "int32 arguments must be 4-byte aligned");
  int32_t ctas = 0;
  int st = resolve_sms(num_sms, &ctas);
  if (st != IDX_OK) return st;
  if (batch == 0) return IDX_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (validate_requested()) {
    st = validate_logits_contents(block_tables, bt_row_stride, bt_width, seq_lens,
                                  seq_lens_stride, batch, max_seq_len, num_blocks, block_size, s);
    if (st != IDX_OK) return st;
  }
  CUtensorMap kv_map, q_map;
  // The kernel loads a request's q rows rounded up to a multiple of 16 (the MMA's N).
  const uint32_t q_box = static_cast<uint32_t>((next_n * num_heads + 15) / 16 * 16);
  const uint64_t q_rows = static_cast<uint64_t>(batch) * next_n * num_heads;
  if (head_dim == 192) {
    st = encode_kblocks_kv(&kv_map, kv_fused, static_cast<uint64_t>(num_blocks),
                           static_cast<uint32_t>(block_size));
    if (st != IDX_OK) return st;
    st = encode_kblocks_q(&q_map, q, q_rows, q_box);
  } else {
    st = encode_rows(&kv_map, kv_fused,
                     static_cast<uint64_t>(num_blocks) * (page_bytes / head_dim),
                     static_cast<uint32_t>(head_dim), static_cast<uint32_t>(block_size));
    if (st != IDX_OK) return st;
    st = encode_rows(&q_map, q, q_rows, static_cast<uint32_t>(head_dim), q_box);
  }
  if (st != IDX_OK) return st;
  idx::LogitsArgs a{};
  a.kv = kv_fused;
  a.weights = weights;
  a.block_tables = block_tables;
  a.bt_stride = bt_row_stride;
  a.bt_width = bt_width;
  a.seq_lens = seq_lens;
  a.sl_stride = seq_lens_stride;
  a.schedule = schedule;
  a.out = out;
  a.out_stride = out_row_stride;
  a.row_ends = row_ends_out;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.batch = batch;
  const cudaError_t e = idx::launch_logits_fp8(
      next_n, output_dtype == IDX_DTYPE_F16 ? idx::LogitsOut::kF16 : idx::LogitsOut::kF32, kv_map,
      q_map, a, ctas, s);
  if (e != cudaSuccess) return cuda_fail(e, "logits launch");
  return IDX_OK;
}

IDX_EXPORT int64_t idx_mxfp4_workspace_bytes(int64_t num_blocks, int32_t block_size,
                                              int32_t batch, int32_t next_n, int32_t num_heads,
                                              int32_t head_dim) {
  if (num_blocks < 0 || block_size <= 0 || batch < 0 || next_n <= 0 || num_heads <= 0 ||
      head_dim <= 0)
    return -1;
  const auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t rows_heads = static_cast<int64_t>(batch) * next_n * num_heads;
  // head_dim 128 with 32 or 64 heads: the KV pages are converted on chip, only q and the
  // weights are staged.
  const bool on_chip = head_dim == 128 && (num_heads == 32 || num_heads == 64);
  const int64_t kv = on_chip ? 0 : up(num_blocks * block_size * (head_dim + 4));
  return kv + up(rows_heads * head_dim) + up(rows_heads * 4);
}

IDX_EXPORT int idx_logits_mxfp4(const uint8_t *q, const uint8_t *q_sf, const uint8_t *kv_fused,
                                int64_t num_blocks, int32_t block_size, const float *weights,
                                const int32_t *block_tables, int64_t bt_row_stride,
                                int32_t bt_width, const int32_t *seq_lens,
                                int64_t seq_lens_stride, int32_t batch, int32_t next_n,
                                int32_t num_heads, int32_t head_dim, int32_t max_seq_len,
                                int32_t num_sms, int32_t output_dtype, void *out,
                                int64_t out_row_stride, int32_t *row_ends_out, void *workspace,
                                int64_t workspace_bytes, void *stream) {
  g_error.clear();
  if (q == nullptr || q_sf == nullptr || kv_fused == nullptr || weights == nullptr ||
      block_tables == nullptr || seq_lens == nullptr || out == nullptr || workspace == nullptr)
    return fail(IDX_INVALID_ARG,
                "q, q_sf, kv_fused, weights, block_tables, seq_lens, out, workspace: NULL");
  if (batch < 0 || max_seq_len < 0 || num_blocks < 1 || bt_width < 0 || seq_lens_stride < 1 ||
      bt_row_stride < bt_width || block_size <= 0 || num_heads <= 0 || head_dim <= 0 ||
      next_n <= 0)
    return fail(IDX_INVALID_ARG, "negative or inconsistent size or stride");
  if ((num_heads != 8 && num_heads != 16 && num_heads != 32 && num_heads != 64) ||
      (head_dim != 64 && head_dim != 128) ||
      (block_size != 32 && block_size != 64 && block_size != 128))
    return fail(IDX_UNSUPPORTED, "this build supports num_heads 8, 16, 32 or 64, head_dim 64 or "
                                 "128, block_size 32, 64 or 128");
  if (next_n > 4) return fail(IDX_UNSUPPORTED, "next_n must be 1..4");
  if (batch > idx::kMaxBatch) return fail(IDX_UNSUPPORTED, "batch above 4096");
  const int64_t need = idx_mxfp4_workspace_bytes(num_blocks, block_size, batch, next_n,
                                                 num_heads, head_dim);
  if (workspace_bytes < need)
    return fail(IDX_INVALID_ARG, "workspace_bytes < idx_mxfp4_workspace_bytes(...) = " +
                                     std::to_string(need));
  if (!aligned(q, 16) || !aligned(kv_fused, 16) || !aligned(workspace, 256) ||
      !aligned(weights, 4))
    return fail(IDX_INVALID_ARG, "q and kv_fused must be 16-byte aligned, workspace 256-byte");
  // The KV pages converted inside the logits kernel (head_dim 128, 32 or 64 heads); otherwise
  // staged in the workspace for the FP8 kernel.
  const bool on_chip = head_dim == 128 && (num_heads == 32 || num_heads == 64);
  if (output_dtype != IDX_DTYPE_F32 && output_dtype != IDX_DTYPE_F16 &&
      !(on_chip && output_dtype == IDX_DTYPE_BF16))
    return fail(IDX_UNSUPPORTED, "output_dtype must be IDX_DTYPE_F32, IDX_DTYPE_F16 or (head_dim "
                                 "128, 32 or 64 heads) IDX_DTYPE_BF16");
  if (out_row_stride < idx_padded_seq_len(max_seq_len) || out_row_stride % 4 != 0)
    return fail(IDX_INVALID_ARG,
                "out_row_stride must be >= idx_padded_seq_len(max_seq_len) and a multiple of 4");
  if (!aligned(out, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
      (row_ends_out != nullptr && !aligned(row_ends_out, 4)))
    return fail(IDX_INVALID_ARG, "out must be 16-byte aligned, int32 arguments 4-byte aligned");
  const int64_t raw_page = static_cast<int64_t>(block_size) * (head_dim / 2 + head_dim / 32);
  if (num_blocks > INT64_MAX / raw_page) return fail(IDX_INVALID_ARG, "num_blocks too large");
  int32_t ctas = 0;
  int st = resolve_sms(num_sms, &ctas);
  if (st != IDX_OK) return st;
  if (batch == 0) return IDX_OK;
  const auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t rows_heads = static_cast<int64_t>(batch) * next_n * num_heads;
  uint8_t *kv8 = static_cast<uint8_t *>(workspace);
  uint8_t *q8 = kv8 + (on_chip ? 0 : up(num_blocks * block_size * (head_dim + 4)));
  float *w8 = reinterpret_cast<float *>(q8 + up(rows_heads * head_dim));
  idx::Mxfp4Stage stg{};
  stg.q4 = q;
  stg.q_sf = q_sf;
  stg.weights = weights;
  stg.kv4 = kv_fused;
  stg.block_tables = block_tables;
  stg.bt_stride = bt_row_stride;
  stg.seq_lens = seq_lens;
  stg.sl_stride = seq_lens_stride;
  stg.q8 = q8;
  stg.w8 = w8;
  stg.kv8 = kv8;
  stg.num_blocks = num_blocks;
  stg.rows_heads = static_cast<int32_t>(rows_heads);
  stg.block_size = block_size;
  stg.head_dim = head_dim;
  stg.batch = batch;
  stg.max_pages = static_cast<int32_t>((static_cast<int64_t>(max_seq_len) + block_size - 1) /
                                      block_size);
  stg.stage_kv = !on_chip;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (on_chip && validate_requested()) {
    st = validate_logits_contents(block_tables, bt_row_stride, bt_width, seq_lens,
                                  seq_lens_stride, batch, max_seq_len, num_blocks, block_size, s);
    if (st != IDX_OK) return st;
  }
  cudaError_t e = idx::launch_mxfp4_stage(stg, s);
  if (e != cudaSuccess) return cuda_fail(e, "MXFP4 staging launch");
  if (on_chip) {
    // q (staged) through TMA; the KV pages converted by the logits kernel's converter warps.
    CUtensorMap q_map;
    st = encode_rows(&q_map, q8, static_cast<uint64_t>(rows_heads), 128u,
                     static_cast<uint32_t>(next_n * num_heads));
    if (st != IDX_OK) return st;
    idx::LogitsArgs a{};
    a.kv = kv_fused;
    a.weights = w8;
    a.block_tables = block_tables;
    a.bt_stride = bt_row_stride;
    a.bt_width = bt_width;
    a.seq_lens = seq_lens;
    a.sl_stride = seq_lens_stride;
    a.out = out;
    a.out_stride = out_row_stride;
    a.row_ends = row_ends_out;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.num_heads = num_heads;
    a.head_dim = head_dim;
    a.batch = batch;
    e = idx::launch_logits_mxfp4(next_n, output_dtype, q_map, a, ctas, s);
    if (e != cudaSuccess) return cuda_fail(e, "MXFP4 logits launch");
    return IDX_OK;
  }
  // The staged tensors are in the FP8 layouts: the FP8 logits path computes the logits.
  return idx_logits_fp8(q8, kv8, num_blocks, block_size, w8, block_tables, bt_row_stride,
                        bt_width, seq_lens, seq_lens_stride, batch, next_n, num_heads, head_dim,
                        max_seq_len, nullptr, num_sms, output_dtype, out, out_row_stride,
                        row_ends_out, stream);
}

IDX_EXPORT int idx_indexer_threshold_select(
    const uint8_t *q, const uint8_t *kv_fused, int64_t num_blocks, int32_t block_size,
    const float *weights, const int32_t *block_tables, int64_t bt_row_stride, int32_t bt_width,
    const int32_t *seq_lens, int64_t seq_lens_stride, int32_t batch, int32_t next_n,
    int32_t num_heads, int32_t head_dim, int32_t max_seq_len, int32_t num_sms, float *thresholds,
    int32_t *counters, int32_t *candidates, int32_t top_k, int32_t capacity, int32_t *arrivals,
    int32_t *ranges, float *scratch, int64_t scratch_row_stride, void *stream) {
  g_error.clear();
  if (q == nullptr || kv_fused == nullptr || weights == nullptr || block_tables == nullptr ||
      seq_lens == nullptr || thresholds == nullptr || counters == nullptr || candidates == nullptr)
    return fail(IDX_INVALID_ARG,
                "q, kv_fused, weights, block_tables, seq_lens, thresholds, counters, "
                "candidates: NULL");
  if (batch < 0 || max_seq_len < 0 || num_blocks < 1 || bt_width < 0 || seq_lens_stride < 1 ||
      bt_row_stride < bt_width || block_size <= 0 || num_heads <= 0 || head_dim <= 0 ||
      next_n <= 0)
    return fail(IDX_INVALID_ARG, "negative or inconsistent size or stride");
  if ((num_heads != 32 && num_heads != 64) || (head_dim != 64 && head_dim != 128) ||
      (block_size != 32 && block_size != 64 && block_size != 128))
    return fail(IDX_UNSUPPORTED, "this build supports num_heads 32 or 64, head_dim 64 or 128, "
                                 "block_size 32, 64 or 128");
  if (next_n > 4) return fail(IDX_UNSUPPORTED, "next_n must be 1..4");
  if (batch > idx::kMaxBatch) return fail(IDX_UNSUPPORTED, "batch above 4096");
  if (top_k < 1 || capacity < 0 || static_cast<int64_t>(top_k) + capacity > (INT32_MAX / 2))
    return fail(IDX_INVALID_ARG, "top_k >= 1 and capacity >= 0 required");
  const int64_t page_bytes = static_cast<int64_t>(block_size) * (head_dim + 4);
  if (num_blocks > (INT64_C(1) << 31) / (page_bytes / head_dim) - 1)
    return fail(IDX_INVALID_ARG, "num_blocks too large for 32-bit TMA row coordinates");
  if (!aligned(q, 16) || !aligned(kv_fused, 16) || !aligned(weights, 16))
    return fail(IDX_INVALID_ARG, "q, kv_fused and weights must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(thresholds, 4) ||
      !aligned(counters, 8) || !aligned(candidates, 8) ||
      (arrivals != nullptr && !aligned(arrivals, 4)) || (ranges != nullptr && !aligned(ranges, 4)))
    return fail(IDX_INVALID_ARG,
                "counters and candidates must be 8-byte aligned, other int32/float32 4-byte");
  if (arrivals != nullptr) {
    if (ranges == nullptr || scratch == nullptr)
      return fail(IDX_INVALID_ARG, "ranges and scratch are required with arrivals");
    if (capacity < top_k - 1)
      return fail(IDX_INVALID_ARG, "with arrivals, capacity must be >= top_k - 1");
    if (scratch_row_stride < idx_padded_seq_len(max_seq_len) || scratch_row_stride % 4 != 0 ||
        !aligned(scratch, 16))
      return fail(IDX_INVALID_ARG,
                  "scratch must be 16-byte aligned with a row stride >= "
                  "idx_padded_seq_len(max_seq_len), a multiple of 4");
  }
  int32_t ctas = 0;
  int st = resolve_sms(num_sms, &ctas);
  if (st != IDX_OK) return st;
  if (batch == 0) return IDX_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (validate_requested()) {
    st = validate_logits_contents(block_tables, bt_row_stride, bt_width, seq_lens,
                                  seq_lens_stride, batch, max_seq_len, num_blocks, block_size, s);
    if (st != IDX_OK) return st;
  }
  CUtensorMap kv_map, q_map;
  st = encode_rows(&kv_map, kv_fused,
                   static_cast<uint64_t>(num_blocks) * (page_bytes / head_dim),
                   static_cast<uint32_t>(head_dim), static_cast<uint32_t>(block_size));
  if (st != IDX_OK) return st;
  st = encode_rows(&q_map, q, static_cast<uint64_t>(batch) * next_n * num_heads,
                   static_cast<uint32_t>(head_dim), static_cast<uint32_t>(next_n * num_heads));
  if (st != IDX_OK) return st;
  idx::LogitsArgs a{};
  a.kv = kv_fused;
  a.weights = weights;
  a.block_tables = block_tables;
  a.bt_stride = bt_row_stride;
  a.bt_width = bt_width;
  a.seq_lens = seq_lens;
  a.sl_stride = seq_lens_stride;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.batch = batch;
  a.thresholds = thresholds;
  a.counters = counters;
  a.candidates = candidates;
  a.top_k = top_k;
  a.capacity = capacity;
  // 1. Every score classified into its row's slots.
  cudaError_t e = idx::launch_logits_fp8(next_n, idx::LogitsOut::kSelect, kv_map, q_map, a, ctas, s);
  if (e != cudaSuccess) return cuda_fail(e, "fused logits launch");
  if (arrivals == nullptr) return IDX_OK;
  // 2. The scores of every request with a row that does not fit, this time stored (the other
  // requests count as empty, and the work split covers only these).
  idx::LogitsArgs r{};
  r.kv = kv_fused;
  r.weights = weights;
  r.block_tables = block_tables;
  r.bt_stride = bt_row_stride;
  r.bt_width = bt_width;
  r.seq_lens = seq_lens;
  r.sl_stride = seq_lens_stride;
  r.num_blocks = num_blocks;
  r.block_size = block_size;
  r.num_heads = num_heads;
  r.head_dim = head_dim;
  r.batch = batch;
  r.out = scratch;
  r.out_stride = scratch_row_stride;
  r.fit_counters = counters;
  r.top_k = top_k;
  r.capacity = capacity;
  e = idx::launch_logits_fp8(next_n, idx::LogitsOut::kF32, kv_map, q_map, r, ctas, s);
  if (e != cudaSuccess) return cuda_fail(e, "rescoring launch");
  // 3. Each row's slot range, after the radix repair of a row that does not fit from its
  // rescored logits.
  idx::FusedRepairArgs f{};
  f.scratch = scratch;
  f.scratch_stride = scratch_row_stride;
  f.seq_lens = seq_lens;
  f.sl_stride = seq_lens_stride;
  f.thresholds = thresholds;
  f.counters = counters;
  f.candidates = candidates;
  f.ranges = ranges;
  f.batch = batch;
  f.next_n = next_n;
  f.top_k = top_k;
  f.capacity = capacity;
  e = idx::launch_fused_repair(f, s);
  if (e != cudaSuccess) return cuda_fail(e, "repair launch");
  return IDX_OK;
}

IDX_EXPORT int idx_threshold_select(const float *logits, int64_t logits_row_stride,
                                    const int32_t *row_ends, int32_t rows, float *thresholds,
                                    int32_t *counters, int32_t *candidates, int32_t top_k,
                                    int32_t capacity, int32_t max_context, int32_t *arrivals,
                                    int32_t *ranges, void *stream) {
  g_error.clear();
  if (logits == nullptr || row_ends == nullptr || thresholds == nullptr || counters == nullptr ||
      candidates == nullptr)
    return fail(IDX_INVALID_ARG, "logits, row_ends, thresholds, counters, candidates: NULL");
  if (rows < 0 || rows > 65535) return fail(IDX_INVALID_ARG, "rows must be 0..65535");
  if (top_k < 1 || capacity < 0 || max_context < 0 ||
      static_cast<int64_t>(top_k) + capacity > (INT32_MAX / 2))
    return fail(IDX_INVALID_ARG, "top_k >= 1, capacity >= 0, max_context >= 0 required");
  if (logits_row_stride < max_context || logits_row_stride % 4 != 0)
    return fail(IDX_INVALID_ARG, "logits_row_stride must be >= max_context and a multiple of 4");
  if (max_context > IDX_SELECT_MAX_CONTEXT)
    return fail(IDX_INVALID_ARG, "max_context must be <= IDX_SELECT_MAX_CONTEXT (65535 * 8192)");
  if (!aligned(logits, 16)) return fail(IDX_INVALID_ARG, "logits must be 16-byte aligned");
  if (!aligned(candidates, 8) || !aligned(counters, 4) || !aligned(thresholds, 4) ||
      !aligned(row_ends, 4))
    return fail(IDX_INVALID_ARG, "candidates must be 8-byte aligned, int32/float32 4-byte");
  if (arrivals != nullptr) {
    if (ranges == nullptr) return fail(IDX_INVALID_ARG, "ranges is required with arrivals");
    if (capacity < top_k - 1)
      return fail(IDX_INVALID_ARG, "with arrivals, capacity must be >= top_k - 1");
  }
  if (rows == 0) return IDX_OK;
  idx::SelectArgs a;
  a.logits = logits;
  a.row_stride = logits_row_stride;
  a.row_ends = row_ends;
  a.thresholds = thresholds;
  a.counters = counters;
  a.candidates = candidates;
  a.arrivals = arrivals;
  a.ranges = ranges;
  a.rows = rows;
  a.top_k = top_k;
  a.capacity = capacity;
  a.max_context = max_context;
  const cudaError_t e = idx::launch_threshold_select(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "select launch");
  return IDX_OK;
}

IDX_EXPORT int idx_threshold_select_static(const float *logits, int64_t logits_row_stride,
                                           const int32_t *row_ends, int32_t rows,
                                           float *thresholds, int32_t *counters,
                                           int32_t *candidates, int32_t top_k, int32_t capacity,
                                           int32_t max_context, int32_t *ranges, void *stream) {
  g_error.clear();
  if (logits == nullptr || row_ends == nullptr || thresholds == nullptr || counters == nullptr ||
      candidates == nullptr || ranges == nullptr)
    return fail(IDX_INVALID_ARG,
                "logits, row_ends, thresholds, counters, candidates, ranges: NULL");
  if (rows < 0 || rows > IDX_STATIC_SELECT_MAX_ROWS)
    return fail(IDX_INVALID_ARG, "rows must be 0.." + std::to_string(IDX_STATIC_SELECT_MAX_ROWS) +
                                     ": the library's static arrival counters hold " +
                                     std::to_string(IDX_STATIC_SELECT_MAX_ROWS) + " rows");
  if (top_k < 1 || capacity < 0 || max_context < 0 ||
      static_cast<int64_t>(top_k) + capacity > (INT32_MAX / 2))
    return fail(IDX_INVALID_ARG, "top_k >= 1, capacity >= 0, max_context >= 0 required");
  if (capacity < top_k - 1) return fail(IDX_INVALID_ARG, "capacity must be >= top_k - 1");
  if (logits_row_stride < max_context || logits_row_stride % 4 != 0)
    return fail(IDX_INVALID_ARG, "logits_row_stride must be >= max_context and a multiple of 4");
  if (max_context > IDX_SELECT_MAX_CONTEXT)
    return fail(IDX_INVALID_ARG, "max_context must be <= IDX_SELECT_MAX_CONTEXT (65535 * 8192)");
  if (!aligned(logits, 16)) return fail(IDX_INVALID_ARG, "logits must be 16-byte aligned");
  if (!aligned(candidates, 8) || !aligned(counters, 4) || !aligned(thresholds, 4) ||
      !aligned(row_ends, 4) || !aligned(ranges, 4))
    return fail(IDX_INVALID_ARG, "candidates must be 8-byte aligned, int32/float32 4-byte");
  if (rows == 0) return IDX_OK;
  idx::SelectArgs a;
  a.logits = logits;
  a.row_stride = logits_row_stride;
  a.row_ends = row_ends;
  a.thresholds = thresholds;
  a.counters = counters;
  a.candidates = candidates;
  a.arrivals = nullptr;  // replaced by the static array
  a.ranges = ranges;
  a.rows = rows;
  a.top_k = top_k;
  a.capacity = capacity;
  a.max_context = max_context;
  const cudaError_t e =
      idx::launch_threshold_select_static(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "static select launch");
  return IDX_OK;
}

IDX_EXPORT int idx_debug_withhold_first_tile(int32_t cta) {
  g_error.clear();
  if (cta < -1 || cta >= 1024) return fail(IDX_INVALID_ARG, "cta must be -1 .. 1023");
  const cudaError_t e = idx::logits_withhold(cta);
  if (e != cudaSuccess) return cuda_fail(e, "fault-injection flag copy");
  return IDX_OK;
}

IDX_EXPORT int idx_device_status(int32_t *status_out, int32_t clear) {
  g_error.clear();
  if (status_out == nullptr) return fail(IDX_INVALID_ARG, "status_out is NULL");
  int32_t a = 0, b = 0, c = 0;
  cudaError_t e = idx::logits_status(&a, clear != 0);
  if (e == cudaSuccess) e = idx::select_status(&b, clear != 0);
  if (e == cudaSuccess) e = idx::mxfp4_status(&c, clear != 0);
  if (e != cudaSuccess) return cuda_fail(e, "status copy");
  *status_out = a | b | c;
  return IDX_OK;
}
