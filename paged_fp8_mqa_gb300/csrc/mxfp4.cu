// mxfp4.cu -- MXFP4 paged MQA logits ("flashinfer.attn_scores", fp4_paged_mqa_logits: formula
// block and Parameters q, q_sf, kv_fused, sf_vec_size), staged through the FP8 logits kernel.
//
//   logits[b*n + t, p] = sum_h w[b*n + t, h] * relu(q[b,t,h,:] . k[p,:]),
//   element d of a row = e2m1(nibble d) * 2^(sf[d / 32] - 127).
//
// A positive power of two commutes with the ReLU, so a row's largest block scale 2^(E - 127)
// can leave the row: for a K token it becomes the FP8 path's per-token scale, for a q head it
// multiplies that head's weight.  What stays is e2m1 * 2^(e - E) per 32-element group, with
// e - E <= 0; e4m3 represents it exactly while e - E >= -8 (the smallest product, 0.5 * 2^-8,
// is e4m3's smallest subnormal 2^-9).  So two conversion kernels stage q (with its weights) and
// every KV page the batch references in the FP8 layout, and the FP8 logits kernel computes the
// MXFP4 logits from them: exactly the same per-head products, the same float32 accumulation in
// the tensor core.  A row whose scales span more than 8 binades (or that carries the NaN scale
// byte 0xFF) is converted with rounding and flagged (IDX_DEV_INEXACT_SCALE).
//
// Workspace (caller memory, idx_mxfp4_workspace_bytes): the staged KV pool (num_blocks pages of
// block_size * (head_dim + 4) bytes, same page ids), the staged q and the scaled weights.

#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/idx.h"
#include "internal.h"
#include "mx_convert.cuh"
#include "mxfp4.h"
#include "ptx.cuh"

namespace idx {

__device__ int g_mxfp4_status;

namespace {

// Converts one row of head_dim elements (head_dim / 2 packed bytes, head_dim / 32 scale bytes)
// into head_dim e4m3 bytes relative to the row's largest scale byte, which it returns.
// *inexact is set if a group is more than 8 binades below it or a scale byte is 0xFF.
template <int D>
__device__ __forceinline__ int stage_row(const uint8_t *packed, const uint8_t *sf, uint8_t *dst,
                                         bool *inexact) {
  constexpr int G = D / 32;
  int e[G];
  int emax = 0;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    e[g] = sf[g];
    emax = max(emax, e[g]);
    if (e[g] == 0xFF) *inexact = true;
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int rel = e[g] - emax;
    const uint2 tab = rel >= -8 ? e2m1_table_entry(-rel) : make_uint2(0u, 0u);
    uint32_t out[8];
    mx_group_to_e4m3(*reinterpret_cast<const uint4 *>(packed + 16 * g), rel, tab, out, inexact);
    uint4 *o = reinterpret_cast<uint4 *>(dst + 32 * g);
    o[0] = make_uint4(out[0], out[1], out[2], out[3]);
    o[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
  return emax;
}

struct Mxfp4Args {
  const uint8_t *q4;       // [rows * H][D/2]
  const uint8_t *q_sf;     // [rows * H][D/32]
  const float *weights;    // [rows][H]
  const uint8_t *kv4;      // [num_blocks][block_size * (D/2 + D/32)]
  const int32_t *block_tables;
  int64_t bt_stride;
  const int32_t *seq_lens;
  int64_t sl_stride;
  uint8_t *q8;             // [rows * H][D]
  float *w8;               // [rows][H]
  uint8_t *kv8;            // [num_blocks][block_size * (D + 4)]
  int64_t num_blocks;
  int32_t rows_heads;      // rows * H
  int32_t block_size;
};

// One thread per (row, head): the staged q row and its weight times the row's largest scale.
template <int D>
__global__ void __launch_bounds__(128) k_mxfp4_q(const Mxfp4Args a) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.rows_heads) return;
  bool inexact = false;
  const int emax = stage_row<D>(a.q4 + static_cast<int64_t>(i) * (D / 2),
                                a.q_sf + static_cast<int64_t>(i) * (D / 32),
                                a.q8 + static_cast<int64_t>(i) * D, &inexact);
  // The weight times the row's largest scale must stay a normal float32 for the product to be
  // exact (a huge or tiny q scale byte could overflow or fall into the subnormals).
  const float w = a.weights[i], w8 = w * pow2f(emax - 127), aw = fabsf(w8);
  a.w8[i] = w8;
  if (w != 0.0f && !(aw >= 1.17549435e-38f && aw <= 3.40282347e38f)) inexact = true;
  if (inexact) atomicOr(&g_mxfp4_status, IDX_DEV_INEXACT_SCALE);
}

// CTA (j, b), one thread per token: page j of request b, if the request has it, staged into
// the same page id of the FP8 pool (values, then the per-token float32 scale).  Only a token
// inside the request's length can raise the inexact flag.  (A page shared by several requests
// is staged by each, with the same bytes.)
template <int D>
__global__ void k_mxfp4_kv(const Mxfp4Args a) {
  griddep_wait();
  griddep_launch_dependents();
  const int j = blockIdx.x, b = blockIdx.y, i = threadIdx.x;
  const int BS = a.block_size;
  const int len = max(0, a.seq_lens[static_cast<int64_t>(b) * a.sl_stride]);
  if (j * BS >= len) return;
  const int id = a.block_tables[static_cast<int64_t>(b) * a.bt_stride + j];
  if (id < 0 || id >= a.num_blocks) {
    if (i == 0) atomicOr(&g_mxfp4_status, IDX_DEV_BAD_PAGE);
    return;
  }
  const uint8_t *src = a.kv4 + static_cast<int64_t>(id) * BS * (D / 2 + D / 32);
  uint8_t *dst = a.kv8 + static_cast<int64_t>(id) * BS * (D + 4);
  bool inexact = false;
  const int emax = stage_row<D>(src + i * (D / 2), src + BS * (D / 2) + i * (D / 32),
                                dst + i * D, &inexact);
  reinterpret_cast<float *>(dst + BS * D)[i] = pow2f(emax - 127);
  if (inexact && j * BS + i < len) atomicOr(&g_mxfp4_status, IDX_DEV_INEXACT_SCALE);
}

template <int D>
cudaError_t launch_stage(const Mxfp4Args &a, int max_pages, int batch, bool stage_kv,
                         cudaStream_t stream) {
  cudaError_t e = launch_dependent(k_mxfp4_q<D>, dim3((a.rows_heads + 127) / 128), dim3(128), 0,
                                   stream, a);
  if (e != cudaSuccess || max_pages == 0 || !stage_kv) return e;
  return launch_dependent(k_mxfp4_kv<D>, dim3(max_pages, batch), dim3(a.block_size), 0, stream,
                          a);
}

}  // namespace

cudaError_t launch_mxfp4_stage(const Mxfp4Stage &s, cudaStream_t stream) {
  Mxfp4Args a{};
  a.q4 = s.q4;
  a.q_sf = s.q_sf;
  a.weights = s.weights;
  a.kv4 = s.kv4;
  a.block_tables = s.block_tables;
  a.bt_stride = s.bt_stride;
  a.seq_lens = s.seq_lens;
  a.sl_stride = s.sl_stride;
  a.q8 = s.q8;
  a.w8 = s.w8;
  a.kv8 = s.kv8;
  a.num_blocks = s.num_blocks;
  a.rows_heads = s.rows_heads;
  a.block_size = s.block_size;
  switch (s.head_dim) {
    case 64: return launch_stage<64>(a, s.max_pages, s.batch, s.stage_kv, stream);
    case 128: return launch_stage<128>(a, s.max_pages, s.batch, s.stage_kv, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t mxfp4_status(int32_t *value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_mxfp4_status, sizeof(int32_t));
  if (e != cudaSuccess || !clear) return e;
  const int32_t zero = 0;
  return cudaMemcpyToSymbol(g_mxfp4_status, &zero, sizeof(int32_t));
}

}  // namespace idx
