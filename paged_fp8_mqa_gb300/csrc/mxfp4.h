// mxfp4.h -- host-side interface of the MXFP4 staging kernels (mxfp4.cu) for the C ABI layer.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace idx {

// MXFP4 staging: q rows (and their weights) and the KV pages the batch references converted to
// the FP8 layouts, with each row's largest block scale moved into the weight / per-token scale.
struct Mxfp4Stage {
  const uint8_t *q4;       // [batch * next_n * num_heads][head_dim / 2] packed E2M1
  const uint8_t *q_sf;     // [batch * next_n * num_heads][head_dim / 32] UE8M0
  const float *weights;    // [batch * next_n][num_heads]
  const uint8_t *kv4;      // [num_blocks][block_size * (head_dim / 2 + head_dim / 32)]
  const int32_t *block_tables;
  int64_t bt_stride;
  const int32_t *seq_lens;
  int64_t sl_stride;
  uint8_t *q8;             // staged q, [batch * next_n * num_heads][head_dim] e4m3
  float *w8;               // staged weights
  uint8_t *kv8;            // staged pool, [num_blocks][block_size * (head_dim + 4)]
  int64_t num_blocks;
  int32_t rows_heads;      // batch * next_n * num_heads
  int32_t block_size;
  int32_t head_dim;        // 64 or 128
  int32_t batch;
  int32_t max_pages;       // ceil(max_seq_len / block_size)
  bool stage_kv;           // false: q and the weights only (the logits kernel converts the KV
                           // pages on chip); kv8 unused
};

cudaError_t launch_mxfp4_stage(const Mxfp4Stage &stage, cudaStream_t stream);

// The staging kernels' device-side status bits (IDX_DEV_*).
cudaError_t mxfp4_status(int32_t *value, bool clear);

}  // namespace idx
