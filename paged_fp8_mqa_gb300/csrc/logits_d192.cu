// logits_d192.cu -- the paged FP8 MQA logits kernel (logits_kernel.cuh) instantiated for
// head_dim 192 ("flashinfer.attn_scores", fp8_paged_mqa_logits: head_dim % 32 == 0, and the
// shared-memory note that 192 fits at 64 heads), 32 or 64 heads, float32 and float16 output: a
// row is three 64-byte K blocks (64-byte swizzle), six K = 32 MMAs per tile.

#include "logits_kernel.cuh"

namespace idx {

cudaError_t launch_logits_d192(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                               const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                               cudaStream_t stream) {
  switch (args.num_heads) {
    case 32: return launch_shape_plain<32, 192>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    case 64: return launch_shape_plain<64, 192>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t logits_d192_status(int32_t *value, bool clear) { return read_unit_status(value, clear); }

cudaError_t logits_d192_withhold(int32_t cta) { return set_unit_withhold(cta); }

}  // namespace idx
