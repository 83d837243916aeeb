// logits_h16.cu -- the paged FP8 MQA logits kernel (logits_kernel.cuh) instantiated for 16 heads
// ("flashinfer.attn_scores", fp8_paged_mqa_logits: num_heads and next_n * num_heads
// restrictions), head_dim 64 and 128, float32 and float16 output, in a translation unit of its
// own (compiled in parallel with the others).

#include "logits_kernel.cuh"

namespace idx {

cudaError_t launch_logits_h16(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                              const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                              cudaStream_t stream) {
  switch (args.head_dim) {
    case 64: return launch_shape_plain<16, 64>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    case 128: return launch_shape_plain<16, 128>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t logits_h16_status(int32_t *value, bool clear) { return read_unit_status(value, clear); }

cudaError_t logits_h16_withhold(int32_t cta) { return set_unit_withhold(cta); }

}  // namespace idx
