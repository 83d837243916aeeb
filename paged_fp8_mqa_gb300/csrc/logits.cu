// logits.cu -- the paged FP8 MQA logits kernel (logits_kernel.cuh) instantiated for
// head_dim 128, and the entry that dispatches every shape ("flashinfer.attn_scores",
// fp8_paged_mqa_logits: Parameters q, num_heads/head_dim restrictions).  The head_dim 64
// instantiations live in logits_d64.cu, compiled in parallel with this unit.

#include "logits_kernel.cuh"

namespace idx {

cudaError_t launch_logits_fp8(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                              const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                              cudaStream_t stream) {
  if (args.head_dim == 192)
    return launch_logits_d192(next_n, mode, kv_map, q_map, args, num_ctas, stream);
  if (args.num_heads == 8) return launch_logits_h8(next_n, mode, kv_map, q_map, args, num_ctas,
                                                    stream);
  if (args.num_heads == 16)
    return launch_logits_h16(next_n, mode, kv_map, q_map, args, num_ctas, stream);
  if (args.head_dim == 64) return launch_logits_d64(next_n, mode, kv_map, q_map, args, num_ctas,
                                                     stream);
  if (args.head_dim != 128) return cudaErrorInvalidValue;
  switch (args.num_heads) {
    case 32: return launch_shape<32, 128>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    case 64: return launch_shape<64, 128>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t logits_withhold(int32_t cta) {
  cudaError_t e = set_unit_withhold(cta);
  if (e == cudaSuccess) e = logits_d64_withhold(cta);
  if (e == cudaSuccess) e = logits_mx_withhold(cta);
  if (e == cudaSuccess) e = logits_h8_withhold(cta);
  if (e == cudaSuccess) e = logits_h16_withhold(cta);
  if (e == cudaSuccess) e = logits_d192_withhold(cta);
  return e;
}

cudaError_t logits_status(int32_t *value, bool clear) {
  int32_t d64 = 0, mx = 0, h8 = 0, h16 = 0, d192 = 0;
  cudaError_t e = read_unit_status(value, clear);
  if (e == cudaSuccess) e = logits_d64_status(&d64, clear);
  if (e == cudaSuccess) e = logits_mx_status(&mx, clear);
  if (e == cudaSuccess) e = logits_h8_status(&h8, clear);
  if (e == cudaSuccess) e = logits_h16_status(&h16, clear);
  if (e == cudaSuccess) e = logits_d192_status(&d192, clear);
  if (e == cudaSuccess) *value |= d64 | mx | h8 | h16 | d192;
  return e;
}

}  // namespace idx
