// logits_d64.cu -- the paged FP8 MQA logits kernel (logits_kernel.cuh) instantiated for
// head_dim 64: rows of 64 bytes, moved by TMA and read by the tensor core with the 64-byte
// swizzle, two K = 32 MMAs per tile.

#include "logits_kernel.cuh"

namespace idx {

cudaError_t launch_logits_d64(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                              const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                              cudaStream_t stream) {
  switch (args.num_heads) {
    case 32: return launch_shape<32, 64>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    case 64: return launch_shape<64, 64>(next_n, mode, kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t logits_d64_status(int32_t *value, bool clear) { return read_unit_status(value, clear); }

cudaError_t logits_d64_withhold(int32_t cta) { return set_unit_withhold(cta); }

}  // namespace idx
