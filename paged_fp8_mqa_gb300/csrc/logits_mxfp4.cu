// logits_mxfp4.cu -- the paged logits kernel (logits_kernel.cuh) reading an MXFP4 KV pool
// ("flashinfer.attn_scores", fp4_paged_mqa_logits: formula block, Parameters kv_fused,
// output_dtype): converter warps turn each tile's E2M1 pages into the e4m3 tile the tensor core
// reads, in shared memory.  Instantiated for head_dim 128, 32 or 64 heads, every page size and
// draft depth, and float32, float16 and bfloat16 output (bfloat16 is the pages' default here).

#include "logits_kernel.cuh"

namespace idx {

namespace {

template <int H, typename OutT>
cudaError_t launch_mx_out(int next_n, const CUtensorMap &q_map, const LogitsArgs &args,
                          int num_ctas, cudaStream_t stream) {
  // The KV tensor map is not used by this variant (bulk copies of whole pages); q's stands in.
  return launch_out<H, 128, OutT, true>(next_n, q_map, q_map, args, num_ctas, stream);
}

template <int H>
cudaError_t launch_mx_heads(int next_n, int output_dtype, const CUtensorMap &q_map,
                            const LogitsArgs &args, int num_ctas, cudaStream_t stream) {
  switch (output_dtype) {
    case IDX_DTYPE_F32: return launch_mx_out<H, float>(next_n, q_map, args, num_ctas, stream);
    case IDX_DTYPE_F16: return launch_mx_out<H, __half>(next_n, q_map, args, num_ctas, stream);
    case IDX_DTYPE_BF16:
      return launch_mx_out<H, __nv_bfloat16>(next_n, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_logits_mxfp4(int next_n, int output_dtype, const CUtensorMap &q_map,
                                const LogitsArgs &args, int num_ctas, cudaStream_t stream) {
  if (args.head_dim != 128) return cudaErrorInvalidValue;
  switch (args.num_heads) {
    case 32: return launch_mx_heads<32>(next_n, output_dtype, q_map, args, num_ctas, stream);
    case 64: return launch_mx_heads<64>(next_n, output_dtype, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t logits_mx_status(int32_t *value, bool clear) { return read_unit_status(value, clear); }

cudaError_t logits_mx_withhold(int32_t cta) { return set_unit_withhold(cta); }

}  // namespace idx
