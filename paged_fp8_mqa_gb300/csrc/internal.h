// internal.h -- host-side interface between the C ABI layer and the kernel translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/idx.h"

namespace idx {

// Launches `kernel` as a programmatic dependent of the previous kernel in `stream`: the launch may
// be processed while that kernel still runs, so its latency hides behind it.  Every kernel of
// this library calls griddep_wait() before it touches global memory, which keeps stream order.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// A kernel attribute (the opt-in to more than 48 KiB of dynamic shared memory) belongs to the
// current device's context, so each launcher sets it once per device: `set` runs on the first
// call made with each device current (devices past the first 64 run it on every call).
class PerDeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F &&set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
    if (bit != 0 && (done_.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = set();
    if (e == cudaSuccess && bit != 0) done_.fetch_or(bit, std::memory_order_release);
    return e;
  }

 private:
  std::atomic<uint64_t> done_{0};
};

// Largest batch (requests per call) the kernels accept: the logits kernel keeps every
// request's length in shared memory.
constexpr int kMaxBatch = 4096;

// Everything the logits kernel needs besides its two tensor maps.
struct LogitsArgs {
  const uint8_t *kv;            // pool base
  const float *weights;         // [batch*next_n, 64]
  const int32_t *block_tables;  // row b at block_tables + b * bt_stride
  int64_t bt_stride;
  int64_t bt_width;             // columns per row the caller provides (only the live ones are read)
  const int32_t *seq_lens;      // element b at seq_lens[b * sl_stride]
  int64_t sl_stride;
  const int32_t *schedule;      // nullable: [num_ctas + 1][2]
  void *out;                    // float or __half elements; row r at out + r * out_stride
  int64_t out_stride;
  int32_t *row_ends;            // nullable: [batch * next_n]
  int64_t num_blocks;
  int32_t batch;
  int32_t block_size;           // tokens per page: 32, 64 or 128
  int32_t num_heads;            // 32 or 64
  int32_t head_dim;             // 128 or 64
  // Rescoring (nullable): the counts of a finished fused pass ([rows][2], 8-byte aligned); only
  // requests with a row that does not fit (by top_k and capacity below) are scored.
  const int32_t *fit_counters;
  // Fused select (LogitsOut::kSelect; rows b * next_n + t): the select's per-row state.
  const float *thresholds;
  int32_t *counters;            // [rows][2], zeroed by the caller
  int32_t *candidates;          // [rows][top_k + capacity][2]
  int32_t top_k;
  int32_t capacity;
};

// What the logits kernel does with each score.
enum class LogitsOut { kF32, kF16, kSelect };

// Launches the logits kernel for draft depth `next_n` (1..4).
cudaError_t launch_logits_fp8(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                              const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                              cudaStream_t stream);

// The head_dim 64 instantiations (a separate translation unit) and their status bits.
cudaError_t launch_logits_d64(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                              const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                              cudaStream_t stream);
cudaError_t logits_d64_status(int32_t *value, bool clear);
cudaError_t logits_d64_withhold(int32_t cta);

// The 8- and 16-head instantiations (translation units of their own; float32 / float16 output).
cudaError_t launch_logits_h8(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                             const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                             cudaStream_t stream);
cudaError_t launch_logits_h16(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                              const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                              cudaStream_t stream);
cudaError_t logits_h8_status(int32_t *value, bool clear);
cudaError_t logits_h16_status(int32_t *value, bool clear);
cudaError_t logits_h8_withhold(int32_t cta);
cudaError_t logits_h16_withhold(int32_t cta);

// The head_dim 192 instantiations (32 or 64 heads; float32 / float16 output).  kv_map views the
// pool as [num_blocks][block_size][3][64] bytes (page stride block_size * 196), q_map as
// [rows][3][64]; both with the 64-byte swizzle and boxes of one K block.
cudaError_t launch_logits_d192(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                               const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                               cudaStream_t stream);
cudaError_t logits_d192_status(int32_t *value, bool clear);
cudaError_t logits_d192_withhold(int32_t cta);

// The same kernel reading an MXFP4 KV pool (head_dim 128; a separate translation unit): q and
// weights already staged in the FP8 layout (q_map over them), args.kv the MXFP4 pool.
// output_dtype: IDX_DTYPE_F32, _F16 or _BF16.
cudaError_t launch_logits_mxfp4(int next_n, int output_dtype, const CUtensorMap &q_map,
                                const LogitsArgs &args, int num_ctas, cudaStream_t stream);
cudaError_t logits_mx_status(int32_t *value, bool clear);
cudaError_t logits_mx_withhold(int32_t cta);

// Launches the standalone schedule kernel.
cudaError_t launch_schedule(const int32_t *seq_lens, int64_t stride, int batch, int num_ctas,
                            int32_t *schedule, cudaStream_t stream);

struct SelectArgs {
  const float *logits;
  int64_t row_stride;
  const int32_t *row_ends;
  float *thresholds;
  int32_t *counters;
  int32_t *candidates;
  int32_t *arrivals;  // nullable
  int32_t *ranges;    // nullable unless arrivals
  int32_t rows;
  int32_t top_k;
  int32_t capacity;
  int32_t max_context;
};

cudaError_t launch_threshold_select(const SelectArgs &args, cudaStream_t stream);

// The fused score + select's last stage: one CTA per row, which writes the range of a row that
// fits and repairs one that does not from its rescored logits.
struct FusedRepairArgs {
  const float *scratch;    // rescored logits, row r at scratch + r * scratch_stride
  int64_t scratch_stride;
  const int32_t *seq_lens;
  int64_t sl_stride;
  float *thresholds;
  int32_t *counters;
  int32_t *candidates;
  int32_t *ranges;
  int32_t batch;
  int32_t next_n;
  int32_t top_k;
  int32_t capacity;
};

cudaError_t launch_fused_repair(const FusedRepairArgs &args, cudaStream_t stream);

// The same launch with `args.arrivals` replaced by the library's own static device array
// (at most IDX_STATIC_SELECT_MAX_ROWS rows; the caller checks).
cudaError_t launch_threshold_select_static(SelectArgs args, cudaStream_t stream);

// Device-side status words of each translation unit (IDX_DEV_* bits).
cudaError_t logits_status(int32_t *value, bool clear);
// (testing only) The logits CTA that withholds its first tile's copies (-1: none), in both
// logits translation units.
cudaError_t logits_withhold(int32_t cta);
cudaError_t select_status(int32_t *value, bool clear);

}  // namespace idx
