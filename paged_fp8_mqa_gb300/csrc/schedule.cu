// schedule.cu -- the standalone work-split kernel ("flashinfer.attn_scores", Parameters:
// schedule_meta; Scheduling and Setup: "one small GPU kernel").  One CTA computes every CTA's
// start point from seq_lens' current contents, so a captured graph re-derives it on replay.

#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "split.cuh"

namespace idx {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    k_schedule(const int32_t *seq_lens, int64_t stride, int batch, int num_ctas,
               int32_t *schedule) {
  // The previous kernel in the stream may still be running: no global memory before this.
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ long long smem[];  // [kThreads/32] warp totals, [batch] prefix, [batch] lens
  long long *s_warp = smem;
  long long *s_incl = smem + kThreads / 32;
  int *s_len = reinterpret_cast<int *>(s_incl + batch);
  const long long total = load_lengths<kThreads>(seq_lens, stride, batch, s_len, s_incl, s_warp);
  for (int c = threadIdx.x; c <= num_ctas; c += kThreads) {
    const int2 at = locate_tile(s_incl, s_len, batch, total * c / num_ctas);
    schedule[2 * c] = at.x;
    schedule[2 * c + 1] = at.y;
  }
}

}  // namespace

cudaError_t launch_schedule(const int32_t *seq_lens, int64_t stride, int batch, int num_ctas,
                            int32_t *schedule, cudaStream_t stream) {
  static PerDeviceOnce configured;
  const cudaError_t e = configured.run([] {
    return cudaFuncSetAttribute(
        k_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(sizeof(long long) * (kThreads / 32 + kMaxBatch) + 4 * kMaxBatch));
  });
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(long long) * (kThreads / 32 + batch) + 4 * static_cast<size_t>(batch);
  return launch_dependent(k_schedule, dim3(1), dim3(kThreads), smem, stream, seq_lens, stride, batch,
                          num_ctas, schedule);
}

}  // namespace idx
