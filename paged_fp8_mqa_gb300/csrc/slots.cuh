// slots.cuh -- candidate and tie slots of the threshold select ("flashinfer.sdsa.
// indexer_threshold_select": description; Parameters counters, candidates), shared by the select
// sweep and the fused logits epilogue.
//
// A key scoring above its row's threshold is a candidate, one neither above nor below it (equal,
// or NaN) a tie.  Both are counted in counters[r] = {candidates, ties}; the n-th candidate is
// stored at slot top_k + n (n < capacity), the n-th tie at slot top_k - 1 - n (n < top_k), each
// as (key index, float32 bits of the score).
#pragma once

#include <cstdint>

namespace idx {

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// One warp-wide classification step (all 32 lanes call it, each offering at most one key of the
// same row): one atomicAdd per warp and kind reserves the slots.
__device__ __forceinline__ void offer(bool is_cand, bool is_tie, int index, float score,
                                      int *counter, int2 *slots, int top_k, int capacity) {
  const int lane = threadIdx.x & 31;
  const unsigned mc = __ballot_sync(0xffffffffu, is_cand);
  if (mc) {
    const int leader = __ffs(mc) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(counter, __popc(mc));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (is_cand) {
      const int n = base + __popc(mc & lanemask_lt());
      if (n < capacity) slots[top_k + n] = make_int2(index, __float_as_int(score));
    }
  }
  const unsigned mt = __ballot_sync(0xffffffffu, is_tie);
  if (mt) {
    const int leader = __ffs(mt) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(counter + 1, __popc(mt));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (is_tie) {
      const int n = base + __popc(mt & lanemask_lt());
      if (n < top_k) slots[top_k - 1 - n] = make_int2(index, __float_as_int(score));
    }
  }
}

// The fit rule: the row's exact top-K' (K' = min(row_end, top_k)) is among its slots when the
// candidates fit capacity and either reach K' alone or, with every tie stored, together with
// the ties.
__device__ __forceinline__ bool row_fits(int nc, int nt, int K, int top_k, int capacity) {
  return nc <= capacity && (nc >= K || (nt <= top_k && nc + nt >= K));
}

}  // namespace idx
