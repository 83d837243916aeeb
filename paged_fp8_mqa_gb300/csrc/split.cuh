// split.cuh -- the persistent logits kernel's work split ("flashinfer.attn_scores",
// Parameters: schedule_meta; Scheduling and Setup), computed on the device from seq_lens.
//
// Request b owns ceil(seq_lens[b] / kTileTokens) tiles of kTileTokens KV positions; the U
// tiles of all requests, flattened request by request, are cut into `num_ctas` contiguous
// ranges, CTA c taking [floor(c*U/num_ctas), floor((c+1)*U/num_ctas)).
#pragma once

#include <cstdint>

#include "internal.h"

namespace idx {

constexpr int kTileTokens = 128;

__device__ __forceinline__ int tiles_of(int len) {
  return len / kTileTokens + (len % kTileTokens != 0 ? 1 : 0);
}

// Exclusive prefix sum over the block; `s_warp` holds THREADS/32 int64 values.
template <int THREADS>
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long *s_warp,
                                                          long long *total) {
  static_assert(THREADS % 32 == 0, "whole warps");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  long long before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) {
    const long long x = s_warp[w];
    if (w < warp) before += x;
    all += x;
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

// Loads seq_lens into s_len[0..batch) and writes the inclusive prefix of tile counts into
// s_incl[0..batch).  Returns the total tile count U (same in every thread).
template <int THREADS>
__device__ __forceinline__ long long load_lengths(const int32_t *seq_lens, int64_t stride,
                                                  int batch, int *s_len, long long *s_incl,
                                                  long long *s_warp) {
  const int per = (batch + THREADS - 1) / THREADS;
  const int lo = threadIdx.x * per;
  const int hi = min(lo + per, batch);
  long long mine = 0;
  for (int b = lo; b < hi; ++b) {
    int len = __ldg(seq_lens + static_cast<int64_t>(b) * stride);
    len = len < 0 ? 0 : len;
    s_len[b] = len;
    mine += tiles_of(len);
  }
  long long total;
  long long run = block_exclusive_scan<THREADS>(mine, s_warp, &total);
  for (int b = lo; b < hi; ++b) {
    run += tiles_of(s_len[b]);
    s_incl[b] = run;
  }
  __syncthreads();
  return total;
}

// (request, tile) of flat tile index `flat` in [0, U]: the first request whose inclusive tile
// prefix exceeds `flat`; flat == U gives (batch, 0).
__device__ __forceinline__ int2 locate_tile(const long long *s_incl, const int *s_len, int batch,
                                            long long flat) {
  int lo = 0, hi = batch;  // first index in [lo, hi) with s_incl[idx] > flat
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_incl[mid] > flat)
      hi = mid;
    else
      lo = mid + 1;
  }
  if (lo >= batch) return make_int2(batch, 0);
  const long long first = s_incl[lo] - tiles_of(s_len[lo]);
  return make_int2(lo, static_cast<int>(flat - first));
}

// Walks one CTA's tiles in order: (b, j) from the start point up to (not including) the end
// point, skipping requests without tiles.  Lengths come from shared memory.
struct TileIter {
  int b, j, b_end, j_end, batch;
  const int *len;

  __device__ __forceinline__ void normalize() {
    while (b < batch && j >= tiles_of(len[b])) {
      ++b;
      j = 0;
    }
  }
  __device__ __forceinline__ bool valid() const {
    return b < batch && (b < b_end || (b == b_end && j < j_end));
  }
  __device__ __forceinline__ void next() {
    ++j;
    normalize();
  }
};

__device__ __forceinline__ TileIter make_iter(int b0, int j0, int b1, int j1, int batch,
                                              const int *len) {
  TileIter it;
  it.b = min(max(b0, 0), batch);
  it.j = max(j0, 0);
  it.b_end = min(max(b1, 0), batch);
  it.j_end = max(j1, 0);
  it.batch = batch;
  it.len = len;
  it.normalize();
  return it;
}

}  // namespace idx
