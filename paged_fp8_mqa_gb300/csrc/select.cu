// select.cu -- per-row threshold top-k over stage-1 logits ("flashinfer.sdsa.
// indexer_threshold_select": description; Parameters row_ends, thresholds, counters,
// candidates, max_context, top_k, arrivals, ranges).
//
// Grid: (ceil(max_context / kChunk), rows).  CTA (c, r) sweeps keys [c*kChunk, (c+1)*kChunk)
// of row r below row_ends[r]: s > thr is a candidate, "neither above nor below" (== or NaN) a
// tie.  Slots are reserved with one atomicAdd per warp and per kind (warp-aggregated), the
// n-th candidate going to slot top_k + n (n < capacity), the n-th tie to top_k - 1 - n
// (n < top_k), each as (key index, raw float32 bits).
//
// With `arrivals`, the last CTA of a row to finish (an atomicAdd ticket, no waiting) decides
// whether the row fits; if not, it repairs it alone: an MSB-first radix select (4 passes of 8
// bits over order-preserving uint32 keys, i.e. IEEE totalOrder) finds the row's K'-th largest
// key v, K' = min(row_end, top_k); a final in-order sweep stores the keys above v as candidates
// and the lowest-index keys equal to v as ties, K' items in all.  It then rewrites counters,
// the threshold (v) and ranges, and returns arrivals[r] to zero.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/idx.h"
#include "internal.h"

namespace idx {

__device__ int g_select_status;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 8192;       // keys per sweeping CTA (16 per thread)
constexpr int kRepairSpan = kThreads * 8;

// Order-preserving map float -> uint32: a < b in IEEE totalOrder iff key(a) < key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// One warp-wide classification step: every lane offers at most one key.
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

// Block-wide exclusive scan of one int per thread; returns the prefix, *total the sum.
__device__ __forceinline__ int block_scan(int v, int *s_warp, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int x = s_warp[w];
    if (w < warp) before += x;
    all += x;
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

// Repairs row `r` (called by every thread of the row's last CTA): see the file comment.
__device__ void repair_row(const float *row, int row_end, int K, int top_k, int2 *slots,
                           int *cand_out, int *tie_out, float *thr_out) {
  __shared__ unsigned s_hist[256];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need, s_cand, s_tie_base;
  __shared__ int s_warp[kWarps];
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_prefix = 0;
    s_mask = 0;
    s_need = K;
  }
  __syncthreads();
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kThreads) s_hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int i = tid * 4; i < row_end; i += kThreads * 4) {
      if (i + 3 < row_end) {
        const float4 v = *reinterpret_cast<const float4 *>(row + i);
        const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t key = order_key(e[k]);
          if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
        }
      } else {
        for (int k = i; k < row_end; ++k) {
          const uint32_t key = order_key(row[k]);
          if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
        }
      }
    }
    __syncthreads();
    if (tid < 32) {
      // Lane l owns digits 255-8l .. 248-8l (descending), so a prefix over lanes counts the keys
      // above each lane's digits.
      const int hi = 255 - 8 * tid;
      unsigned local = 0;
#pragma unroll
      for (int d = 0; d < 8; ++d) local += s_hist[hi - d];
      unsigned incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      const unsigned above = incl - local;
      const unsigned need = static_cast<unsigned>(s_need);
      if (above < need && need <= incl) {
        unsigned cum = above;
        for (int d = 0; d < 8; ++d) {
          const unsigned h = s_hist[hi - d];
          if (cum + h >= need) {
            s_prefix = s_prefix | (static_cast<uint32_t>(hi - d) << shift);
            s_mask = s_mask | (0xFFu << shift);
            s_need = static_cast<int>(need - cum);
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
  }
  const uint32_t vkey = s_prefix;
  const int m = s_need;        // keys equal to v that are kept
  const int c = K - m;         // keys above v (all kept)
  if (tid == 0) {
    s_cand = 0;
    s_tie_base = 0;
  }
  __syncthreads();
  for (int i0 = 0; i0 < row_end; i0 += kRepairSpan) {
    const int first = i0 + tid * 8;
    uint32_t keys[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) keys[k] = 0u;  // key 0 is below every real key's tie/candidate
    if (first + 7 < row_end) {
      const float4 a = *reinterpret_cast<const float4 *>(row + first);
      const float4 b = *reinterpret_cast<const float4 *>(row + first + 4);
      keys[0] = order_key(a.x); keys[1] = order_key(a.y); keys[2] = order_key(a.z);
      keys[3] = order_key(a.w); keys[4] = order_key(b.x); keys[5] = order_key(b.y);
      keys[6] = order_key(b.z); keys[7] = order_key(b.w);
    } else {
      for (int k = 0; k < 8; ++k)
        if (first + k < row_end) keys[k] = order_key(row[first + k]);
    }
    int mine = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool valid = first + k < row_end;
      if (valid && keys[k] > vkey) {
        const int n = atomicAdd(&s_cand, 1);
        if (n < c) slots[top_k + n] = make_int2(first + k, __float_as_int(key_value(keys[k])));
      }
      mine += (valid && keys[k] == vkey) ? 1 : 0;
    }
    int total;
    int rank = s_tie_base + block_scan(mine, s_warp, &total);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (first + k < row_end && keys[k] == vkey) {
        if (rank < m) slots[top_k - 1 - rank] = make_int2(first + k, __float_as_int(key_value(vkey)));
        ++rank;
      }
    }
    __syncthreads();
    if (tid == 0) s_tie_base += total;
    __syncthreads();
  }
  if (tid == 0) {
    *cand_out = c;
    *tie_out = m;
    *thr_out = key_value(vkey);
  }
}

__global__ void __launch_bounds__(kThreads) k_threshold_select(const SelectArgs a) {
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  int row_end = a.row_ends[r];
  row_end = row_end < 0 ? 0 : (row_end > a.max_context ? a.max_context : row_end);
  const float thr = a.thresholds[r];
  const float *row = a.logits + static_cast<int64_t>(r) * a.row_stride;
  int2 *slots = reinterpret_cast<int2 *>(a.candidates) +
                static_cast<int64_t>(r) * (a.top_k + a.capacity);
  int *counter = a.counters + 2 * r;

  // ---- sweep: classify this CTA's keys ------------------------------------------------------
  const int begin = blockIdx.x * kChunk;
  const int end = min(begin + kChunk, row_end);
  for (int i0 = begin; i0 < end; i0 += kThreads * 4) {
    const int i = i0 + tid * 4;
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (i + 3 < end) {
      const float4 x = __ldcs(reinterpret_cast<const float4 *>(row + i));
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (i + k < end) v[k] = row[i + k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const bool valid = i + k < end;
      const float s = v[k];
      const bool is_cand = valid && s > thr;
      const bool is_tie = valid && !(s > thr) && !(s < thr);
      offer(is_cand, is_tie, i + k, s, counter, slots, a.top_k, a.capacity);
    }
  }
  if (a.arrivals == nullptr) return;

  // ---- last CTA of the row: fit test, repair, reset -----------------------------------------
  __shared__ int s_last, s_fits, s_nc, s_nt;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.arrivals + r, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int K = row_end < a.top_k ? row_end : a.top_k;
  if (tid == 0) {
    const int nc = atomicAdd(counter, 0);
    const int nt = atomicAdd(counter + 1, 0);
    s_nc = nc;
    s_nt = nt;
    s_fits = nc <= a.capacity && (nc >= K || (nt <= a.top_k && nc + nt >= K));
  }
  __syncthreads();
  if (s_fits) {
    if (tid == 0) {
      a.ranges[r] = a.top_k - min(s_nt, a.top_k);
      a.ranges[a.rows + r] = a.top_k + min(s_nc, a.capacity);
    }
  } else {
    __shared__ int s_c, s_m;
    __shared__ float s_v;
    repair_row(row, row_end, K, a.top_k, slots, &s_c, &s_m, &s_v);
    __syncthreads();
    if (tid == 0) {
      counter[0] = s_c;
      counter[1] = s_m;
      a.thresholds[r] = s_v;
      a.ranges[r] = a.top_k - s_m;
      a.ranges[a.rows + r] = a.top_k + s_c;
    }
  }
  if (tid == 0) a.arrivals[r] = 0;
}

}  // namespace

cudaError_t launch_threshold_select(const SelectArgs &args, cudaStream_t stream) {
  const int per_row = args.max_context > 0 ? (args.max_context + kChunk - 1) / kChunk : 1;
  const dim3 grid(per_row, args.rows);
  k_threshold_select<<<grid, kThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

// ---- allocation-free variant ---------------------------------------------------------------
// Arrival counters used by idx_threshold_select_static instead of a caller-provided workspace:
// one int32 per logits row, IDX_STATIC_SELECT_MAX_ROWS of them (64 KiB), resident on every GPU
// that loads this library until the process exits.  All calls share it.
static __device__ __align__(256) int32_t g_static_arrivals[IDX_STATIC_SELECT_MAX_ROWS];

cudaError_t launch_threshold_select_static(SelectArgs args, cudaStream_t stream) {
  constexpr int kMaxDevices = 64;
  static std::mutex mutex;
  static int32_t *device_address[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int32_t *arrivals = nullptr;
  {
    // Once per device, with that device current: the array's device address.  In host code the
    // name g_static_arrivals denotes a host-side stand-in, never usable as a kernel argument.
    std::lock_guard<std::mutex> lock(mutex);
    if (device_address[dev] == nullptr) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_arrivals);
      if (e != cudaSuccess) return e;
      device_address[dev] = static_cast<int32_t *>(p);
    }
    arrivals = device_address[dev];
  }
  // The kernel returns every counter it uses to zero, but a call cut short (an error, a
  // killed context) could leave a stale count behind: start each call from zero.
  e = cudaMemsetAsync(arrivals, 0, sizeof(int32_t) * static_cast<size_t>(args.rows), stream);
  if (e != cudaSuccess) return e;
  args.arrivals = arrivals;
  return launch_threshold_select(args, stream);
}

cudaError_t select_status(int32_t *value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_select_status, sizeof(int32_t));
  if (e != cudaSuccess || !clear) return e;
  const int32_t zero = 0;
  return cudaMemcpyToSymbol(g_select_status, &zero, sizeof(int32_t));
}

}  // namespace idx
