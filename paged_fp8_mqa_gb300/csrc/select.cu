// select.cu -- per-row threshold top-k over stage-1 logits ("flashinfer.sdsa.
// indexer_threshold_select": description; Parameters row_ends, thresholds, counters,
// candidates, max_context, top_k, arrivals, ranges).
//
// Launch 1, grid (rows, ceil(max_context / kChunk)) of 512-thread CTAs (two per SM): CTA (r, c)
// sweeps keys [c*kChunk, (c+1)*kChunk) of row r below row_ends[r]: s > thr is a candidate,
// "neither above nor below" (== or NaN) a tie.  Slots are reserved with one atomicAdd per warp
// and per kind for all the warp's 512 keys (a warp scan of the counts), the n-th candidate going
// to slot top_k + n (n < capacity), the n-th tie to top_k - 1 - n (n < top_k), each as (key
// index, raw float32 bits).
//
// With `arrivals`, a second launch (a programmatic dependent: it proceeds only once launch 1 has
// finished, so every count is final) decides for each row whether it fits and, if not, repairs
// it with one 1024-thread CTA (one CTA per row, or per SM taking rows in turn when there are
// more rows than SMs): an MSB-first radix select over order-preserving uint32 keys (i.e.
// IEEE totalOrder) finds the row's K'-th largest key v, K' = min(row_end, top_k), and the row's
// keys above v become candidates and its lowest-index keys equal to v ties, K' items in all.  It
// then rewrites counters, the threshold (v) and ranges, and zeroes arrivals[r] (which nothing
// reads: no CTA waits for or counts the others).  The repair first needs a key lo <= v: 0 if the
// whole row fits a 6144-key shared-memory buffer, else the row's threshold if the classification
// counted between K' and 6144 keys at or above it, else a bound read off a sample of 2048 of
// the row's keys with a safety margin.  One sweep gathers every key >= lo into the buffer (one
// shared atomic per warp and 32 keys), where three histogram passes (11, 11, 10 bits) find v
// and the output is written.  If fewer than K' or more than 6144 keys are >= lo, it falls back
// to two sweeps (an 11-bit histogram of the row finds the bin holding v; a second sweep stores
// the keys of higher bins as candidates and gathers the bin into the buffer), and if that bin is
// too large, to four 8-bit passes over the row and a final in-order sweep.
//
// k_fused_repair is the last launch of the fused score + select: one CTA per row, which writes
// the slot range of a row that fits and repairs one that does not, with the same code, from the
// row's rescored logits.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/idx.h"
#include "internal.h"
#include "ptx.cuh"
#include "slots.cuh"

namespace idx {

__device__ int g_select_status;

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kClsThreads = 512;  // threads of a classifying CTA (two per SM)
constexpr int kChunk = 8192;       // keys per classifying CTA
constexpr int kSweepLoads = kChunk / (kClsThreads * 4);  // float4 per thread, all in flight
constexpr int kBufKeys = 6144;                  // keys of the bin holding v, kept in shared memory
constexpr int kTieRank = 2048;                  // ties ranked in shared memory (ordered case)
constexpr uint32_t kSelectSmem = 2048 * 4 + kBufKeys * 8;  // dynamic: histogram + (key, index)
constexpr int kPassLoads = 8;                   // 16-byte loads in flight per thread, histogram
constexpr int kSamples = 2048;                  // keys sampled to bound the K'-th from below
constexpr int kSweepKeys = 16;                  // contiguous keys per thread, final sweep
constexpr int kRepairSpan = kThreads * kSweepKeys;

// Scores are handled as their bit patterns from the load on: a float-typed NaN may not keep its
// bits (a NaN read as a float and turned into its order key gave the key of -0 on this GPU), and
// the repair must order +NaN above +inf and -NaN below -inf, and store every score's own bits.
__device__ __forceinline__ uint32_t ldg_bits(const float *p) {
  return __ldg(reinterpret_cast<const unsigned *>(p));
}
// Order-preserving map of a binary32's bits -> uint32: a < b in IEEE totalOrder iff
// key(a) < key(b); key_bits is its inverse.
__device__ __forceinline__ uint32_t order_key(uint32_t u) {
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_bits(uint32_t k) {
  return (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
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

// The bin of the need-th largest key of a histogram of nbins (2048 or 1024) bins, counting from
// the top: *s_bin and *s_above (the count of keys in higher bins); both are left unchanged if
// the histogram holds fewer than `need` keys.  All threads call it.  Warp w sums the w-th range
// of nbins / 32 bins from the top; warp 0 scans the 32 sums, then the bins of the range that
// holds the need-th key, and publishes the bin (two block barriers in all).
__device__ __forceinline__ void find_bin(const unsigned *h, int nbins, unsigned need,
                                         int *s_bin, unsigned *s_above, int *s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_warp = nbins / kWarps;  // 64 or 32
  const int per_lane = per_warp / 32;   // 2 or 1
  unsigned *s_wsum = reinterpret_cast<unsigned *>(s_warp);
  {
    const int top = nbins - 1 - warp * per_warp - lane * per_lane;
    unsigned x = 0;
    for (int j = 0; j < per_lane; ++j) x += h[top - j];
    x = __reduce_add_sync(0xffffffffu, x);
    if (lane == 0) s_wsum[warp] = x;
  }
  __syncthreads();
  if (warp == 0) {
    const auto scan = [&](unsigned v) {  // inclusive scan over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      return v;
    };
    const unsigned ws = s_wsum[lane];  // range `lane`, counted from the top
    const unsigned incl = scan(ws), excl = incl - ws;
    const unsigned hit = __ballot_sync(0xffffffffu, excl < need && need <= incl);
    if (hit) {
      const int w = __ffs(hit) - 1;
      const unsigned above = __shfl_sync(0xffffffffu, excl, w);
      const int top = nbins - 1 - w * per_warp - lane * per_lane;
      unsigned v = 0;
      for (int j = 0; j < per_lane; ++j) v += h[top - j];
      const unsigned incl2 = scan(v), excl2 = incl2 - v;
      const unsigned need2 = need - above;
      const unsigned hit2 = __ballot_sync(0xffffffffu, excl2 < need2 && need2 <= incl2);
      if (hit2 && lane == __ffs(hit2) - 1) {
        unsigned cum = above + excl2;
        for (int j = 0; j < per_lane; ++j) {
          const unsigned c = h[top - j];
          if (cum + c >= need) {
            *s_bin = top - j;
            *s_above = cum;
            break;
          }
          cum += c;
        }
      }
    }
  }
  __syncthreads();
}

// Finishes a repair from the shared-memory buffer of nb (key, index) pairs.  The buffer holds
// every key of the row that is >= v (the K-th largest), except the `*s_cand` keys already stored
// as candidates, which all lie above the buffer's keys.  need = K - *s_cand.  With b1 >= 0 every
// buffered key has leading 11 bits b1; with b1 < 0 the buffer may span any bins (b1 == -2: the
// histogram of their leading 11 bits is already in s_h).  Writes the
// buffered keys above v as candidates and the ties (all of them, or the m lowest indices).
// Returns false, having written nothing, if more than kTieRank tied keys would need ranking.
__device__ bool finish_from_buffer(const uint32_t *s_bkey, const int *s_bidx, int nb, int b1_in,
                                   unsigned need, int K, int top_k, int2 *slots, int *s_cand,
                                   unsigned *s_h, int *cand_out, int *tie_out, uint32_t *thr_out) {
  __shared__ int s_bin, s_ntie;
  __shared__ unsigned s_above;
  __shared__ int s_warp[kWarps];
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bin = 0;
    s_above = 0;
    s_ntie = 0;
  }
  uint32_t b1 = static_cast<uint32_t>(b1_in);
  if (b1_in < 0) {  // the leading 11 bits (b1_in == -2: their histogram is already in s_h)
    if (b1_in == -1) {
      for (int i = tid; i < 2048; i += kThreads) s_h[i] = 0;
      __syncthreads();
      for (int j = tid; j < nb; j += kThreads) atomicAdd(&s_h[s_bkey[j] >> 21], 1u);
    }
    __syncthreads();
    find_bin(s_h, 2048, need, &s_bin, &s_above, s_warp);
    b1 = static_cast<uint32_t>(s_bin);
    need -= s_above;
  }
  // The next 11 bits among the keys of bin b1, then the last 10.
  for (int i = tid; i < 2048; i += kThreads) s_h[i] = 0;
  __syncthreads();
  for (int j = tid; j < nb; j += kThreads)
    if ((s_bkey[j] >> 21) == b1) atomicAdd(&s_h[(s_bkey[j] >> 10) & 2047u], 1u);
  __syncthreads();
  find_bin(s_h, 2048, need, &s_bin, &s_above, s_warp);
  const uint32_t p2 = (b1 << 11) | static_cast<uint32_t>(s_bin);
  const unsigned need2 = need - s_above;
  for (int i = tid; i < 1024; i += kThreads) s_h[i] = 0;
  __syncthreads();
  for (int j = tid; j < nb; j += kThreads)
    if ((s_bkey[j] >> 10) == p2) atomicAdd(&s_h[s_bkey[j] & 1023u], 1u);
  __syncthreads();
  find_bin(s_h, 1024, need2, &s_bin, &s_above, s_warp);
  const uint32_t vkey = (p2 << 10) | static_cast<uint32_t>(s_bin);
  const int m = static_cast<int>(need2 - s_above);  // keys equal to v that are kept
  const int ties = static_cast<int>(s_h[s_bin]);    // keys equal to v in the row
  const int c = K - m;                              // keys above v
  if (ties > m && ties > kTieRank) return false;
  // ---- write the buffered keys above v, and the ties (all, or the m lowest indices)
  int *s_tidx = reinterpret_cast<int *>(s_h);  // tie indices when they must be ranked
  __syncthreads();
  const int lane = tid & 31;
  for (int j0 = 0; j0 < nb; j0 += kThreads) {  // slots reserved with one atomic per warp
    const int j = j0 + tid;
    const uint32_t key = j < nb ? s_bkey[j] : 0u;
    const bool is_c = j < nb && key > vkey;
    const bool is_t = j < nb && key == vkey;
    const unsigned mc = __ballot_sync(0xffffffffu, is_c);
    if (mc) {
      const int leader = __ffs(mc) - 1;
      int n = 0;
      if (lane == leader) n = atomicAdd(s_cand, __popc(mc));
      n = __shfl_sync(0xffffffffu, n, leader) + __popc(mc & lanemask_lt());
      if (is_c) slots[top_k + n] = make_int2(s_bidx[j], static_cast<int>(key_bits(key)));
    }
    const unsigned mt = __ballot_sync(0xffffffffu, is_t);
    if (mt) {
      const int leader = __ffs(mt) - 1;
      int n = 0;
      if (lane == leader) n = atomicAdd(&s_ntie, __popc(mt));
      n = __shfl_sync(0xffffffffu, n, leader) + __popc(mt & lanemask_lt());
      if (is_t) {
        if (ties == m)
          slots[top_k - 1 - n] = make_int2(s_bidx[j], static_cast<int>(key_bits(vkey)));
        else
          s_tidx[n] = s_bidx[j];
      }
    }
  }
  __syncthreads();
  if (ties > m) {
    // Keep the m lowest indices: a tie's rank is the number of ties with a smaller index.
    for (int j = tid; j < ties; j += kThreads) {
      const int mine = s_tidx[j];
      int rank = 0;
      for (int q = 0; q < ties; ++q) rank += s_tidx[q] < mine ? 1 : 0;
      if (rank < m) slots[top_k - 1 - rank] = make_int2(mine, static_cast<int>(key_bits(vkey)));
    }
  }
  if (tid == 0) {
    *cand_out = c;
    *tie_out = m;
    *thr_out = key_bits(vkey);
  }
  return true;
}

// kPassLoads 16-byte loads of the row per thread, all in flight before any is used (the row is
// L2-resident; one load at a time would leave a sweep bound by the L2 latency), as bits.  Keys
// past row_end read as 0 and must be masked by the caller.
__device__ __forceinline__ void load_pass(const float *row, int row_end, int base,
                                          uint4 (&v)[kPassLoads]) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int u = 0; u < kPassLoads; ++u) {
    const int i = base + (u * kThreads + tid) * 4;
    if (i + 3 < row_end) {
      v[u] = __ldg(reinterpret_cast<const uint4 *>(row + i));
    } else {
      v[u].x = i < row_end ? ldg_bits(row + i) : 0u;
      v[u].y = i + 1 < row_end ? ldg_bits(row + i + 1) : 0u;
      v[u].z = i + 2 < row_end ? ldg_bits(row + i + 2) : 0u;
      v[u].w = 0u;
    }
  }
}

// One-sweep repair of a row (see the file comment): gathers every key >= lo into the buffer and
// finishes there.  lo: 0 (every key) when the row fits the buffer; else `lo_hint` when the caller
// has one (the row's threshold, when the classification counted between K and kBufKeys keys at
// or above it); else the 22-bit prefix of the key of a sample of kSamples keys that ranks at 1.5
// times the rank the K-th largest is expected at, plus 16 (found by two histogram passes).
// Returns false, having written nothing, unless between K and kBufKeys keys are >= lo (and the
// ties can be ranked).
__device__ bool repair_row_gather(const float *row, int row_end, int K, int top_k, int2 *slots,
                                  bool have_hint, uint32_t lo_hint, int *cand_out, int *tie_out,
                                  uint32_t *thr_out, uint8_t *dyn) {
  unsigned *s_h = reinterpret_cast<unsigned *>(dyn);                // [2048]: samples, histogram
  uint32_t *s_bkey = reinterpret_cast<uint32_t *>(dyn + 2048 * 4);  // [kBufKeys]
  int *s_bidx = reinterpret_cast<int *>(s_bkey + kBufKeys);         // [kBufKeys]
  __shared__ int s_nbuf, s_cand;
  const int tid = threadIdx.x;
  if (K > kBufKeys) return false;
  uint32_t lo = 0;
  if (row_end > kBufKeys) {
    if (have_hint) {
      lo = lo_hint;
    } else {
      // kSamples keys evenly spread over the row; two histogram passes (leading 11 bits, then
      // the next 11 within the bin) find the sample of the wanted rank, whose 22-bit prefix is lo.
      __shared__ int s_sbin;
      __shared__ unsigned s_sabove;
      __shared__ int s_swarp[kWarps];
      uint32_t smp[kSamples / kThreads];
#pragma unroll
      for (int q = 0; q < kSamples / kThreads; ++q)
        smp[q] = order_key(
            ldg_bits(row + static_cast<int64_t>(q * kThreads + tid) * row_end / kSamples));
      const int64_t want =
          static_cast<int64_t>(K) * kSamples * 3 / (2 * static_cast<int64_t>(row_end));
      const unsigned rank = static_cast<unsigned>(min(static_cast<int64_t>(kSamples), want + 17));
      for (int i = tid; i < 2048; i += kThreads) s_h[i] = 0;
      if (tid == 0) {
        s_sbin = 0;
        s_sabove = 0;
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < kSamples / kThreads; ++q) atomicAdd(&s_h[smp[q] >> 21], 1u);
      __syncthreads();
      find_bin(s_h, 2048, rank, &s_sbin, &s_sabove, s_swarp);
      const uint32_t sb1 = static_cast<uint32_t>(s_sbin);
      const unsigned rank2 = rank - s_sabove;
      for (int i = tid; i < 2048; i += kThreads) s_h[i] = 0;
      __syncthreads();
#pragma unroll
      for (int q = 0; q < kSamples / kThreads; ++q)
        if ((smp[q] >> 21) == sb1) atomicAdd(&s_h[(smp[q] >> 10) & 2047u], 1u);
      __syncthreads();
      find_bin(s_h, 2048, rank2, &s_sbin, &s_sabove, s_swarp);
      lo = (sb1 << 21) | (static_cast<uint32_t>(s_sbin) << 10);
      __syncthreads();
    }
  }
  for (int i = tid; i < 2048; i += kThreads) s_h[i] = 0;  // the taken keys' leading 11 bits
  if (tid == 0) {
    s_nbuf = 0;
    s_cand = 0;
  }
  __syncthreads();
  const int lane = tid & 31;
  for (int base = 0; base < row_end; base += kThreads * 4 * kPassLoads) {
    uint4 v[kPassLoads];
    load_pass(row, row_end, base, v);
    // This thread's keys >= lo as a bit mask; then one warp scan and one shared atomic per warp
    // place them in the buffer, each lane storing only its own (few) keys, re-read from L1.
    uint32_t take = 0;
    if (base + kThreads * 4 * kPassLoads <= row_end && lo >= 0x80000000u) {
      // lo is a non-negative float's key: key(x) >= lo exactly when x's bits, read as a signed
      // integer, are >= lo's float bits (negative x and -NaN read negative; +NaN above +inf).
      const int lo_bits = static_cast<int>(lo & 0x7FFFFFFFu);
#pragma unroll
      for (int u = 0; u < kPassLoads; ++u) {
        take |= (static_cast<int>(v[u].x) >= lo_bits ? 1u : 0u) << (4 * u);
        take |= (static_cast<int>(v[u].y) >= lo_bits ? 1u : 0u) << (4 * u + 1);
        take |= (static_cast<int>(v[u].z) >= lo_bits ? 1u : 0u) << (4 * u + 2);
        take |= (static_cast<int>(v[u].w) >= lo_bits ? 1u : 0u) << (4 * u + 3);
      }
    } else if (base + kThreads * 4 * kPassLoads <= row_end) {
#pragma unroll
      for (int u = 0; u < kPassLoads; ++u) {
        take |= (order_key(v[u].x) >= lo ? 1u : 0u) << (4 * u);
        take |= (order_key(v[u].y) >= lo ? 1u : 0u) << (4 * u + 1);
        take |= (order_key(v[u].z) >= lo ? 1u : 0u) << (4 * u + 2);
        take |= (order_key(v[u].w) >= lo ? 1u : 0u) << (4 * u + 3);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kPassLoads; ++u) {
        const int i = base + (u * kThreads + tid) * 4;
        const uint32_t e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (i + k < row_end && order_key(e[k]) >= lo) take |= 1u << (4 * u + k);
      }
    }
    const int cnt = __popc(take);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int n = 0;
    if (lane == 31 && incl > 0) n = atomicAdd(&s_nbuf, incl);
    n = __shfl_sync(0xffffffffu, n, 31) + incl - cnt;
    while (take) {
      const int bit = __ffs(take) - 1;
      take &= take - 1;
      const int i = base + ((bit >> 2) * kThreads + tid) * 4 + (bit & 3);
      const uint32_t key = order_key(ldg_bits(row + i));
      atomicAdd(&s_h[key >> 21], 1u);
      if (n < kBufKeys) {
        s_bkey[n] = key;
        s_bidx[n] = i;
      }
      ++n;
    }
  }
  __syncthreads();
  const int nb = s_nbuf;
  if (nb < K || nb > kBufKeys) return false;
  return finish_from_buffer(s_bkey, s_bidx, nb, -2, static_cast<unsigned>(K), K, top_k, slots,
                            &s_cand, s_h, cand_out, tie_out, thr_out);
}

// Two-sweep repair of a row (see the file comment); false if the bin holding v has more keys than
// the buffer, or more tied keys than can be ranked, in which case nothing it wrote is counted and
// the caller falls back to repair_row.
__device__ bool repair_row_fast(const float *row, int row_end, int K, int top_k, int2 *slots,
                                int *cand_out, int *tie_out, uint32_t *thr_out, uint8_t *dyn) {
  unsigned *s_h = reinterpret_cast<unsigned *>(dyn);                // [2048]
  uint32_t *s_bkey = reinterpret_cast<uint32_t *>(dyn + 2048 * 4);  // [kBufKeys]
  int *s_bidx = reinterpret_cast<int *>(s_bkey + kBufKeys);         // [kBufKeys]
  __shared__ int s_bin, s_nbuf, s_cand;
  __shared__ unsigned s_above;
  __shared__ int s_warp[kWarps];
  const int tid = threadIdx.x;
  for (int i = tid; i < 2048; i += kThreads) s_h[i] = 0;
  if (tid == 0) {
    s_nbuf = 0;
    s_cand = 0;
    s_bin = 0;
    s_above = 0;
  }
  __syncthreads();
  // ---- sweep 1: histogram of the leading 11 key bits
  for (int base = 0; base < row_end; base += kThreads * 4 * kPassLoads) {
    uint4 v[kPassLoads];
    load_pass(row, row_end, base, v);
#pragma unroll
    for (int u = 0; u < kPassLoads; ++u) {
      const int i = base + (u * kThreads + tid) * 4;
      const uint32_t e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (i + k < row_end) atomicAdd(&s_h[order_key(e[k]) >> 21], 1u);
    }
  }
  __syncthreads();
  find_bin(s_h, 2048, static_cast<unsigned>(K), &s_bin, &s_above, s_warp);
  const uint32_t b1 = static_cast<uint32_t>(s_bin);
  const unsigned above1 = s_above;
  const int nb = static_cast<int>(s_h[b1]);
  if (nb > kBufKeys) return false;
  // ---- sweep 2: keys of higher bins are candidates; the bin's own keys go to the buffer
  for (int base = 0; base < row_end; base += kThreads * 4 * kPassLoads) {
    uint4 v[kPassLoads];
    load_pass(row, row_end, base, v);
#pragma unroll
    for (int u = 0; u < kPassLoads; ++u) {
      const int i = base + (u * kThreads + tid) * 4;
      const uint32_t e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (i + k >= row_end) continue;
        const uint32_t key = order_key(e[k]);
        const uint32_t bin = key >> 21;
        if (bin > b1) {
          const int n = atomicAdd(&s_cand, 1);
          slots[top_k + n] = make_int2(i + k, static_cast<int>(e[k]));
        } else if (bin == b1) {
          const int n = atomicAdd(&s_nbuf, 1);
          s_bkey[n] = key;
          s_bidx[n] = i + k;
        }
      }
    }
  }
  __syncthreads();
  return finish_from_buffer(s_bkey, s_bidx, nb, static_cast<int>(b1),
                            static_cast<unsigned>(K) - above1, K, top_k, slots, &s_cand, s_h,
                            cand_out, tie_out, thr_out);
}

// Repairs a row (called by every thread of the repairing CTA): see the file comment.
__device__ void repair_row(const float *row, int row_end, int K, int top_k, int2 *slots,
                           int *cand_out, int *tie_out, uint32_t *thr_out) {
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
    // kPassLoads 16-byte loads per thread in flight before any is used (the row is L2-resident; one
    // load at a time would leave each pass bound by the L2 latency).
    for (int base = 0; base < row_end; base += kThreads * 4 * kPassLoads) {
      uint4 v[kPassLoads];
      load_pass(row, row_end, base, v);
#pragma unroll
      for (int u = 0; u < kPassLoads; ++u) {
        const int i = base + (u * kThreads + tid) * 4;
        const uint32_t e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t key = order_key(e[k]);
          if (i + k < row_end && (key & mask) == prefix)
            atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
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
    // Each thread takes kSweepKeys consecutive keys (four 16-byte loads in flight), so that one
    // block scan per span ranks the ties in index order.
    const int first = i0 + tid * kSweepKeys;
    uint32_t keys[kSweepKeys];
    if (first + kSweepKeys - 1 < row_end) {
      uint4 v[kSweepKeys / 4];
#pragma unroll
      for (int u = 0; u < kSweepKeys / 4; ++u)
        v[u] = __ldg(reinterpret_cast<const uint4 *>(row + first) + u);
#pragma unroll
      for (int u = 0; u < kSweepKeys / 4; ++u) {
        keys[4 * u] = order_key(v[u].x);
        keys[4 * u + 1] = order_key(v[u].y);
        keys[4 * u + 2] = order_key(v[u].z);
        keys[4 * u + 3] = order_key(v[u].w);
      }
    } else {
#pragma unroll
      for (int k = 0; k < kSweepKeys; ++k)  // key 0 is below every real key's tie/candidate
        keys[k] = first + k < row_end ? order_key(ldg_bits(row + first + k)) : 0u;
    }
    int mine = 0;
#pragma unroll
    for (int k = 0; k < kSweepKeys; ++k) {
      const bool valid = first + k < row_end;
      if (valid && keys[k] > vkey) {
        const int n = atomicAdd(&s_cand, 1);
        if (n < c) slots[top_k + n] = make_int2(first + k, static_cast<int>(key_bits(keys[k])));
      }
      mine += (valid && keys[k] == vkey) ? 1 : 0;
    }
    int total;
    int rank = s_tie_base + block_scan(mine, s_warp, &total);
#pragma unroll
    for (int k = 0; k < kSweepKeys; ++k) {
      if (first + k < row_end && keys[k] == vkey) {
        if (rank < m)
          slots[top_k - 1 - rank] = make_int2(first + k, static_cast<int>(key_bits(vkey)));
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
    *thr_out = key_bits(vkey);
  }
}

// Repair of a row of K' = row_end keys (at most top_k): every key is selected, so v is the row's
// smallest key (one reduction) and one pass writes the keys above it as candidates and the keys
// equal to it as ties, with no radix passes.
__device__ void repair_all_keys(const float *row, int row_end, int top_k, int2 *slots, int *c_out,
                                int *m_out, uint32_t *v_out) {
  __shared__ unsigned s_min;
  __shared__ int s_nc, s_nt;
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) {
    s_min = 0xFFFFFFFFu;
    s_nc = 0;
    s_nt = 0;
  }
  __syncthreads();
  unsigned mn = 0xFFFFFFFFu;
  for (int i = tid; i < row_end; i += kThreads) mn = min(mn, order_key(ldg_bits(row + i)));
  mn = __reduce_min_sync(0xffffffffu, mn);
  if (lane == 0) atomicMin(&s_min, mn);
  __syncthreads();
  const uint32_t v = s_min;
  for (int i0 = 0; i0 < row_end; i0 += kThreads) {  // slots reserved with one atomic per warp
    const int i = i0 + tid;
    const uint32_t key = i < row_end ? order_key(ldg_bits(row + i)) : 0u;
    const bool is_c = i < row_end && key > v;
    const bool is_t = i < row_end && key == v;
    const unsigned mc = __ballot_sync(0xffffffffu, is_c);
    if (mc) {
      const int leader = __ffs(mc) - 1;
      int n = 0;
      if (lane == leader) n = atomicAdd(&s_nc, __popc(mc));
      n = __shfl_sync(0xffffffffu, n, leader) + __popc(mc & lanemask_lt());
      if (is_c) slots[top_k + n] = make_int2(i, static_cast<int>(key_bits(key)));
    }
    const unsigned mt = __ballot_sync(0xffffffffu, is_t);
    if (mt) {
      const int leader = __ffs(mt) - 1;
      int n = 0;
      if (lane == leader) n = atomicAdd(&s_nt, __popc(mt));
      n = __shfl_sync(0xffffffffu, n, leader) + __popc(mt & lanemask_lt());
      if (is_t) slots[top_k - 1 - n] = make_int2(i, static_cast<int>(key_bits(v)));
    }
  }
  __syncthreads();
  if (tid == 0) {
    *c_out = s_nc;
    *m_out = s_nt;
    *v_out = key_bits(v);
  }
}

// Repairs a row that does not fit (every thread of the CTA calls it): its slots get exactly its
// top-K', and *c_out / *m_out / *v_out (shared) the keys above v, the keys equal to v kept, and v.
// thr, nc, nt: the row's threshold and classification counts.
__device__ __forceinline__ void repair_any(const float *row, int row_end, int K, float thr, int nc,
                                           int nt, int top_k, int2 *slots, int *c_out, int *m_out,
                                           uint32_t *v_out, uint8_t *dyn) {
  // The threshold bounds the K'-th key from below when at least K' and at most a buffer's worth
  // of keys were counted at or above it (NaN thresholds excepted).
  if (K == row_end) {  // a row of at most top_k keys: all of them
    repair_all_keys(row, row_end, top_k, slots, c_out, m_out, v_out);
    __syncthreads();
    return;
  }
  const bool hint = thr == thr && nc + nt >= K && nc + nt <= kBufKeys;
  const uint32_t thr_key = order_key(__float_as_uint(thr));
  if (!repair_row_gather(row, row_end, K, top_k, slots, hint, thr_key, c_out, m_out, v_out, dyn)) {
    __syncthreads();
    if (!repair_row_fast(row, row_end, K, top_k, slots, c_out, m_out, v_out, dyn)) {
      __syncthreads();
      repair_row(row, row_end, K, top_k, slots, c_out, m_out, v_out);
    }
  }
  __syncthreads();
}

// Classifies keys [begin, end) of row r (a chunk of at most kChunk keys); every thread of the
// CTA calls it.
__device__ __forceinline__ void classify_chunk(const SelectArgs &a, int r, int begin, int end) {
  const int tid = threadIdx.x;
  const float thr = a.thresholds[r];
  const float *row = a.logits + static_cast<int64_t>(r) * a.row_stride;
  int2 *slots = reinterpret_cast<int2 *>(a.candidates) +
                static_cast<int64_t>(r) * (a.top_k + a.capacity);
  int *counter = a.counters + 2 * r;
  float4 v[kSweepLoads];  // all of this thread's loads in flight before any is classified
#pragma unroll
  for (int u = 0; u < kSweepLoads; ++u) {
    const int i = begin + (u * kClsThreads + tid) * 4;
    if (i + 3 < end) {
      v[u] = __ldg(reinterpret_cast<const float4 *>(row + i));
    } else {
      v[u].x = i < end ? row[i] : 0.0f;
      v[u].y = i + 1 < end ? row[i + 1] : 0.0f;
      v[u].z = i + 2 < end ? row[i + 2] : 0.0f;
      v[u].w = 0.0f;
    }
  }
  // The thread's candidates and ties as bit masks; one warp scan of both counts and one
  // atomicAdd per warp and kind reserve all the warp's slots at once (a reservation per
  // 32 keys would put a round trip to L2 on the path for each of them).
  static_assert(kSweepLoads * 4 <= 16, "16 keys per thread fit the 16-bit counts");
  uint32_t cm = 0, tm = 0;
#pragma unroll
  for (int u = 0; u < kSweepLoads; ++u) {
    const int i = begin + (u * kClsThreads + tid) * 4;
    const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const bool valid = i + k < end;
      const float s = e[k];
      cm |= (valid && s > thr ? 1u : 0u) << (4 * u + k);
      tm |= (valid && !(s > thr) && !(s < thr) ? 1u : 0u) << (4 * u + k);
    }
  }
  const int lane = tid & 31;
  const int mine = __popc(cm) | (__popc(tm) << 16);  // a warp's sums stay below 2^16
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int excl = incl - mine;
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int bc = 0, bt = 0;
  if (lane == 0) {
    if (total & 0xFFFF) bc = atomicAdd(counter, total & 0xFFFF);
    if (total >> 16) bt = atomicAdd(counter + 1, total >> 16);
  }
  int nc = __shfl_sync(0xffffffffu, bc, 0) + (excl & 0xFFFF);
  int nt = __shfl_sync(0xffffffffu, bt, 0) + (excl >> 16);
  // The few keys taken are re-read (L1 hits) rather than kept in registers.
  for (uint32_t m = cm | tm; m != 0u; m &= m - 1u) {
    const int bit = __ffs(m) - 1;
    const int i = begin + ((bit >> 2) * kClsThreads + tid) * 4 + (bit & 3);
    const int2 item = make_int2(i, static_cast<int>(ldg_bits(row + i)));
    if ((cm >> bit) & 1u) {
      if (nc < a.capacity) slots[a.top_k + nc] = item;
      ++nc;
    } else {
      if (nt < a.top_k) slots[a.top_k - 1 - nt] = item;
      ++nt;
    }
  }
}

// Launch 1, one CTA per chunk: CTA (r, c) classifies keys [c*kChunk, (c+1)*kChunk) of row r
// below row_ends[r]; a CTA past the row's keys leaves at once.  The rows are the grid's fast
// dimension, so every row's first chunk is dispatched before any row's second: with rows of
// mixed lengths, the CTAs with keys start in the first wave and those past the ends come last.
__global__ void __launch_bounds__(kClsThreads) k_select_classify(const SelectArgs a) {
  // The previous kernel in the stream may still be running: no global memory before this.
  griddep_wait();
  griddep_launch_dependents();
  const int r = blockIdx.x;
  int row_end = a.row_ends[r];
  row_end = row_end < 0 ? 0 : (row_end > a.max_context ? a.max_context : row_end);
  const int begin = blockIdx.y * kChunk;
  const int end = min(begin + kChunk, row_end);
  if (begin >= end) return;
  classify_chunk(a, r, begin, end);
}

// Launch 2 (with arrivals), at most one row per SM: CTA r applies the fit rule to row r and
// repairs it if it does not fit.  It starts once launch 1 has finished and its writes are visible
// (programmatic dependent launch: griddepcontrol.wait returns only then), so the counts are
// final.
__global__ void __launch_bounds__(kThreads) k_select_finish_row(const SelectArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t select_smem[];
  __shared__ int s_c, s_m;
  __shared__ uint32_t s_v;
  const int tid = threadIdx.x;
  const int r = blockIdx.x;
  int row_end = a.row_ends[r];
  row_end = row_end < 0 ? 0 : (row_end > a.max_context ? a.max_context : row_end);
  const int K = row_end < a.top_k ? row_end : a.top_k;
  int *counter = a.counters + 2 * r;
  const int nc = counter[0], nt = counter[1];
  if (row_fits(nc, nt, K, a.top_k, a.capacity)) {
    if (tid == 0) {
      a.ranges[r] = a.top_k - min(nt, a.top_k);
      a.ranges[a.rows + r] = a.top_k + min(nc, a.capacity);
      a.arrivals[r] = 0;
    }
    return;
  }
  int2 *slots = reinterpret_cast<int2 *>(a.candidates) +
                static_cast<int64_t>(r) * (a.top_k + a.capacity);
  repair_any(a.logits + static_cast<int64_t>(r) * a.row_stride, row_end, K, a.thresholds[r], nc,
             nt, a.top_k, slots, &s_c, &s_m, &s_v, select_smem);
  if (tid == 0) {
    counter[0] = s_c;
    counter[1] = s_m;
    reinterpret_cast<uint32_t *>(a.thresholds)[r] = s_v;  // v's own bits
    a.ranges[r] = a.top_k - s_m;
    a.ranges[a.rows + r] = a.top_k + s_c;
    a.arrivals[r] = 0;
  }
}

// Launch 2 (with arrivals), more rows than SMs: CTA j takes rows j, j + gridDim.x, ...: one
// thread per row applies the fit rule and writes the slot range of a row that fits (and zeroes
// its arrivals entry); the rows that do not fit are then repaired one after another by the
// whole CTA.
__global__ void __launch_bounds__(kThreads) k_select_finish(const SelectArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t select_smem[];
  __shared__ int s_list[kThreads];  // this round's rows that do not fit
  __shared__ int s_n;
  __shared__ int s_c, s_m;
  __shared__ uint32_t s_v;
  const int tid = threadIdx.x;
  const auto clamp_end = [&](int r) {
    const int e = a.row_ends[r];
    return e < 0 ? 0 : (e > a.max_context ? a.max_context : e);
  };
  const int stride = gridDim.x;
  for (int first = blockIdx.x; first < a.rows; first += stride * kThreads) {
    if (tid == 0) s_n = 0;
    __syncthreads();
    const int r = first + tid * stride;
    if (r < a.rows) {
      const int row_end = clamp_end(r);
      const int K = row_end < a.top_k ? row_end : a.top_k;
      const int nc = a.counters[2 * r], nt = a.counters[2 * r + 1];
      if (row_fits(nc, nt, K, a.top_k, a.capacity)) {
        a.ranges[r] = a.top_k - min(nt, a.top_k);
        a.ranges[a.rows + r] = a.top_k + min(nc, a.capacity);
      } else {
        s_list[atomicAdd(&s_n, 1)] = r;
      }
      a.arrivals[r] = 0;
    }
    __syncthreads();
    const int n = s_n;
    for (int j = 0; j < n; ++j) {
      const int rr = s_list[j];
      const int row_end = clamp_end(rr);
      const int K = row_end < a.top_k ? row_end : a.top_k;
      int *counter = a.counters + 2 * rr;
      int2 *slots = reinterpret_cast<int2 *>(a.candidates) +
                    static_cast<int64_t>(rr) * (a.top_k + a.capacity);
      repair_any(a.logits + static_cast<int64_t>(rr) * a.row_stride, row_end, K,
                 a.thresholds[rr], counter[0], counter[1], a.top_k, slots, &s_c, &s_m, &s_v,
                 select_smem);
      if (tid == 0) {
        counter[0] = s_c;
        counter[1] = s_m;
        reinterpret_cast<uint32_t *>(a.thresholds)[rr] = s_v;  // v's own bits
        a.ranges[rr] = a.top_k - s_m;
        a.ranges[a.rows + rr] = a.top_k + s_c;
      }
      __syncthreads();
    }
  }
}

// The last stage of the fused score + select: CTA (b, t) for row r = b * next_n + t, after the
// fused pass (counts and slots) and the rescoring launch (the logits of every request with a row
// that does not fit, in the scratch rows).  A row that fits gets its slot range; one that does
// not is repaired from its scratch row.
__global__ void __launch_bounds__(kThreads) k_fused_repair(const FusedRepairArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ __align__(16) uint8_t select_smem[];
  const int b = blockIdx.x, t = blockIdx.y;
  const int len = max(0, a.seq_lens[static_cast<int64_t>(b) * a.sl_stride]);
  const int r = b * a.next_n + t;
  const int rows = a.batch * a.next_n;
  const int row_end = max(0, len - a.next_n + t + 1);
  const int K = min(row_end, a.top_k);
  int *counter = a.counters + 2 * r;
  const int nc = counter[0], nt = counter[1];
  if (row_fits(nc, nt, K, a.top_k, a.capacity)) {
    if (threadIdx.x == 0) {
      a.ranges[r] = a.top_k - min(nt, a.top_k);
      a.ranges[rows + r] = a.top_k + min(nc, a.capacity);
    }
    return;
  }
  __shared__ int s_c, s_m;
  __shared__ uint32_t s_v;
  int2 *slots = reinterpret_cast<int2 *>(a.candidates) +
                static_cast<int64_t>(r) * (a.top_k + a.capacity);
  repair_any(a.scratch + static_cast<int64_t>(r) * a.scratch_stride, row_end, K, a.thresholds[r],
             nc, nt, a.top_k, slots, &s_c, &s_m, &s_v, select_smem);
  if (threadIdx.x == 0) {
    counter[0] = s_c;
    counter[1] = s_m;
    reinterpret_cast<uint32_t *>(a.thresholds)[r] = s_v;
    a.ranges[r] = a.top_k - s_m;
    a.ranges[rows + r] = a.top_k + s_c;
  }
}

}  // namespace

cudaError_t launch_threshold_select(const SelectArgs &args, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int per_row = args.max_context > 0 ? (args.max_context + kChunk - 1) / kChunk : 1;
  e = launch_dependent(k_select_classify, dim3(args.rows, per_row), dim3(kClsThreads), 0, stream,
                       args);
  if (e != cudaSuccess || args.arrivals == nullptr) return e;
  static PerDeviceOnce configured;
  e = configured.run([] {
    cudaError_t e2 = cudaFuncSetAttribute(
        k_select_finish_row, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelectSmem);
    if (e2 != cudaSuccess) return e2;
    return cudaFuncSetAttribute(k_select_finish, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSelectSmem);
  });
  if (e != cudaSuccess) return e;
  if (args.rows <= sms)
    return launch_dependent(k_select_finish_row, dim3(args.rows), dim3(kThreads), kSelectSmem,
                            stream, args);
  return launch_dependent(k_select_finish, dim3(sms), dim3(kThreads), kSelectSmem, stream, args);
}

cudaError_t launch_fused_repair(const FusedRepairArgs &args, cudaStream_t stream) {
  static PerDeviceOnce configured;
  const cudaError_t e = configured.run([] {
    return cudaFuncSetAttribute(k_fused_repair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSelectSmem);
  });
  if (e != cudaSuccess) return e;
  return launch_dependent(k_fused_repair, dim3(args.batch, args.next_n), dim3(kThreads),
                          kSelectSmem, stream, args);
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
