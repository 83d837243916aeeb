// logits.cu -- paged FP8 MQA logits on sm_103a ("flashinfer.attn_scores",
// fp8_paged_mqa_logits: formula block, Note, Parameters).
//
//   out[b*n + t, p] = scale[p] * sum_h w[b*n + t, h] * relu(q[b, t, h, :] . k[p, :])
//
// One persistent CTA per SM walks a contiguous run of 128-position KV tiles (split.cuh).
// Warp roles, all iterating the same tile sequence:
//   warp 0     producer: reads the block table 32 entries at a time, and for each tile TMA-loads
//              the two 64-token pages' e4m3 values (8 KiB each, 128-byte swizzled) and bulk-
//              copies their 256-byte float32 scale regions into one pipeline stage; loads q
//              and w of each new request into one of two q/w buffers.
//   warp 1     MMA issuer (one thread): per tile, 4 x tcgen05.mma.kind::f8f6f4 (K = 32 each)
//              D[128 positions, n*64 query rows] += K_tile[128, 32] * q[n*64, 32]^T into a
//              TMEM accumulator (float32), then commits to the stage's and the accumulator's
//              barriers.  The KV tile is the MMA's M side, so TMEM lane = KV position.
//   warps 2-5  epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (one position per thread),
//              computes scale * sum_h w_h * max(s_h, 0) for each draft slot in float32, and
//              stores it: 32 consecutive positions per warp, one 128-byte line per row.
// The per-head reduction is per-thread (heads are TMEM columns of the thread's own lane), so it
// needs no shuffles.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/idx.h"
#include "internal.h"
#include "ptx.cuh"
#include "split.cuh"

namespace idx {

__device__ int g_logits_status;

namespace {

constexpr int kThreads = 192;                     // 6 warps
constexpr int kHeads = 64;
constexpr int kHeadDim = 128;
constexpr int kBlock = 64;                        // tokens per page
constexpr int kPageBytes = kBlock * (kHeadDim + 4);  // 8448
constexpr int kPageRows = kPageBytes / 128;       // 66 rows of 128 bytes per page
constexpr int kValueBytes = kBlock * kHeadDim;    // 8192
constexpr uint32_t kStageBytes = kTileTokens * kHeadDim;  // 16384: two pages of values
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far beyond any legitimate wait

template <int NN>
struct Cfg {
  static constexpr int N = NN * kHeads;  // MMA N: query rows of one request
  static constexpr int STAGES = NN == 1 ? 10 : (NN == 2 ? 10 : (NN == 3 ? 9 : 8));
  static constexpr int ACC = NN <= 2 ? 4 : 2;
  static constexpr int TMEM_COLS = (ACC * N <= 256) ? 256 : 512;
  static constexpr uint32_t Q_BYTES = N * kHeadDim;
  static constexpr uint32_t W_FLOATS = NN * kHeads;
  static constexpr uint32_t OFF_KV = 0;
  static constexpr uint32_t OFF_Q = OFF_KV + STAGES * kStageBytes;
  static constexpr uint32_t OFF_SCALE = OFF_Q + 2 * Q_BYTES;
  static constexpr uint32_t OFF_W = OFF_SCALE + STAGES * kTileTokens * 4;
  static constexpr uint32_t OFF_BAR = OFF_W + 2 * W_FLOATS * 4;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * ACC + 4 + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t OFF_LEN = OFF_MISC + 128;
  static constexpr uint32_t smem_bytes(int batch) {
    return OFF_LEN + 4u * static_cast<uint32_t>(batch) + 1024u;  // + alignment slack
  }
  static_assert(OFF_Q % 1024 == 0 && Q_BYTES % 1024 == 0, "swizzled tiles 1024-aligned");
  static_assert(OFF_SCALE % 16 == 0 && OFF_W % 16 == 0, "bulk-copy destinations");
  static_assert(smem_bytes(kMaxBatch) <= 232448, "fits the 227 KiB per-CTA limit");
  static_assert(ACC * N <= TMEM_COLS, "accumulators fit the allocation");
};

__device__ __forceinline__ void flag_error(int bits) { atomicOr(&g_logits_status, bits); }

// scale-free part of one logit: sum over the 64 heads of w_h * max(s_h, 0), in float32 with
// eight interleaved partial sums (eight terms each) combined pairwise.
__device__ __forceinline__ float weighted_relu_sum(const uint32_t (&lo)[32],
                                                   const uint32_t (&hi)[32], const float *w) {
  const float4 *w4 = reinterpret_cast<const float4 *>(w);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 ww = w4[i];
    const int base = (i & 1) * 4;
    acc[base + 0] = fmaf(ww.x, fmaxf(__uint_as_float(lo[4 * i + 0]), 0.0f), acc[base + 0]);
    acc[base + 1] = fmaf(ww.y, fmaxf(__uint_as_float(lo[4 * i + 1]), 0.0f), acc[base + 1]);
    acc[base + 2] = fmaf(ww.z, fmaxf(__uint_as_float(lo[4 * i + 2]), 0.0f), acc[base + 2]);
    acc[base + 3] = fmaf(ww.w, fmaxf(__uint_as_float(lo[4 * i + 3]), 0.0f), acc[base + 3]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 ww = w4[8 + i];
    const int base = (i & 1) * 4;
    acc[base + 0] = fmaf(ww.x, fmaxf(__uint_as_float(hi[4 * i + 0]), 0.0f), acc[base + 0]);
    acc[base + 1] = fmaf(ww.y, fmaxf(__uint_as_float(hi[4 * i + 1]), 0.0f), acc[base + 1]);
    acc[base + 2] = fmaf(ww.z, fmaxf(__uint_as_float(hi[4 * i + 2]), 0.0f), acc[base + 2]);
    acc[base + 3] = fmaf(ww.w, fmaxf(__uint_as_float(hi[4 * i + 3]), 0.0f), acc[base + 3]);
  }
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

template <int NN>
__global__ void __launch_bounds__(kThreads, 1)
    k_logits_fp8(const __grid_constant__ CUtensorMap kv_map,
                 const __grid_constant__ CUtensorMap q_map, const LogitsArgs a) {
  using C = Cfg<NN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  uint8_t *s_kv = smem + C::OFF_KV;
  uint8_t *s_q = smem + C::OFF_Q;
  float *s_scale = reinterpret_cast<float *>(smem + C::OFF_SCALE);
  float *s_w = reinterpret_cast<float *>(smem + C::OFF_W);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES;
  uint64_t *acc_empty = acc_full + C::ACC;
  uint64_t *q_full = acc_empty + C::ACC;
  uint64_t *q_empty = q_full + 2;
  uint64_t *drain = q_empty + 2;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  int *s_split = reinterpret_cast<int *>(smem + C::OFF_MISC + 16);      // 4 ints
  long long *s_warp = reinterpret_cast<long long *>(smem + C::OFF_MISC + 64);  // 6 int64
  int *s_len = reinterpret_cast<int *>(smem + C::OFF_LEN);
  // Prologue scratch: the inclusive tile prefix lives in the (still unused) KV stages.
  long long *s_incl = reinterpret_cast<long long *>(s_kv);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int batch = a.batch;

  // ---- 1. lengths and this CTA's tile range --------------------------------------------------
  {
    const long long total = load_lengths<kThreads>(a.seq_lens, a.sl_stride, batch, s_len, s_incl,
                                                   s_warp);
    if (tid == 0) {
      int2 s0, s1;
      if (a.schedule != nullptr) {
        s0 = make_int2(__ldg(a.schedule + 2 * blockIdx.x), __ldg(a.schedule + 2 * blockIdx.x + 1));
        s1 = make_int2(__ldg(a.schedule + 2 * blockIdx.x + 2),
                       __ldg(a.schedule + 2 * blockIdx.x + 3));
      } else {
        const long long g = gridDim.x;
        s0 = locate_tile(s_incl, s_len, batch, total * blockIdx.x / g);
        s1 = locate_tile(s_incl, s_len, batch, total * (blockIdx.x + 1) / g);
      }
      s_split[0] = s0.x;
      s_split[1] = s0.y;
      s_split[2] = s1.x;
      s_split[3] = s1.y;
    }
    if (a.row_ends != nullptr) {
      for (int b = blockIdx.x * kThreads + tid; b < batch; b += gridDim.x * kThreads) {
        const int len = s_len[b];
#pragma unroll
        for (int t = 0; t < NN; ++t) a.row_ends[b * NN + t] = max(0, len - NN + t + 1);
      }
    }
  }

  // ---- 2. barriers, tensor memory -------------------------------------------------------------
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + 4);  // MMA commit + one arrival per epilogue warp
    }
    for (int c = 0; c < C::ACC; ++c) {
      mbar_init(&acc_full[c], 1);
      mbar_init(&acc_empty[c], 4);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(&q_full[c], 1);
      mbar_init(&q_empty[c], 1 + 4);
    }
    mbar_init(drain, 1);
    fence_barrier_init();
    prefetch_tensor_map(&kv_map);
    prefetch_tensor_map(&q_map);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  // The prologue wrote the KV stages with ordinary stores; TMA writes them next.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;
  const TileIter first = make_iter(s_split[0], s_split[1], s_split[2], s_split[3], batch, s_len);

  if (warp == 0) {
    // ================================ producer ================================================
    const uint64_t pol_stream = l2_policy_evict_first();
    const uint64_t pol_keep = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int qcount = 0, cur_b = -1;
    int win_b = -1, win_base = 0, win_val = 0;
    int issued = 0;
    bool ok = true;
    for (TileIter it = first; it.valid(); it.next()) {
      const int b = it.b, j = it.j;
      if (b != cur_b) {
        const int qb = qcount & 1;
        if (!mbar_wait(&q_empty[qb], ((qcount >> 1) & 1) ^ 1, kWaitLimitNs)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[qb], C::Q_BYTES + C::W_FLOATS * 4);
          tma_load_2d(s_q + qb * C::Q_BYTES, &q_map, &q_full[qb], 0, b * C::N, pol_keep);
          bulk_load(s_w + qb * C::W_FLOATS, a.weights + static_cast<int64_t>(b) * C::W_FLOATS,
                    C::W_FLOATS * 4, &q_full[qb], pol_keep);
        }
        cur_b = b;
        ++qcount;
      }
      const int npages = s_len[b] / kBlock + (s_len[b] % kBlock != 0 ? 1 : 0);
      const int pg0 = 2 * j;
      const bool has1 = pg0 + 1 < npages;
      if (b != win_b || pg0 < win_base || pg0 >= win_base + 32) {
        win_b = b;
        win_base = pg0 & ~31;
        const int e = win_base + lane;
        win_val = e < npages ? __ldg(a.block_tables + static_cast<int64_t>(b) * a.bt_stride + e) : 0;
      }
      const int page0 = __shfl_sync(0xffffffffu, win_val, pg0 - win_base);
      const int page1 = __shfl_sync(0xffffffffu, win_val, pg0 + 1 - win_base);
      if (!mbar_wait(&empty[stage], phase ^ 1, kWaitLimitNs)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const bool v0 = page0 >= 0 && page0 < a.num_blocks;
        const bool v1 = has1 && page1 >= 0 && page1 < a.num_blocks;
        if (!v0 || (has1 && !v1)) flag_error(IDX_DEV_BAD_PAGE);
        mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(kPageBytes) * (v0 + v1));
        uint8_t *dst = s_kv + stage * kStageBytes;
        float *sdst = s_scale + stage * kTileTokens;
        if (v0) {
          tma_load_2d(dst, &kv_map, &full[stage], 0, page0 * kPageRows, pol_stream);
          bulk_load(sdst, a.kv + static_cast<int64_t>(page0) * kPageBytes + kValueBytes,
                    kBlock * 4, &full[stage], pol_stream);
        }
        if (v1) {
          tma_load_2d(dst + kValueBytes, &kv_map, &full[stage], 0, page1 * kPageRows, pol_stream);
          bulk_load(sdst + kBlock, a.kv + static_cast<int64_t>(page1) * kPageBytes + kValueBytes,
                    kBlock * 4, &full[stage], pol_stream);
        }
      }
      __syncwarp();
      ++issued;
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!ok) flag_error(IDX_DEV_WAIT_TIMEOUT);
    // Never leave copies in flight: wait for the last loads issued into each stage.
    const int tail = issued < C::STAGES ? issued : C::STAGES;
    for (int k = 1; k <= tail; ++k) {
      const int s = ((stage - k) % C::STAGES + C::STAGES) % C::STAGES;
      const uint32_t ph = (stage - k < 0) ? (phase ^ 1) : phase;
      if (!mbar_wait(&full[s], ph, kWaitLimitNs)) flag_error(IDX_DEV_WAIT_TIMEOUT);
    }
    if (qcount > 0 &&
        !mbar_wait(&q_full[(qcount - 1) & 1], ((qcount - 1) >> 1) & 1, kWaitLimitNs))
      flag_error(IDX_DEV_WAIT_TIMEOUT);
  } else if (warp == 1) {
    // ================================ MMA issuer ==============================================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kTileTokens, C::N);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int qcount = 0, cur_b = -1, qb = 0;
      bool ok = true;
      for (TileIter it = first; it.valid();) {
        const int b = it.b;
        if (b != cur_b) {
          qb = qcount & 1;
          if (!mbar_wait(&q_full[qb], (qcount >> 1) & 1, kWaitLimitNs)) {
            ok = false;
            break;
          }
          cur_b = b;
          ++qcount;
        }
        if (!mbar_wait(&full[stage], phase, kWaitLimitNs) ||
            !mbar_wait(&acc_empty[acc], acc_phase ^ 1, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = smem_addr(s_kv + stage * kStageBytes);
        const uint32_t b_addr = smem_addr(s_q + qb * C::Q_BYTES);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::N);
#pragma unroll
        for (int k = 0; k < kHeadDim / 32; ++k)
          mma_f8f6f4(d_tmem, smem_desc_sw128(a_addr + 32 * k), smem_desc_sw128(b_addr + 32 * k),
                     idesc, k > 0 ? 1u : 0u);
        mma_commit(&empty[stage]);
        mma_commit(&acc_full[acc]);
        it.next();
        if (!it.valid() || it.b != b) mma_commit(&q_empty[qb]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (++acc == C::ACC) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) flag_error(IDX_DEV_WAIT_TIMEOUT);
      // Every MMA issued above has completed once this commit arrives.
      mma_commit(drain);
      if (!mbar_wait(drain, 0, kWaitLimitNs)) flag_error(IDX_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ================================ epilogue ================================================
    const int quarter = warp & 3;
    const int pos = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    int qcount = 0, cur_b = -1, qb = 0;
    bool ok = true;
    for (TileIter it = first; it.valid();) {
      const int b = it.b, j = it.j;
      if (b != cur_b) {
        qb = qcount & 1;
        if (!mbar_wait(&q_full[qb], (qcount >> 1) & 1, kWaitLimitNs)) {
          ok = false;
          break;
        }
        cur_b = b;
        ++qcount;
      }
      // The stage's scales (the MMA has consumed its values already or will shortly).
      if (!mbar_wait(&full[stage], phase, kWaitLimitNs)) {
        ok = false;
        break;
      }
      const float scale = s_scale[stage * kTileTokens + pos];
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (!mbar_wait(&acc_full[acc], acc_phase, kWaitLimitNs)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float *w = s_w + qb * C::W_FLOATS;
      const int p = j * kTileTokens + pos;
      const bool store = p < s_len[b];
      float *dst = a.out + static_cast<int64_t>(b * NN) * a.out_stride + p;
      // One draft slot at a time (a rolled loop: unrolled, ptxas hoists the next slot's TMEM
      // loads above this slot's arithmetic and runs out of registers at next_n >= 3).
#pragma unroll 1
      for (int t = 0; t < NN; ++t) {
        uint32_t lo[32], hi[32];
        const uint32_t col = static_cast<uint32_t>(acc * C::N + t * kHeads);
        tmem_ld_32x32b_x32(lane_base + col, lo);
        tmem_ld_32x32b_x32(lane_base + col + 32, hi);
        tmem_ld_wait();
        reg_fence(lo);
        reg_fence(hi);
        const float v = scale * weighted_relu_sum(lo, hi, w + t * kHeads);
        if (store) dst[static_cast<int64_t>(t) * a.out_stride] = v;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      it.next();
      if (!it.valid() || it.b != b) {
        if (lane == 0) mbar_arrive(&q_empty[qb]);
      }
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1;
      }
      if (++acc == C::ACC) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (!ok) flag_error(IDX_DEV_WAIT_TIMEOUT);
  }

  // ---- 3. teardown ----------------------------------------------------------------------------
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int NN>
cudaError_t launch_nn(const CUtensorMap &kv_map, const CUtensorMap &q_map, const LogitsArgs &args,
                      int num_ctas, cudaStream_t stream) {
  using C = Cfg<NN>;
  const uint32_t smem = C::smem_bytes(args.batch);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_logits_fp8<NN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::smem_bytes(kMaxBatch));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k_logits_fp8<NN><<<num_ctas, kThreads, smem, stream>>>(kv_map, q_map, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_logits_fp8(int next_n, const CUtensorMap &kv_map, const CUtensorMap &q_map,
                              const LogitsArgs &args, int num_ctas, cudaStream_t stream) {
  switch (next_n) {
    case 1: return launch_nn<1>(kv_map, q_map, args, num_ctas, stream);
    case 2: return launch_nn<2>(kv_map, q_map, args, num_ctas, stream);
    case 3: return launch_nn<3>(kv_map, q_map, args, num_ctas, stream);
    case 4: return launch_nn<4>(kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t logits_status(int32_t *value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_logits_status, sizeof(int32_t));
  if (e != cudaSuccess || !clear) return e;
  const int32_t zero = 0;
  return cudaMemcpyToSymbol(g_logits_status, &zero, sizeof(int32_t));
}

}  // namespace idx
