// logits_kernel.cuh -- paged FP8 MQA logits on sm_103a ("flashinfer.attn_scores",
// fp8_paged_mqa_logits: formula block, Note, Parameters).
//
//   out[b*n + t, p] = scale[p] * sum_h w[b*n + t, h] * relu(q[b, t, h, :] . k[p, :])
//
// One persistent CTA per SM owns a contiguous run of 128-position KV tiles (split.cuh).  Warp 0
// first turns the run into a tile list in shared memory, up to kMaxList tiles at a time:
// {request | first/last-of-request flags | present pages | request ordinal, tile, page ids of
// its one to four pages (of 128, 64 or 32 tokens; the kernel is instantiated per page size)},
// issuing the block-table reads of the whole list in parallel.  The producer and the MMA issuer
// then walk the whole list, each epilogue team only its own tiles:
// The kernel is instantiated per head count H (8, 16, 32, 64), head_dim D (64, 128, 192), output
// type and page size; H = 64, D = 128 below.  A row of 64 or 128 e4m3 bytes is one swizzle atom
// wide (64- or 128-byte swizzle); a row of 192 is three 64-byte atoms.
//   warp 0     producer (one thread): per tile, TMA-loads the pages' e4m3 values (128-byte
//              swizzled, 16 KiB per tile) into a KV stage and bulk-copies their float32 scales
//              (512 B per tile) into a scale slot; per request, TMA-loads q and bulk-copies w
//              into one of two q/w buffers.
//   warp 1     MMA issuer (one thread): D/32 = 4 x tcgen05.mma.kind::f8f6f4 (K = 32 each),
//              D[128 positions, n*64 query rows] += K_tile[128, 32] * q[n*64, 32]^T into a
//              float32 TMEM accumulator, then one commit that marks the tile done.
//              The KV tile is the MMA's M side, so TMEM lane = KV position.
//   warps 2-   epilogue, two teams taking alternate tiles: 8 warps, or 16 for next_n*H >= 192,
//              where the two warps of a lane quadrant share a tile's draft slots (four epilogue
//              warps per scheduler hide the arithmetic's latency).  Warp w owns TMEM
//              lanes 32*(w%4)..+31 and reads them with the 16x256b shape, so that a thread
//              holds four positions for 16 of the 64 heads (8 of 32): it needs only those heads'
//              weights, which stay in registers for the whole request.  Per draft slot a thread forms
//              its four partial sums of w_h * max(s_h, 0) in float32 (packed FMAs), the four
//              threads of a quad exchange them (reduce-scatter) so that each ends with one
//              position's complete sum, and the warp stores 32 consecutive positions (one
//              128-byte line per output row) after multiplying by the position's scale.
// Fused select ("flashinfer.sdsa.indexer_threshold_select": description).  Instantiated with
// SelectOut, the epilogue classifies each score against its row's threshold into the row's
// candidate and tie slots (slots.cuh) instead of storing it.  A launch given fit_counters (the
// counts of a finished fused pass) rescores only the requests with a row that does not fit.
// Barriers.  The issuing thread is the serial point of the pipeline, so it waits on one barrier
// and commits to one barrier per tile:
//   full[s]   tile k may be multiplied: its TMA bytes landed (producer's expect_tx), and the
//             accumulator it overwrites is free (the four epilogue warps that read tile k - ACC,
//             or the producer for the first ACC tiles).
//   done[s]   tile k's MMAs completed (one commit): the producer may reuse stage s, and the
//             epilogue may read tile k's accumulator.
// Tile k uses stage k % STAGES and accumulator k % ACC.  With ACC even and ACC <= STAGES the
// parities never alias: the MMA cannot pass tile k + ACC before tile k's epilogue arrived, so
// done[s] cannot complete tile k + STAGES's phase before tile k's epilogue has waited on it.
// A run longer than kMaxList tiles is processed list by list, the whole CTA synchronising between
// lists.

#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "../../include/idx.h"
#include "internal.h"
#include "mx_convert.cuh"
#include "ptx.cuh"
#include "slots.cuh"
#include "split.cuh"

namespace idx {
namespace {

// Device-side status bits (IDX_DEV_*) of the kernels of the including translation unit.
__device__ int g_logits_status;
// Fault injection for testing the time-limited waits (idx_debug_withhold_first_tile): the CTA
// with this index issues none of its first tile's copies, so the waits on that tile run out.
// -1 (the default): off.
__device__ int g_withhold_cta = -1;

constexpr int kEpiWarpBase = 2;                  // epilogue warps 2, 3, ...
constexpr int kMaxList = 256;                     // tiles per tile list
constexpr int kFirstFlag = 1 << 16;               // record.x = request | flags | page mask
constexpr int kLastFlag = 1 << 17;
constexpr int kMaskShift = 18;                    // bit 18 + p: the tile's page p is present
constexpr int kOrdShift = 22;                     // bits 22-29: the request's ordinal mod 256
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far beyond any legitimate wait

// next_n = NN draft slots of H heads each (H = 8, 16, 32 or 64), head_dim D (64, 128 or 192).
// MX: the KV pool holds MXFP4 pages, which converter warps turn into the e4m3 tile in shared
// memory (D = 128 only).
template <int NN, int H, int D, bool MX_ = false>
struct Cfg {
  static constexpr bool MX = MX_;
  static constexpr int N = NN * H;  // query rows of one request
  // The MMA's N: N rounded up to a multiple of 16 (8 heads at next_n 1 or 3); the extra q rows
  // (the next request's, or zeros past the end of q) give accumulator columns nobody reads.
  static constexpr int NP = (N + 15) / 16 * 16;
  static constexpr int R = H / 8;   // 8-column chunks a thread holds per position and slot
  static constexpr uint32_t STAGE_BYTES = kTileTokens * D;  // a tile's values
  // head_dim 192: rows of 192 bytes are three 64-byte K blocks, each a [rows x 64] tile with the
  // 64-byte swizzle (KB blocks per tile, KBLOCK bytes apart); 64 and 128 are one block of the
  // 64- or 128-byte swizzle.
  static constexpr int KB = D == 192 ? 3 : 1;
  static constexpr uint32_t KBLOCK = kTileTokens * (D / KB);
  // relu_scaled's exactness needs every score below 2^26 in magnitude: D * 448^2 < 2^26.
  static_assert(D == 128 || D == 64 || D == 192, "head_dim 64, 128 or 192");
  // Epilogue: two teams take alternate tiles.  A team has SPLIT warps per TMEM lane quadrant;
  // with N >= 192 the two warps of a quadrant share a tile's draft slots, which gives each
  // scheduler four epilogue warps to hide the arithmetic's latency with.
  static constexpr int SPLIT = N <= 128 ? 1 : 2;
  static constexpr int TEAMS = 2;                       // teams taking tiles in turn
  static constexpr int TEAM_WARPS = 4 * SPLIT;          // warps reading one tile
  static constexpr int EPI_WARPS = TEAMS * TEAM_WARPS;
  // (MX) Converter warps.  A tile's conversion is 256 units (a token's half row: two 32-element
  // groups); eight warps take one unit per thread, or two warps four each where the epilogue's
  // 16 warps leave registers for only two more.
  static constexpr int CONV_WARPS = MX ? (N >= 192 ? 2 : 8) : 0;
  // (MX) The converter warps form groups taking tiles in turn (four groups of two warps, or two
  // of one), so that one tile's waits (for its raw pages and for its stage's previous MMAs)
  // overlap the others' conversions.
  static constexpr int CONV_GROUPS = MX ? (N >= 192 ? 2 : 4) : 1;
  static constexpr int GROUP_WARPS = MX ? CONV_WARPS / CONV_GROUPS : 1;
  static constexpr int CONV_BASE = kEpiWarpBase + EPI_WARPS;  // first converter warp
  static constexpr int THREADS = (kEpiWarpBase + EPI_WARPS + CONV_WARPS) * 32;
  static constexpr int SLOTS = (NN + SPLIT - 1) / SPLIT;  // draft slots per epilogue warp (max)
  // KV stages (e4m3 tiles the MMA reads).  MX: few, since the loads land in a ring of raw MXFP4
  // tiles first (RAW_STAGES of RAW_BYTES: a tile's pages, packed rows then scale bytes each).
  static constexpr int STAGES =
      MX ? 4
         : D == 192 ? (N <= 64 ? 7 : (N <= 128 ? 6 : (N == 192 ? 5 : 4)))
                    : (N <= 128 ? 10 : (N == 192 ? 9 : 8));
  static constexpr uint32_t RAW_BYTES = MX ? kTileTokens * (D / 2 + D / 32) : 0;
  static constexpr int RAW_STAGES = MX ? (N <= 192 ? 8 : 6) : 0;
  static constexpr int ACC = N <= 128 ? 4 : 2;  // even: tile k's accumulator belongs to team k&1
  static constexpr int TMEM_COLS = (ACC * NP <= 256) ? 256 : 512;
  static constexpr uint32_t Q_BYTES = NP * D;
  static constexpr uint32_t W_FLOATS = NN * H;
  static constexpr uint32_t OFF_KV = 0;
  static constexpr uint32_t OFF_Q = OFF_KV + STAGES * STAGE_BYTES;
  static constexpr uint32_t OFF_W = OFF_Q + 2 * Q_BYTES;
  // Tile k's scales live in slot k % SCALE_SLOTS.  The producer refills a slot only after tile
  // k + ACC's MMAs started, which needs tile k's epilogue to have released its accumulator, and
  // the epilogue reads its scale before that release.
  static constexpr int SCALE_SLOTS = STAGES + ACC;
  static constexpr uint32_t OFF_RAW = OFF_W + 2 * W_FLOATS * 4;
  static constexpr uint32_t OFF_SCALE = OFF_RAW + RAW_STAGES * RAW_BYTES;
  static constexpr uint32_t OFF_LIST = OFF_SCALE + SCALE_SLOTS * kTileTokens * 4;
  static constexpr uint32_t OFF_PG2 = OFF_LIST + kMaxList * 16;  // pages 2, 3 (32-token pages)
  static constexpr uint32_t OFF_BAR = OFF_PG2 + kMaxList * 8;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 4 + 1 + 2 * RAW_STAGES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // TMEM address, list length, table
  static constexpr uint32_t OFF_LEN = OFF_MISC + 64 + 80;
  static constexpr uint32_t smem_bytes(int batch) {
    return OFF_LEN + 4u * static_cast<uint32_t>(batch) + 1024u;  // + alignment slack
  }
  static_assert(OFF_Q % 1024 == 0 && Q_BYTES % 1024 == 0, "swizzled tiles 1024-aligned");
  static_assert(OFF_W % 16 == 0 && OFF_LIST % 16 == 0 && OFF_SCALE % 16 == 0 &&
                    OFF_RAW % 16 == 0 && RAW_BYTES % 16 == 0,
                "copy destinations 16-byte aligned");
  static_assert(!MX || D == 128, "MXFP4 tiles: head_dim 128");
  static_assert(!MX || (STAGES % CONV_GROUPS == 0 && RAW_STAGES % CONV_GROUPS == 0),
                "(MX) a converter group's tiles keep to its own stages");
  static_assert(smem_bytes(kMaxBatch) <= 232448, "fits the 227 KiB per-CTA limit");
  static_assert(ACC * NP <= TMEM_COLS && ACC % 2 == 0 && ACC <= STAGES, "accumulators");
  static_assert(H == 8 || H == 16 || H == 32 || H == 64, "8, 16, 32 or 64 heads");
};

__device__ __forceinline__ void flag_error(int bits) { atomicOr(&g_logits_status, bits); }

// The output element: float32, or float16 rounded to nearest even (the pages' output_dtype).
__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__half *p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// The fused score + select output ("flashinfer.sdsa.indexer_threshold_select": description):
// instead of being stored, each score is classified against its row's threshold into the row's
// candidate and tie slots.
struct SelectOut {};

// A warp's candidate-slot reservation for one draft slot, whose atomicAdd result is used only at
// the warp's next tile (or request change), so that the atomic's round trip to L2 overlaps that
// tile's work instead of stalling the epilogue.  mask: lanes holding a candidate (warp-uniform;
// 0 = nothing pending); base: the reserved position (leader lane only).
struct PendingCands {
  unsigned mask;
  int base;
  int row;
  int index;
  float score;
};

__device__ __forceinline__ void finish_cands(PendingCands &pc, int2 *candidates, int top_k,
                                             int capacity, int lane) {
  if (pc.mask == 0u) return;
  const int base = __shfl_sync(0xffffffffu, pc.base, __ffs(pc.mask) - 1);
  if ((pc.mask >> lane) & 1u) {
    const int n = base + __popc(pc.mask & lanemask_lt());
    if (n < capacity)
      candidates[static_cast<int64_t>(pc.row) * (top_k + capacity) + top_k + n] =
          make_int2(pc.index, __float_as_int(pc.score));
  }
  pc.mask = 0u;
}

// relu(s) * 2^-26 on the FMA pipe: a saturating multiply clamps to [0, 1] (NaN to 0), and
// every score satisfies |s| <= 192 * 448^2 < 2^26, so the product is exact (and a nonzero score,
// a multiple of 2^-18, stays a normal float).
__device__ __forceinline__ float relu_scaled(float s) {
  float r;
  asm("mul.rn.sat.f32 %0, %1, 0f32800000;" : "=f"(r) : "f"(s));  // 0f32800000 = 2^-26
  return r;
}

// Partial logits of the two positions one 16x256b load of R 8-column chunks covers (lanes g and
// g + 8 of its window): sums over this thread's 2R heads {8r + 2c, 8r + 2c + 1 : r < R} (of
// H = 8R) of w_h * max(s_h, 0) in float32, the head pair of each r in one packed FMA.  Even r
// take the ReLU as max(s, 0) on the ALU pipe, odd r as relu_scaled on the FMA pipe, which
// balances the two pipes; the latter's sums are 2^-26 times what max(s, 0) would have produced
// (a power-of-two scaling commutes with every rounding), so the final 2^26 rescale makes the
// result identical to an all-max(s, 0) evaluation of the same summation order.
template <int R>
__device__ __forceinline__ float2 quad_partials(const uint32_t (&v)[4 * R],
                                                const float2 (&w)[R]) {
  float2 u0 = make_float2(0.0f, 0.0f), u1 = u0, s0 = u0, s1 = u0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float a0 = __uint_as_float(v[4 * r]), a1 = __uint_as_float(v[4 * r + 1]);
    const float b0 = __uint_as_float(v[4 * r + 2]), b1 = __uint_as_float(v[4 * r + 3]);
    if (r & 1) {
      s0 = __ffma2_rn(w[r], make_float2(relu_scaled(a0), relu_scaled(a1)), s0);
      s1 = __ffma2_rn(w[r], make_float2(relu_scaled(b0), relu_scaled(b1)), s1);
    } else {
      u0 = __ffma2_rn(w[r], make_float2(fmaxf(a0, 0.0f), fmaxf(a1, 0.0f)), u0);
      u1 = __ffma2_rn(w[r], make_float2(fmaxf(b0, 0.0f), fmaxf(b1, 0.0f)), u1);
    }
  }
  constexpr float kUnscale = 67108864.0f;  // 2^26
  return make_float2((u0.x + u0.y) + (s0.x + s0.y) * kUnscale,
                     (u1.x + u1.y) + (s1.x + s1.y) * kUnscale);
}

// The four threads of a quad (same g, c = 0..3) hold partial sums of positions g, g + 8, g + 16,
// g + 24 over disjoint head sets.  Two exchange steps leave thread c with the complete sum of
// position g + 8c.
__device__ __forceinline__ float quad_reduce_scatter(float p0, float p1, float p2, float p3, int c) {
  const bool upper = (c & 2) != 0;  // keeps positions 2, 3
  float keep0 = upper ? p2 : p0, keep1 = upper ? p3 : p1;
  const float give0 = upper ? p0 : p2, give1 = upper ? p1 : p3;
  keep0 += __shfl_xor_sync(0xffffffffu, give0, 2);
  keep1 += __shfl_xor_sync(0xffffffffu, give1, 2);
  const bool odd = (c & 1) != 0;  // keeps the second of the two
  const float mine = odd ? keep1 : keep0, give = odd ? keep0 : keep1;
  return mine + __shfl_xor_sync(0xffffffffu, give, 1);
}

// Finds, in one warp, the (request, tile) of the flat tile indices f0 and f1 (< f0 + 2^31) given
// each lane's segment [seg_lo, seg_hi) of requests, the lane's exclusive tile prefix and its tile
// count: the lanes holding them walk their segment once.  An index >= total gives (batch, 0).
__device__ __forceinline__ void warp_locate2(long long f0, long long f1, long long total,
                                             int seg_lo, int seg_hi, long long excl,
                                             long long mine, const int *s_len, int batch,
                                             int2 &at0, int2 &at1) {
  at0 = make_int2(batch, 0);
  at1 = make_int2(batch, 0);
  const bool here0 = f0 < total && f0 >= excl && f0 < excl + mine;
  const bool here1 = f1 < total && f1 >= excl && f1 < excl + mine;
  if (here0 || here1) {
    long long run = excl;
    for (int b = seg_lo; b < seg_hi; ++b) {
      const int t = tiles_of(s_len[b]);
      if (here0 && f0 >= run && f0 < run + t) at0 = make_int2(b, static_cast<int>(f0 - run));
      if (here1 && f1 >= run && f1 < run + t) at1 = make_int2(b, static_cast<int>(f1 - run));
      run += t;
    }
  }
  const unsigned who0 = __ballot_sync(0xffffffffu, here0);
  const unsigned who1 = __ballot_sync(0xffffffffu, here1);
  const int src0 = who0 ? __ffs(who0) - 1 : 0, src1 = who1 ? __ffs(who1) - 1 : 0;
  const int2 r0 = make_int2(__shfl_sync(0xffffffffu, at0.x, src0),
                            __shfl_sync(0xffffffffu, at0.y, src0));
  const int2 r1 = make_int2(__shfl_sync(0xffffffffu, at1.x, src1),
                            __shfl_sync(0xffffffffu, at1.y, src1));
  if (who0) at0 = r0;
  if (who1) at1 = r1;
}

// Where one warp is in the CTA's tile run while it writes tile lists.
struct ListCursor {
  int b, j;      // next tile to list
  int b_end, j_end;
  int prev_b;    // request of the last tile of the previous list (-1 before the first)
  int ord;       // ordinal of that request in the run (requests with tiles count 1, 2, ...)
};

// The list builder's state after a list: where the next list starts, and this list's length.
struct ListResult {
  ListCursor cur;
  int n;
};

// Writes the next list (at most kMaxList tiles) into s_list (and s_pg2); called by all 32 lanes of
// one warp.  A tile of 128 positions spans 1 << PPT_SHIFT pages.  Record: x = request |
// kFirstFlag | kLastFlag | (mask of the tile's present pages) << kMaskShift, y = tile, z / w =
// page id of the tile's page 0 / 1, s_pg2 = pages 2 / 3 (-1: absent, or outside the pool).
// x also carries the request's ordinal in the CTA's run (mod 256) << kOrdShift.
//
// Requests are taken 32 at a time, lane l covering request b + l.  After a scan of their tile
// counts every record is produced by one lane, 32 * PER records per round (PER per lane), which
// finds the record's request by a binary search over the scanned counts.  A round first places
// all its records, then issues all their block-table reads, then writes: a list of up to
// 32 * PER tiles costs one memory round trip.  (PER = 1 where the kernel's register budget is
// tight.)  Everything is passed by value, so that nothing of the caller's lives in local memory.
template <int PER, int PPT_SHIFT>
__device__ __noinline__ ListResult build_list(ListCursor cur, int batch, const int *s_len,
                                              int4 *s_list, int2 *s_pg2,
                                              const int32_t *block_tables, int64_t bt_stride,
                                              int64_t num_blocks, int lane) {
  constexpr int PPT = 1 << PPT_SHIFT;  // pages per tile: 1, 2 or 4
  constexpr int BS_SHIFT = 7 - PPT_SHIFT;
  int n = 0;
  int b = cur.b, j = cur.j;
  while (n < kMaxList && b < batch && (b < cur.b_end || (b == cur.b_end && j < cur.j_end))) {
    const int rb = b + lane;
    int jlo = 0, jhi = 0;
    if (rb < batch && rb <= cur.b_end) {
      jlo = lane == 0 ? j : 0;
      const int live = tiles_of(s_len[rb]);
      // A stale caller schedule may name tiles past the live length: never list those.
      jhi = rb == cur.b_end ? min(cur.j_end, live) : live;
      jhi = max(jhi, jlo);
    }
    const int cnt = jhi - jlo;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - cnt;
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int room = kMaxList - n;
    const int take = min(total, room);
    // Request ordinals: the requests with tiles are numbered along the run; lane 0's request
    // keeps its number when it continues the previous list's last request.
    const unsigned act = __ballot_sync(0xffffffffu, cnt > 0);
    const bool cont = n == 0 && cur.prev_b == b;
    const unsigned le = lane == 31 ? 0xffffffffu : (2u << lane) - 1u;
    const int my_ord = cur.ord + __popc(act & le) - (cont ? 1 : 0);
    for (int c0 = 0; c0 < take; c0 += 32 * PER) {
      int rx[PER], rj[PER], npg[PER], id[PER][PPT];
      const int32_t *row[PER];
#pragma unroll
      for (int h = 0; h < PER; ++h) {
        const int idx = c0 + 32 * h + lane;
        // The lane (request) owning record idx: the last lane whose exclusive count <= idx.
        int src = 0;
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1)
          if (__shfl_sync(0xffffffffu, excl, src + step) <= idx) src += step;
        const int e_s = __shfl_sync(0xffffffffu, excl, src);
        const int c_s = __shfl_sync(0xffffffffu, cnt, src);
        const int j_s = __shfl_sync(0xffffffffu, jlo, src);
        const int o_s = __shfl_sync(0xffffffffu, my_ord, src) & 255;
        rx[h] = -1;
        rj[h] = 0;
        npg[h] = 0;
        row[h] = block_tables;
        if (idx < take) {
          const int req = b + src;
          const int tile = j_s + (idx - e_s);
          const bool first = n + idx == 0 ? cur.prev_b != req : idx == e_s;
          const bool last = idx == e_s + c_s - 1;
          rx[h] = req | (first ? kFirstFlag : 0) | (last ? kLastFlag : 0) | (o_s << kOrdShift);
          rj[h] = tile;
          const int len = s_len[req];
          const int npages = (len + (1 << BS_SHIFT) - 1) >> BS_SHIFT;
          const int first_page = tile << PPT_SHIFT;
          row[h] = block_tables + static_cast<int64_t>(req) * bt_stride + first_page;
          npg[h] = min(npages - first_page, PPT);  // the tile's pages, >= 1
        }
      }
#pragma unroll
      for (int h = 0; h < PER; ++h)
#pragma unroll
        for (int pg = 0; pg < PPT; ++pg) id[h][pg] = pg < npg[h] ? __ldg(row[h] + pg) : -1;
#pragma unroll
      for (int h = 0; h < PER; ++h) {
        if (rx[h] >= 0) {
          int mask = 0;
          bool bad = false;
#pragma unroll
          for (int pg = 0; pg < PPT; ++pg) {
            if (pg >= npg[h]) continue;
            if (id[h][pg] < 0 || id[h][pg] >= num_blocks) {
              bad = true;
              id[h][pg] = -1;
            } else {
              mask |= 1 << pg;
            }
          }
          if (bad) flag_error(IDX_DEV_BAD_PAGE);
          const int k = n + c0 + 32 * h + lane;
          s_list[k] = make_int4(rx[h] | (mask << kMaskShift), rj[h], id[h][0],
                                PPT >= 2 ? id[h][PPT >= 2 ? 1 : 0] : -1);
          if constexpr (PPT == 4) s_pg2[k] = make_int2(id[h][2], id[h][3]);
        }
      }
    }
    if (total <= room) {
      n += total;
      b += 32;
      j = 0;
      cur.ord += __popc(act) - (cont ? 1 : 0);
    } else {
      // The list ends inside request L, which continues in the next list, or just before L's
      // first tile here: then L is not in this list, and the ordinal carried over is that of
      // the list's last request, so that L numbers itself in the next list.
      const int L = __ffs(__ballot_sync(0xffffffffu, incl > room)) - 1;
      const int l_excl = __shfl_sync(0xffffffffu, excl, L);
      const int l_jlo = __shfl_sync(0xffffffffu, jlo, L);
      const int l_ord = __shfl_sync(0xffffffffu, my_ord, L);
      cur.ord = room == l_excl ? l_ord - 1 : l_ord;
      b += L;
      j = l_jlo + (room - l_excl);
      n = kMaxList;
    }
  }
  __syncwarp();
  if (n > 0) cur.prev_b = s_list[n - 1].x & 0xFFFF;
  cur.b = b;
  cur.j = j;
  return ListResult{cur, n};
}

template <int NN, int H, int D, typename OutT, int BS_SHIFT, bool MX = false>
__global__ void __launch_bounds__(Cfg<NN, H, D, MX>::THREADS, 1)
    k_logits_fp8(const __grid_constant__ CUtensorMap kv_map,
                 const __grid_constant__ CUtensorMap q_map, const LogitsArgs a) {
  using C = Cfg<NN, H, D, MX>;
  constexpr bool kSelect = std::is_same<OutT, SelectOut>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  uint8_t *s_kv = smem + C::OFF_KV;
  uint8_t *s_q = smem + C::OFF_Q;
  float *s_w = reinterpret_cast<float *>(smem + C::OFF_W);
  float *s_scale = reinterpret_cast<float *>(smem + C::OFF_SCALE);
  int4 *s_list = reinterpret_cast<int4 *>(smem + C::OFF_LIST);
  int2 *s_pg2 = reinterpret_cast<int2 *>(smem + C::OFF_PG2);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *done = full + C::STAGES;
  uint64_t *q_full = done + C::STAGES;
  uint64_t *q_empty = q_full + 2;
  uint64_t *drain = q_empty + 2;
  uint64_t *raw_full = drain + 1;                // (MX) a raw tile landed
  uint64_t *raw_empty = raw_full + C::RAW_STAGES;  // (MX) a raw tile was converted
  uint8_t *s_raw = smem + C::OFF_RAW;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  int *s_count = reinterpret_cast<int *>(smem + C::OFF_MISC + 16);  // current list length
  uint2 *s_tab = reinterpret_cast<uint2 *>(smem + C::OFF_MISC + 64);  // (MX) 9 e4m3 tables
  int *s_len = reinterpret_cast<int *>(smem + C::OFF_LEN);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // The previous kernel in the stream may still be running: nothing is read before griddep_wait.
  // L2 prefetches read nothing (L2 is where that kernel's writes land, so later loads still see
  // them): seq_lens and this CTA's share of the block table start their way from DRAM while the
  // previous kernel drains.  Block-table lines hold at least one byte of a row's declared width.
  // (A rescoring launch reads few rows of the table, if any: it prefetches none.)
  if (warp == 0) {
    if (a.sl_stride == 1) {
      for (int l = lane; l * 32 < a.batch; l += 32) prefetch_l2(a.seq_lens + l * 32);
    } else {
      for (int b = lane; b < a.batch; b += 32) prefetch_l2(a.seq_lens + b * a.sl_stride);
    }
  } else if (warp == kEpiWarpBase && a.bt_width > 0 && a.fit_counters == nullptr &&
             static_cast<int64_t>(a.batch) * a.bt_width <= (int64_t{1} << 21)) {
    for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
      const int32_t *row = a.block_tables + static_cast<int64_t>(b) * a.bt_stride;
      const uintptr_t first = reinterpret_cast<uintptr_t>(row) & ~uintptr_t{127};
      const uintptr_t last = reinterpret_cast<uintptr_t>(row + a.bt_width - 1) & ~uintptr_t{127};
      for (uintptr_t line = first + 128u * lane; line <= last; line += 128u * 32u)
        prefetch_l2(reinterpret_cast<const void *>(line));
    }
  }
  griddep_wait();
  griddep_launch_dependents();

  const int batch = a.batch;
  // Pages of 1 << BS_SHIFT = 32, 64 or 128 tokens: that many 128-byte value rows, then that
  // many float32 scales.
  constexpr int bs_shift = BS_SHIFT;
  ListCursor cursor{};

  // ---- 1. set-up: warp 0 finds the CTA's tile run, warp 1 prepares barriers and TMEM --------
  if (warp == 0) {
    const int per = (batch + 31) / 32;
    const int lo = min(lane * per, batch);
    const int hi = min(lo + per, batch);
    long long mine = 0;
    for (int b = lo; b < hi; ++b) {
      int len = __ldg(a.seq_lens + static_cast<int64_t>(b) * a.sl_stride);
      len = len < 0 ? 0 : len;
      if (a.fit_counters != nullptr) {
        // Rescoring: a request whose rows all fit counts as empty.
        bool fits = true;
#pragma unroll
        for (int t = 0; t < NN; ++t) {
          const int2 c = *reinterpret_cast<const int2 *>(a.fit_counters + 2 * (b * NN + t));
          fits = fits && row_fits(c.x, c.y, min(max(0, len - NN + t + 1), a.top_k), a.top_k,
                                  a.capacity);
        }
        if (fits) len = 0;
      }
      s_len[b] = len;
      mine += tiles_of(len);
    }
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const long long total = __shfl_sync(0xffffffffu, incl, 31);
    const long long excl = incl - mine;
    int2 s0, s1;
    if (a.schedule != nullptr) {
      s0 = make_int2(__ldg(a.schedule + 2 * blockIdx.x), __ldg(a.schedule + 2 * blockIdx.x + 1));
      s1 = make_int2(__ldg(a.schedule + 2 * blockIdx.x + 2),
                     __ldg(a.schedule + 2 * blockIdx.x + 3));
    } else {
      // The CTA's share [total * c / g, total * (c + 1) / g), in 32-bit arithmetic whenever the
      // products fit (64-bit division is a long software sequence).
      const unsigned g = gridDim.x, cb = blockIdx.x;
      long long f0, f1;
      if (total <= static_cast<long long>(0xFFFFFFFFu / g)) {
        const unsigned t32 = static_cast<unsigned>(total);
        f0 = (t32 * cb) / g;
        f1 = (t32 * (cb + 1)) / g;
      } else {
        f0 = total * cb / g;
        f1 = total * (cb + 1) / g;
      }
      warp_locate2(f0, f1, total, lo, hi, excl, mine, s_len, batch, s0, s1);
    }
    __syncwarp();
    // Start at the first tile that exists (a stale schedule or empty requests may point past it).
    const TileIter it = make_iter(s0.x, s0.y, s1.x, s1.y, batch, s_len);
    cursor = ListCursor{it.b, it.j, it.b_end, it.j_end, -1, 0};
    if (lane == 0) *s_count = it.valid() ? 1 : 0;  // (rescoring) whether the run has a tile
    if (a.row_ends != nullptr) {
      for (int b = blockIdx.x + lane * gridDim.x; b < batch; b += 32 * gridDim.x) {
        const int len = s_len[b];
#pragma unroll
        for (int t = 0; t < NN; ++t) a.row_ends[b * NN + t] = max(0, len - NN + t + 1);
      }
    }
  }
  // Warp 1: barriers and TMEM.  A rescoring launch first learns whether this CTA has any tile to
  // rescore (usually none): an empty CTA leaves here, having set up nothing.
  if (a.fit_counters != nullptr) {
    __syncthreads();
    if (*s_count == 0) return;
  }
  if (warp == 1) {
    if (lane == 0) {
      prefetch_tensor_map(&kv_map);
      prefetch_tensor_map(&q_map);
      for (int s = 0; s < C::STAGES; ++s) {
        // The producer (MX: the converter warps) + the accumulator's last readers.
        mbar_init(&full[s], (C::MX ? C::GROUP_WARPS : 1) + C::TEAM_WARPS);
        mbar_init(&done[s], 1);  // the MMA's commit
      }
      for (int s = 0; s < C::RAW_STAGES; ++s) {
        mbar_init(&raw_full[s], 1);
        mbar_init(&raw_empty[s], C::GROUP_WARPS);
      }
      for (int c = 0; c < 2; ++c) {
        mbar_init(&q_full[c], 1);
        mbar_init(&q_empty[c], 1 + C::EPI_WARPS);  // MMA commit + every epilogue warp
      }
      mbar_init(drain, 1);
      fence_barrier_init();
    }
    __syncwarp();
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }

  if constexpr (C::MX) {
    const int ct = tid - C::CONV_BASE * 32;
    if (ct >= 0 && ct < 9) s_tab[ct] = e2m1_table_entry(ct);  // read after the next barrier
  }

  // Per-role pipeline state, kept across lists.  (MX) The producer's stage / phase follow the
  // raw ring; the converters' follow the KV stages, their rstage / rphase the raw ring.
  int stage = 0;
  uint32_t phase = 0;
  int rstage = 0;
  uint32_t rphase = 0;
  int qcount = 0, qb = 0;
  int kbase = 0;  // CTA-wide index of the current list's first tile
  bool ok = true;
  bool drained = false;  // (MMA issuer) the drain commit is out
  uint32_t tmem_base = 0;
  // (epilogue) The request whose weights are in registers, by its ordinal in the run (mod 256;
  // 0: none yet), the ordinal up to which this warp has arrived on q_empty, and the weights of
  // this thread's heads {8r + 2c, 8r + 2c + 1} per draft slot.
  int wseq = 0;
  int released = 0;
  float2 wreg[C::SLOTS][C::R];
  // (epilogue, fused select) The thresholds of the current request's rows, per draft slot.
  float thr_u[C::SLOTS];
  // (fused select, one warp per lane quadrant) Each draft slot's candidate reservation of the
  // warp's previous tile.
  constexpr bool kDefer = kSelect && C::SPLIT == 1;
  PendingCands pend[C::SLOTS];
#pragma unroll
  for (int u = 0; u < C::SLOTS; ++u) pend[u].mask = 0u;
  const auto finish_all = [&]() {
#pragma unroll
    for (int u = 0; u < C::SLOTS; ++u)
      finish_cands(pend[u], reinterpret_cast<int2 *>(a.candidates), a.top_k, a.capacity, lane);
  };

  for (;;) {
    if (warp == 0) {
      constexpr int PER = NN <= 2 ? 2 : 1;
      const ListResult lr = build_list<PER, 7 - BS_SHIFT>(cursor, batch, s_len, s_list, s_pg2,
                                                           a.block_tables, a.bt_stride,
                                                           a.num_blocks, lane);
      cursor = lr.cur;
      if (lane == 0) *s_count = lr.n;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    tmem_base = *s_tmem;
    const int n = *s_count;
    if (n == 0) break;

    if (warp == 0) {
      // ============================== producer ================================================
      // This thread's per-tile work sits on the pipeline's critical path, so its loop is
      // specialised on the page size (one to four pages per tile) and keeps to constants.
      if (lane == 0 && ok) {
        const uint64_t pol_stream = l2_policy_evict_first();
        const uint64_t pol_keep = l2_policy_evict_last();
        // (testing only) The first tile whose copies are never issued, or -1.
        const int withhold = g_withhold_cta == static_cast<int>(blockIdx.x) ? 0 : -1;
        const auto produce = [&](auto page_tokens) {
          constexpr int BS = decltype(page_tokens)::value;
          constexpr uint32_t kValue = BS * D, kScale = BS * 4;
          constexpr int64_t kPage = BS * (D + 4);
          // Rows of D bytes per page (head_dim 64, 128; the pool viewed as such rows).
          constexpr int kRows = C::KB == 1 ? static_cast<int>(kPage / D) : 0;
          static_assert(C::KB != 1 || kPage % D == 0, "a page is a whole number of D-byte rows");
          const auto page = [&](int pg, int id, uint8_t *dst, float *sdst) {
            if (id < 0) return;
            if constexpr (C::KB == 1) {
              tma_load_2d(dst + pg * kValue, &kv_map, &full[stage], 0, id * kRows, pol_stream);
            } else {
              // The pool as [page][token][K block][64 bytes]: block j of the page's tokens
              // lands in K block j of the tile, at the page's rows.
#pragma unroll
              for (int j = 0; j < C::KB; ++j)
                tma_load_4d(dst + j * C::KBLOCK + pg * BS * (D / C::KB), &kv_map, &full[stage],
                            0, j, 0, id, pol_stream);
            }
            bulk_load(sdst + pg * BS, a.kv + static_cast<int64_t>(id) * kPage + kValue, kScale,
                      &full[stage], pol_stream);
          };
          // (MX) A page is BS packed rows of D/2 bytes, then BS * D/32 scale bytes: one bulk
          // copy into the raw tile, at page p's place.
          constexpr uint32_t kRawPage = BS * (D / 2 + D / 32);
          for (int i = 0; i < n; ++i) {
            const int4 r = s_list[i];
            const int2 hi = BS == 32 ? s_pg2[i] : make_int2(-1, -1);
            const uint32_t pages = (r.z >= 0 ? 1u : 0u) + (r.w >= 0 ? 1u : 0u) +
                                   (hi.x >= 0 ? 1u : 0u) + (hi.y >= 0 ? 1u : 0u);
            if constexpr (C::MX) {
              if (!mbar_wait(&raw_empty[stage], phase ^ 1, kWaitLimitNs)) {
                ok = false;
                break;
              }
              if (kbase + i != withhold) {
                mbar_arrive_expect_tx(&raw_full[stage], kRawPage * pages);
                uint8_t *dst = s_raw + stage * C::RAW_BYTES;
                const int ids[4] = {r.z, r.w, hi.x, hi.y};
#pragma unroll
                for (int pg = 0; pg < (kTileTokens / BS); ++pg)
                  if (ids[pg] >= 0)
                    bulk_load(dst + pg * kRawPage, a.kv + static_cast<int64_t>(ids[pg]) * kRawPage,
                              kRawPage, &raw_full[stage], pol_stream);
              }
              if (++stage == C::RAW_STAGES) {
                stage = 0;
                phase ^= 1;
              }
            } else {
              if (!mbar_wait(&done[stage], phase ^ 1, kWaitLimitNs)) {
                ok = false;
                break;
              }
              if (kbase + i != withhold) {
                mbar_arrive_expect_tx(&full[stage], (kValue + kScale) * pages);
                // The first ACC tiles' accumulators were never read: stand in for their readers.
                if (kbase + i < C::ACC) mbar_arrive_count(&full[stage], C::TEAM_WARPS);
                uint8_t *dst = s_kv + stage * C::STAGE_BYTES;
                float *sdst = s_scale + ((kbase + i) % C::SCALE_SLOTS) * kTileTokens;
                page(0, r.z, dst, sdst);
                if (BS <= 64) page(1, r.w, dst, sdst);
                if (BS == 32) {
                  page(2, hi.x, dst, sdst);
                  page(3, hi.y, dst, sdst);
                }
              }
              if (++stage == C::STAGES) {  // (before the q wait, so a timeout there still drains)
                stage = 0;
                phase ^= 1;
              }
            }
            // A new request's q and w go out after its first KV tile, whose latency is longer.
            if (r.x & kFirstFlag) {
              const int b = r.x & 0xFFFF;
              const int buf = qcount & 1;
              if (!mbar_wait(&q_empty[buf], ((qcount >> 1) & 1) ^ 1, kWaitLimitNs)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&q_full[buf], C::Q_BYTES + C::W_FLOATS * 4);
              if constexpr (C::KB == 1) {
                tma_load_2d(s_q + buf * C::Q_BYTES, &q_map, &q_full[buf], 0, b * C::N, pol_keep);
              } else {
#pragma unroll
                for (int j = 0; j < C::KB; ++j)
                  tma_load_3d(s_q + buf * C::Q_BYTES + j * C::NP * (D / C::KB), &q_map,
                              &q_full[buf], 0, j, b * C::N, pol_keep);
              }
              bulk_load(s_w + buf * C::W_FLOATS,
                        a.weights + static_cast<int64_t>(b) * C::W_FLOATS, C::W_FLOATS * 4,
                        &q_full[buf], pol_keep);
              ++qcount;
            }
          }
        };
        produce(std::integral_constant<int, 1 << BS_SHIFT>{});
      }
      __syncwarp();
    } else if (warp == 1) {
      // ============================== MMA issuer ==============================================
      // This thread is the pipeline's serial point: the tensor core idles whenever it falls
      // behind, and it shares its scheduler with busy epilogue warps (each instruction of its
      // serial chain waits for an issue slot), so its loop is kept to a few instructions per
      // tile: the next record's flags are loaded a tile ahead, and the shared-memory descriptors
      // are kept as (start-address word, constant word) pairs of which only the start address is
      // advanced (addresses stay below 256 KiB, so the 14-bit field never carries).
      if (lane == 0 && ok) {
        constexpr uint32_t idesc = idesc_e4m3_f32(kTileTokens, C::NP);
        constexpr int kSteps = D / C::KB / 32;  // K steps of 32 bytes per K block
        constexpr uint32_t kStageStep = C::STAGE_BYTES >> 4, kQStep = C::Q_BYTES >> 4;
        const uint64_t a0 = smem_desc_rows<D / C::KB>(smem_addr(s_kv));
        const uint64_t b0 = smem_desc_rows<D / C::KB>(smem_addr(s_q));
        const uint32_t a_hi = static_cast<uint32_t>(a0 >> 32), b_hi = static_cast<uint32_t>(b0 >> 32);
        const uint32_t a_lo0 = static_cast<uint32_t>(a0), b_lo0 = static_cast<uint32_t>(b0);
        int acc = kbase % C::ACC;
        uint32_t a_lo = a_lo0 + static_cast<uint32_t>(stage) * kStageStep;
        uint32_t b_lo = b_lo0 + static_cast<uint32_t>(qb) * kQStep;
        uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::NP);
        int rx = s_list[0].x;
        for (int i = 0; i < n; ++i) {
          const int rx_next = i + 1 < n ? s_list[i + 1].x : 0;
          if (rx & kFirstFlag) {
            qb = qcount & 1;
            b_lo = b_lo0 + static_cast<uint32_t>(qb) * kQStep;
            if (!mbar_wait(&q_full[qb], (qcount >> 1) & 1, kWaitLimitNs)) {
              ok = false;
              break;
            }
            ++qcount;
          }
          if (!mbar_wait(&full[stage], phase, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int j = 0; j < C::KB; ++j)
#pragma unroll
            for (int kk = 0; kk < kSteps; ++kk)  // K step of 32 bytes = 2 in the address field
              mma_f8f6f4(d_tmem, a_lo + static_cast<uint32_t>(j * (C::KBLOCK >> 4) + 2 * kk), a_hi,
                         b_lo + static_cast<uint32_t>(j * (C::NP * (D / C::KB) >> 4) + 2 * kk),
                         b_hi, idesc, j + kk > 0 ? 1u : 0u);
          mma_commit(&done[stage]);
          if (rx & kLastFlag) mma_commit(&q_empty[qb]);
          rx = rx_next;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
            a_lo = a_lo0;
          } else {
            a_lo += kStageStep;
          }
          if (++acc == C::ACC) acc = 0;
          d_tmem = tmem_base + static_cast<uint32_t>(acc * C::NP);
        }
        // A short list is the run's last: commit the drain behind its MMAs now, so that it has
        // completed by the teardown.
        if (ok && n < kMaxList) {
          mma_commit(drain);
          drained = true;
        }
      }
      __syncwarp();
    } else if (C::MX && warp >= C::CONV_BASE) {
      // ============================== converters (MX) =========================================
      // Unit u of a tile = token ct = u / 2, half hf = u % 2: the token's groups 2hf and 2hf + 1
      // (64 elements) are converted from the raw packed row into the e4m3 row of the KV stage
      // (128 bytes, stored with the 128-byte swizzle the TMA would have applied: 16-byte chunk c
      // of row ct at chunk c ^ (ct % 8)), relative to the token's largest scale byte E (all four
      // bytes are read); half 0 writes the token's float32 scale 2^(E - 127) into the tile's
      // scale slot.  Rows of absent pages become zeros.  Then the raw tile is released and the
      // stage marked full for the MMA (after a proxy fence: the tensor core reads shared memory
      // through the async proxy).  The two groups of a unit are read in an order rotated by
      // token (ct / 2), which spreads a quarter warp's reads over distinct banks.
      if (ok) {
        constexpr int BS = 1 << BS_SHIFT;
        constexpr uint32_t kRawPage = BS * (D / 2 + D / 32);
        constexpr int kGroupThreads = C::GROUP_WARPS * 32;
        const int grp = (warp - C::CONV_BASE) / C::GROUP_WARPS;
        const int gtid = tid - (C::CONV_BASE + grp * C::GROUP_WARPS) * 32;
        for (int i = (grp - kbase % C::CONV_GROUPS + C::CONV_GROUPS) % C::CONV_GROUPS; i < n;
             i += C::CONV_GROUPS) {
          const int k = kbase + i;
          const int stage = k % C::STAGES, rstage = k % C::RAW_STAGES;
          const uint32_t phase = (k / C::STAGES) & 1, rphase = (k / C::RAW_STAGES) & 1;
          const int4 r = s_list[i];
          if (!mbar_wait(&raw_full[rstage], rphase, kWaitLimitNs) ||
              !mbar_wait(&done[stage], phase ^ 1, kWaitLimitNs)) {
            ok = false;
            break;
          }
          bool inexact = false;
          const int live = s_len[r.x & 0xFFFF] - r.y * kTileTokens;  // tokens below seq_len
          for (int u = gtid; u < 2 * kTileTokens; u += kGroupThreads) {
            const int ct = u >> 1, hf = u & 1;
            const int pg = ct >> BS_SHIFT, tt = ct & (BS - 1);
            uint8_t *row = s_kv + stage * C::STAGE_BYTES + ct * 128;
            const bool have = (static_cast<uint32_t>(r.x) >> (kMaskShift + pg)) & 1u;
            if (have) {
              const uint8_t *raw = s_raw + rstage * C::RAW_BYTES + pg * kRawPage;
              const uint32_t sf = *reinterpret_cast<const uint32_t *>(raw + BS * (D / 2) + tt * 4);
              int emax = 0;
#pragma unroll
              for (int g = 0; g < 4; ++g) emax = max(emax, static_cast<int>((sf >> (8 * g)) & 0xFFu));
              // A 0xFF (NaN) scale byte: a zero byte of ~sf.
              const uint32_t nsf = ~sf;
              if (((nsf - 0x01010101u) & ~nsf & 0x80808080u) != 0u && ct < live) inexact = true;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int g = 2 * hf + ((j + (ct >> 1)) & 1);
                const int rel = static_cast<int>((sf >> (8 * g)) & 0xFFu) - emax;
                uint32_t out[8];
                bool lost = false;
                mx_group_to_e4m3(*reinterpret_cast<const uint4 *>(raw + tt * (D / 2) + 16 * g), rel,
                                 s_tab[rel >= -8 ? -rel : 0], out, &lost);
                if (lost && ct < live) inexact = true;
                *reinterpret_cast<uint4 *>(row + (((2 * g) ^ (ct & 7)) << 4)) =
                    make_uint4(out[0], out[1], out[2], out[3]);
                *reinterpret_cast<uint4 *>(row + (((2 * g + 1) ^ (ct & 7)) << 4)) =
                    make_uint4(out[4], out[5], out[6], out[7]);
              }
              if (hf == 0) s_scale[(k % C::SCALE_SLOTS) * kTileTokens + ct] = pow2f(emax - 127);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4 *>(row + (((4 * hf + j) ^ (ct & 7)) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
              if (hf == 0) s_scale[(k % C::SCALE_SLOTS) * kTileTokens + ct] = 0.0f;
            }
          }
          if (inexact) flag_error(IDX_DEV_INEXACT_SCALE);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&raw_empty[rstage]);
            mbar_arrive(&full[stage]);
            // The first ACC tiles' accumulators were never read: stand in for their readers.
            if (gtid == 0 && k < C::ACC) mbar_arrive_count(&full[stage], C::TEAM_WARPS);
          }
        }
      }
    } else {
      // ============================== epilogue ================================================
      const int team = (warp - kEpiWarpBase) / C::TEAM_WARPS;  // takes tiles k % TEAMS == team
      const int t_first = ((warp - kEpiWarpBase) / 4) % C::SPLIT * C::SLOTS;  // first draft slot
      const int quarter = warp & 3;
      const int c = lane & 3;
      const int pos = quarter * 32 + (lane >> 2) + 8 * c;  // the position this thread stores
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      // A warp walks only its team's tiles.  The q/w buffers it no longer needs are released
      // lazily: on reaching a tile of a new request (by ordinal o), it first arrives on q_empty
      // for every earlier request it has not released, then waits for the new request's q/w.
      // (The producer needs request j released only to load request j + 2's q/w, and a warp
      // releases j before it waits for anything beyond j, so the two cannot wait on each other.)
      // wseq, released and wreg carry over from one tile list to the next.
      if (ok) {
        // Tile k's stage, its parity, scale slot and accumulator, advanced by TEAMS per own tile
        // (no division in the loop; with the slot split, where registers are scarcer and the
        // moduli cheaper, they are derived from k instead).
        const int i0 = (team - kbase % C::TEAMS + C::TEAMS) % C::TEAMS;
        int e_stage = (kbase + i0) % C::STAGES, e_sslot = (kbase + i0) % C::SCALE_SLOTS;
        int e_acc = (kbase + i0) % C::ACC;
        uint32_t par = ((kbase + i0) / C::STAGES) & 1;
        for (int i = i0; i < n; i += C::TEAMS) {
          const int4 r = s_list[i];
          const int b = r.x & 0xFFFF;
          if constexpr (C::SPLIT == 2) {
            const int k = kbase + i;
            e_stage = k % C::STAGES;
            e_sslot = k % C::SCALE_SLOTS;
            e_acc = k % C::ACC;
            par = (k / C::STAGES) & 1;
          }
          {
            const int o = (r.x >> kOrdShift) & 255;
            if (o != wseq) {
              __syncwarp();
              if constexpr (kSelect) {
#pragma unroll
                for (int u = 0; u < C::SLOTS; ++u)
                  thr_u[u] = t_first + u < NN ? a.thresholds[b * NN + t_first + u] : 0.0f;
              }
              for (int q = (released + 1) & 255; q != o; q = (q + 1) & 255)
                if (lane == 0) mbar_arrive(&q_empty[(q - 1) & 1]);
              released = (o - 1) & 255;
              const int qbuf = (o - 1) & 1;
              if (!mbar_wait(&q_full[qbuf], ((o - 1) >> 1) & 1, kWaitLimitNs)) {
                ok = false;
                break;
              }
              const float2 *w2 = reinterpret_cast<const float2 *>(s_w + qbuf * C::W_FLOATS);
#pragma unroll
              for (int u = 0; u < C::SLOTS; ++u)
#pragma unroll
                for (int q = 0; q < C::R; ++q)
                  wreg[u][q] = t_first + u < NN ? w2[(t_first + u) * (H / 2) + 4 * q + c]
                                                : make_float2(0.0f, 0.0f);
              wseq = o;
            }
            const int stage = e_stage;
            // done: tile k's MMAs (so its accumulator) completed.  full: makes the tile's
            // TMA-written scales visible to this thread (the phase is complete by then).
            if (!mbar_wait(&done[stage], par, kWaitLimitNs) ||
                !mbar_wait(&full[stage], par, kWaitLimitNs)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const bool have = (static_cast<uint32_t>(r.x) >> (kMaskShift + (pos >> bs_shift))) & 1u;
            const float scale = have ? s_scale[e_sslot * kTileTokens + pos] : 0.0f;
            const int p = r.y * kTileTokens + pos;
            const int len_b = s_len[b];
            const bool store = p < len_b;
            OutT *dst = nullptr;
            if constexpr (!kSelect)
              dst = static_cast<OutT *>(a.out) + static_cast<int64_t>(b * NN) * a.out_stride + p;
            // Draft slot t_first + u's score at position p: stored (p < seq_lens[b]), or
            // classified (p inside the row's extent, p < seq_lens[b] - next_n + t + 1), which
            // the whole warp does together.
            const auto emit = [&](int u, float logit) {
              const int t = t_first + u;
              if constexpr (kDefer) {
                const int row = b * NN + t;
                const bool valid = p + (NN - 1 - t) < len_b;
                const float thr = thr_u[u];
                const bool is_c = valid && logit > thr;
                finish_cands(pend[u], reinterpret_cast<int2 *>(a.candidates), a.top_k,
                             a.capacity, lane);
                const unsigned mc = __ballot_sync(0xffffffffu, is_c);
                if (mc) {
                  pend[u].mask = mc;
                  pend[u].row = row;
                  pend[u].index = p;
                  pend[u].score = logit;
                  if (lane == __ffs(mc) - 1) pend[u].base = atomicAdd(a.counters + 2 * row, __popc(mc));
                }
                // Ties (rare: equal scores or NaN) are reserved and stored at once.
                offer(false, valid && !(logit > thr) && !(logit < thr), p, logit,
                      a.counters + 2 * row,
                      reinterpret_cast<int2 *>(a.candidates) +
                          static_cast<int64_t>(row) * (a.top_k + a.capacity),
                      a.top_k, a.capacity);
              } else if constexpr (kSelect) {
                const int row = b * NN + t;
                const bool valid = p + (NN - 1 - t) < len_b;
                const float thr = thr_u[u];
                offer(valid && logit > thr, valid && !(logit > thr) && !(logit < thr), p, logit,
                      a.counters + 2 * row,
                      reinterpret_cast<int2 *>(a.candidates) +
                          static_cast<int64_t>(row) * (a.top_k + a.capacity),
                      a.top_k, a.capacity);
              } else {
                if (store) store_out(dst + static_cast<int64_t>(t) * a.out_stride, logit);
              }
            };
            const uint32_t col0 = static_cast<uint32_t>(e_acc * C::NP);
            const int nslots = min(C::SLOTS, NN - t_first);
            // The quadrant's two 16-lane windows hold positions (g, g + 8) and (g + 16, g + 24).
            // With the slot split (more warps, fewer registers each) they are read one after the
            // other, so that only 32 values are live.  Without it, the next slot's loads are
            // issued before this slot's quad reduction, so the shuffles overlap their latency
            // (with the split that ordering measured slower).
            uint32_t va[4 * C::R], vb[4 * C::R];
            float4 part[C::SLOTS];  // (slot split) each slot's partial sums, reduced at the end
#pragma unroll
            for (int u = 0; u < C::SLOTS; ++u) {
              if (u >= nslots) break;
              const int t = t_first + u;
              const uint32_t col = col0 + static_cast<uint32_t>(t * H);
              float2 p01;
              if (C::SPLIT == 2 || u == 0) {
                tmem_ld_16x256b<C::R>(lane_base + col, va);
                if constexpr (C::SPLIT == 1) tmem_ld_16x256b<C::R>(lane_base + (16u << 16) + col, vb);
              }
              if constexpr (C::SPLIT == 2) {
                tmem_ld_wait();
                reg_fence(va);
                p01 = quad_partials<C::R>(va, wreg[u]);
                asm volatile("" : "+f"(p01.x), "+f"(p01.y));  // before the next load
                tmem_ld_16x256b<C::R>(lane_base + (16u << 16) + col, vb);
              }
              tmem_ld_wait();
              if constexpr (C::SPLIT == 1) reg_fence(va);
              reg_fence(vb);
              if (u == nslots - 1) {
                // The accumulator is in registers: free it for tile k + ACC before the arithmetic.
                tc_fence_before_sync();
                __syncwarp();
                const int rel = e_stage + C::ACC;  // tile k + ACC's stage
                if (lane == 0) mbar_arrive(&full[rel >= C::STAGES ? rel - C::STAGES : rel]);
              }
              if constexpr (C::SPLIT == 1) p01 = quad_partials<C::R>(va, wreg[u]);
              float2 p23 = quad_partials<C::R>(vb, wreg[u]);
              // This slot's values are consumed before the next slot's loads reuse the registers
              // (volatile asm keeps its order).
              asm volatile("" : "+f"(p01.x), "+f"(p01.y), "+f"(p23.x), "+f"(p23.y));
              if (C::SPLIT == 1 && u + 1 < nslots) {
                tmem_ld_16x256b<C::R>(lane_base + col + H, va);
                tmem_ld_16x256b<C::R>(lane_base + (16u << 16) + col + H, vb);
              }
              if constexpr (C::SPLIT == 2) {
                // The shuffles and stores wait until every slot has been read, which frees the
                // accumulator earlier (its release gates the MMA of tile k + ACC).
                part[u] = make_float4(p01.x, p01.y, p23.x, p23.y);
              } else {
                emit(u, scale * quad_reduce_scatter(p01.x, p01.y, p23.x, p23.y, c));
              }
            }
            if constexpr (C::SPLIT == 2) {
#pragma unroll
              for (int u = 0; u < C::SLOTS; ++u) {
                if (u >= nslots) break;
                const float4 q = part[u];
                emit(u, scale * quad_reduce_scatter(q.x, q.y, q.z, q.w, c));
              }
            }
          }
          if constexpr (C::SPLIT == 1) {
            if ((e_stage += C::TEAMS) >= C::STAGES) {
              e_stage -= C::STAGES;
              par ^= 1;
            }
            if ((e_sslot += C::TEAMS) >= C::SCALE_SLOTS) e_sslot -= C::SCALE_SLOTS;
            if ((e_acc += C::TEAMS) >= C::ACC) e_acc -= C::ACC;
          }
        }
      }
    }
    kbase += n;
    if (n < kMaxList) break;  // the run ended inside this list
    // Everyone is done with this list before warp 0 overwrites it.
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
  }

  if constexpr (kSelect) {
    // The candidates still pending from the warp's last tile.
    if (warp >= kEpiWarpBase) finish_all();
  }

  // ---- 3. teardown ----------------------------------------------------------------------------
  // When every role finished its lists, every copy issued was consumed (the MMA waited for it)
  // and every MMA completed (the epilogue waited for it).  Only after a wait gave up can copies
  // still be in flight; then the producer waits for the last loads of each stage and the last q/w.
  if (__syncthreads_or(!ok)) {
    if (!ok) flag_error(IDX_DEV_WAIT_TIMEOUT);
    if (warp == 0 && lane == 0) {
      // The producer's copies land on full (MX: on raw_full, the raw ring's barriers).
      constexpr int kRing = C::MX ? C::RAW_STAGES : C::STAGES;
      uint64_t *landed = C::MX ? raw_full : full;
      const int tail = kbase < kRing ? kbase : kRing;
      for (int d = 1; d <= tail; ++d) {
        const int s = ((stage - d) % kRing + kRing) % kRing;
        const uint32_t ph = (stage - d < 0) ? (phase ^ 1) : phase;
        if (!mbar_wait(&landed[s], ph, kWaitLimitNs)) flag_error(IDX_DEV_WAIT_TIMEOUT);
      }
      if (qcount > 0 &&
          !mbar_wait(&q_full[(qcount - 1) & 1], ((qcount - 1) >> 1) & 1, kWaitLimitNs))
        flag_error(IDX_DEV_WAIT_TIMEOUT);
    }
  }
  if (warp == 1 && lane == 0) {
    // Every MMA issued (and every commit behind one) has completed once the drain arrives.
    if (!drained) mma_commit(drain);
    if (!mbar_wait(drain, 0, kWaitLimitNs)) flag_error(IDX_DEV_WAIT_TIMEOUT);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

template <int NN, int H, int D, typename OutT, int BS_SHIFT, bool MX = false>
cudaError_t launch_nn(const CUtensorMap &kv_map, const CUtensorMap &q_map, const LogitsArgs &args,
                      int num_ctas, cudaStream_t stream) {
  using C = Cfg<NN, H, D, MX>;
  const uint32_t smem = C::smem_bytes(args.batch);
  static PerDeviceOnce configured;
  const cudaError_t e = configured.run([] {
    return cudaFuncSetAttribute(k_logits_fp8<NN, H, D, OutT, BS_SHIFT, MX>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::smem_bytes(kMaxBatch));
  });
  if (e != cudaSuccess) return e;
  return launch_dependent(k_logits_fp8<NN, H, D, OutT, BS_SHIFT, MX>, dim3(num_ctas),
                          dim3(C::THREADS), smem, stream, kv_map, q_map, args);
}

template <int H, int D, typename OutT, int BS_SHIFT, bool MX = false>
cudaError_t launch_bs(int next_n, const CUtensorMap &kv_map, const CUtensorMap &q_map,
                      const LogitsArgs &args, int num_ctas, cudaStream_t stream) {
  switch (next_n) {
    case 1: return launch_nn<1, H, D, OutT, BS_SHIFT, MX>(kv_map, q_map, args, num_ctas, stream);
    case 2: return launch_nn<2, H, D, OutT, BS_SHIFT, MX>(kv_map, q_map, args, num_ctas, stream);
    case 3: return launch_nn<3, H, D, OutT, BS_SHIFT, MX>(kv_map, q_map, args, num_ctas, stream);
    case 4: return launch_nn<4, H, D, OutT, BS_SHIFT, MX>(kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int H, int D, typename OutT, bool MX = false>
cudaError_t launch_out(int next_n, const CUtensorMap &kv_map, const CUtensorMap &q_map,
                       const LogitsArgs &args, int num_ctas, cudaStream_t stream) {
  switch (args.block_size) {
    case 32: return launch_bs<H, D, OutT, 5, MX>(next_n, kv_map, q_map, args, num_ctas, stream);
    case 64: return launch_bs<H, D, OutT, 6, MX>(next_n, kv_map, q_map, args, num_ctas, stream);
    case 128: return launch_bs<H, D, OutT, 7, MX>(next_n, kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int H, int D>
cudaError_t launch_shape(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                         const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                         cudaStream_t stream) {
  switch (mode) {
    case LogitsOut::kF32:
      return launch_out<H, D, float>(next_n, kv_map, q_map, args, num_ctas, stream);
    case LogitsOut::kF16:
      return launch_out<H, D, __half>(next_n, kv_map, q_map, args, num_ctas, stream);
    case LogitsOut::kSelect:
      return launch_out<H, D, SelectOut>(next_n, kv_map, q_map, args, num_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

// Sets this translation unit's fault-injection CTA (-1: off); synchronous.
inline cudaError_t set_unit_withhold(int32_t cta) {
  return cudaMemcpyToSymbol(g_withhold_cta, &cta, sizeof(int32_t));
}

// 8 or 16 heads: float32 and float16 output only (the fused select takes 32 or 64 heads).
template <int H, int D>
cudaError_t launch_shape_plain(int next_n, LogitsOut mode, const CUtensorMap &kv_map,
                               const CUtensorMap &q_map, const LogitsArgs &args, int num_ctas,
                               cudaStream_t stream) {
  switch (mode) {
    case LogitsOut::kF32:
      return launch_out<H, D, float>(next_n, kv_map, q_map, args, num_ctas, stream);
    case LogitsOut::kF16:
      return launch_out<H, D, __half>(next_n, kv_map, q_map, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Reads (and, if `clear`, resets) this translation unit's status bits.
inline cudaError_t read_unit_status(int32_t *value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_logits_status, sizeof(int32_t));
  if (e != cudaSuccess || !clear) return e;
  const int32_t zero = 0;
  return cudaMemcpyToSymbol(g_logits_status, &zero, sizeof(int32_t));
}

}  // namespace
}  // namespace idx
