// mx_convert.cuh -- MXFP4 -> e4m3 conversion of one 32-element group ("flashinfer.attn_scores",
// fp4_paged_mqa_logits: Parameters q, q_sf, kv_fused; sf_vec_size = 32), shared by the staging
// kernels (mxfp4.cu) and the logits kernel's converter warps (logits_kernel.cuh).
//
// An element is e2m1(nibble) * 2^(e - 127) with e its group's UE8M0 scale byte.  A row's largest
// scale 2^(E - 127) leaves the row (it multiplies the q head's weight, or becomes the K token's
// float32 scale: a positive power of two commutes with the ReLU), and what stays of a group is
// e2m1 * 2^(e - E), e - E <= 0.  For e - E >= -8 every such value is an e4m3 number (the
// smallest, 0.5 * 2^-8, is e4m3's smallest subnormal 2^-9), so the conversion is exact; below
// that, or for the NaN scale byte 0xFF, it rounds (to nearest, saturating) and reports it.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace idx {

// An E2M1 code (OCP microscaling FP4: sign, 2 exponent bits with bias 1, 1 mantissa bit) as a
// float: built from its fields; exponent field 0 is the subnormal m/2.
__device__ __forceinline__ float e2m1_value(uint32_t nibble) {
  const uint32_t e = (nibble >> 1) & 3u, m = nibble & 1u;
  const float mag = e != 0u ? __uint_as_float(((e + 126u) << 23) | (m << 22)) : 0.5f * m;
  return (nibble & 8u) ? -mag : mag;
}

// 2^k for -149 <= k <= 127 (k = -127 .. -149 as float32 subnormals).
__device__ __forceinline__ float pow2f(int k) {
  return k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23)
                   : __uint_as_float(1u << (k + 149));
}

// The e4m3 bytes of the eight E2M1 magnitudes (codes 0..7) times 2^-r, r = 0..8, as two words
// (bytes 0..3, 4..7): the table the fast conversion looks up.  Exact (see the file comment).
__device__ __forceinline__ uint2 e2m1_table_entry(int r) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float v = e2m1_value(static_cast<uint32_t>(m)) * pow2f(-r);
    const uint32_t byte = __nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3) & 0xFFu;
    w[m >> 2] |= byte << (8 * (m & 3));
  }
  return make_uint2(w[0], w[1]);
}

// prmt.b32 in its default mode: each selector nibble picks one of the eight bytes of {hi, lo}
// (bits 2..0); with bit 3 set, that byte's bit 7 is replicated over the result byte.
__device__ __forceinline__ uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(lo), "r"(hi), "r"(sel));
  return d;
}

// Eight E2M1 codes (one packed word, element 2j in the low nibble of byte j) -> eight e4m3 bytes
// (two words, elements 0..3 and 4..7), with the magnitudes looked up in `tab` (one table entry).
// Magnitude: a byte permute indexed by the nibbles' low 3 bits.  Sign: a byte permute in
// sign-replicating mode picks, for each element, the byte of w or w << 4 whose bit 7 is the
// nibble's bit 3.
__device__ __forceinline__ void e2m1x8_to_e4m3(uint32_t w, uint2 tab, uint32_t &a, uint32_t &b) {
  const uint32_t w4 = w << 4;
  const uint32_t m = w & 0x77777777u;        // the eight codes' magnitudes; prmt reads a
  const uint32_t ma = prmt(tab.x, tab.y, m);  // selector's low 16 bits only
  const uint32_t mb = prmt(tab.x, tab.y, m >> 16);
  const uint32_t sa = prmt(w, w4, 0x9D8Cu);  // elements 0..3: bytes 4, 0, 5, 1 (sign mode)
  const uint32_t sb = prmt(w, w4, 0xBFAEu);  // elements 4..7: bytes 6, 2, 7, 3 (sign mode)
  a = ma | (sa & 0x80808080u);
  b = mb | (sb & 0x80808080u);
}

// One group of 32 codes (16 packed bytes) at relative exponent rel = e - E <= 0 -> 32 e4m3 bytes
// (out[0..7], element order).  Exact for rel >= -8 (table lookups, `tab` = the entry for -rel);
// otherwise each element is rounded through float32, and *inexact is set if the group is not
// all zeros.
__device__ __forceinline__ void mx_group_to_e4m3(uint4 in, int rel, uint2 tab, uint32_t (&out)[8],
                                                 bool *inexact) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  if (rel >= -8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) e2m1x8_to_e4m3(w[k], tab, out[2 * k], out[2 * k + 1]);
    return;
  }
  const float f = pow2f(max(rel, -149));
  bool nonzero = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    nonzero = nonzero || (w[k] & 0x77777777u) != 0u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t bits = w[k] >> (16 * half);  // elements 8k+4h .. +3, low nibble first
      uint32_t word = 0;
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        const float2 v = make_float2(e2m1_value((bits >> (8 * pr)) & 0xFu) * f,
                                     e2m1_value((bits >> (8 * pr + 4)) & 0xFu) * f);
        const uint32_t two = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
        word |= (two & 0xFFFFu) << (16 * pr);
      }
      out[2 * k + half] = word;
    }
  }
  if (nonzero) *inexact = true;
}

}  // namespace idx
