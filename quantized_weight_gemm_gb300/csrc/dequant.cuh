// Register-level decoding of packed 4-bit weight words.  The GEMM kernels and the
// dequant-debug kernel call exactly these functions.
//
// BF16 activations (tensor-core operand BF16): a 32-bit word holds K-elements 8j..8j+7 of
// one weight row with nibbles ordered [e0, e2, e4, e6, e1, e3, e5, e7] from bit 0, so pair
// i = (e_2i, e_2i+1) sits in nibble i (bits 4i..) and nibble 4+i (bits 16+4i..) and one
// 0x000F000F mask of (word >> 4i) yields both 16-bit lanes.
//   INT4: the nibble u is ORed into the mantissa of 128.0 (bf16 0x4300), giving 128 + u
//   exactly; subtracting 128 + z gives the exact integer u - z; one BF16 multiply by the
//   group scale s then rounds (u - z) * s to nearest even, the value a BF16 MMA consumes.
//   Symmetric INT4 is stored as u = q + 8 and decoded with z = 8 (the "magic number"
//   construction of Kim et al., "Who Says Elephants Can't Run?", 2022, restated from the
//   bfloat16 format definition).
//   INT4 with BF16 scales runs on FP16 operands instead (the same construction in FP16:
//   1024.0 = 0x6400 has a unit last place, so 0x6400 | u is 1024 + u): one FP16 multiply
//   by s * 2^k rounds (u - z) * s * 2^k to 11 significant bits, where BF16 would keep 8
//   of the up to 12 that the product has.
//   MXFP4 (codes in natural order, one byte = two elements): a byte permute places the
//   byte's two nibbles at bits 0..3 and 16..19; then the e2m1 magnitude bits (e1 e0 m) are
//   moved to bf16 bits 8..6 and the sign to
//   bit 15, which is the bf16 number e2m1(q) * 2^-126 (a subnormal for e = 0); multiplying
//   by 2^(E-1) (or by 2^127 and then 2^(E-128) when E > 128) gives e2m1(q) * 2^(E-127),
//   exact unless it overflows bf16.
//   MXINT4: the INT4 decode with z = 8 and the scale 2^(E-127) as a BF16 factor (the
//   subnormal 2^-127 for E = 0): q * 2^(E-127), exact unless it overflows bf16.
//   NVFP4: the MXFP4 bit move, then one multiply by the E4M3 group scale s times 2^118,
//   giving e2m1(q) * s * 2^-8 -- exact, since e2m1 and E4M3 significands have 2 and 4 bits
//   and the result stays in the normal range; the GEMM multiplies its FP32 accumulators by
//   2^8 and the per-tensor scale.
//
// FP8 activations (tensor-core operand E4M3 with block scales): a word holds K-elements
// 8j..8j+7 with nibbles [e0, e4, e1, e5, e2, e6, e3, e7], so masking low nibbles gives
// bytes for e0..e3 and high nibbles bytes for e4..e7.  An e2m1 code s e1 e0 m becomes the
// e4m3 byte s 0 0 e1 e0 m 0 0, whose value is exactly e2m1(q) * 2^-6 (also for the
// subnormal code); the factor 2^6 is returned through the activation-side block scale.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace qgemm {

// INT4 word -> 4 bf16x2 (pairs 0..3).  zz = bf16x2(128 + z), s2 = bf16x2(scale).
__device__ __forceinline__ void decode_int4_word(uint32_t w, uint32_t zz, uint32_t s2,
                                                 uint32_t* out) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = ptx::lop3_and_or(w >> (4 * i), 0x000F000Fu, 0x43004300u);
    out[i] = ptx::bf16x2_mul(ptx::bf16x2_sub(t, zz), s2);
  }
}

// INT4 word -> 4 f16x2 (pairs 0..3).  zz = f16x2(1024 + z), zz64 = f16x2(64 + z),
// s2 = f16x2(scale * 2^k).  Pairs 0 and 2 sit in nibbles 0 / 4 (of w and of w >> 8): ORed
// into the mantissa of 1024.0 they give 1024 + q.  Pairs 1 and 3 sit in nibbles 1 / 5, bits
// 4..7 of each half: ORed into 64.0 (0x5400, whose last place is 1/16) they give 64 + q, so
// no shift is needed for them.  Subtracting the matching 1024 + z or 64 + z is exact.
__device__ __forceinline__ void decode_int4_word_f16(uint32_t w, uint32_t zz, uint32_t zz64,
                                                     uint32_t s2, uint32_t* out) {
  const uint32_t w8 = w >> 8;
  out[0] = ptx::f16x2_mul(ptx::f16x2_sub(ptx::lop3_and_or(w, 0x000F000Fu, 0x64006400u), zz), s2);
  out[1] = ptx::f16x2_mul(ptx::f16x2_sub(ptx::lop3_and_or(w, 0x00F000F0u, 0x54005400u), zz64), s2);
  out[2] = ptx::f16x2_mul(ptx::f16x2_sub(ptx::lop3_and_or(w8, 0x000F000Fu, 0x64006400u), zz), s2);
  out[3] = ptx::f16x2_mul(ptx::f16x2_sub(ptx::lop3_and_or(w8, 0x00F000F0u, 0x54005400u), zz64), s2);
}

// f16x2 of a BF16 scale (bits) times the power of two p, rounded once to FP16.
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t s_bf16, float p) {
  const float v = __uint_as_float(s_bf16 << 16) * p;
  return ptx::cvt_f16x2_f32(v, v);
}

// MXFP4 word -> 4 bf16x2.  sa, sb: bf16x2 factors (sb == 0 means single multiply).
__device__ __forceinline__ void decode_mxfp4_word(uint32_t w, uint32_t sa, uint32_t sb,
                                                  bool two_step, uint32_t* out) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = (w >> (4 * i)) & 0x000F000Fu;
    const uint32_t v = (t * 0x1040u) & 0x81C081C0u;   // sign -> bit 15, e1 e0 m -> bits 8..6
    uint32_t r = ptx::bf16x2_mul(v, sa);
    if (two_step) r = ptx::bf16x2_mul(r, sb);
    out[i] = r;
  }
}

// MXFP4 word in natural order (element 2j in the low nibble of byte j) -> 4 bf16x2: the low
// and the high nibbles of all four bytes are masked out once (u, v); one byte permute then
// takes byte j of u to byte 0 and byte j of v to byte 2, with zero bytes between (the
// selector's sign-replicate bit on a byte below 16), which puts pair j's two codes at bits
// 0..3 and 16..19; then the bit move above.
__device__ __forceinline__ void decode_mxfp4_word_nat(uint32_t w, uint32_t sa, uint32_t sb,
                                                      bool two_step, uint32_t* out) {
  const uint32_t u = w & 0x0F0F0F0Fu, v = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = ptx::prmt(u, v, 0x8080u | uint32_t(i) | (uint32_t(4 + i) << 8));
    const uint32_t x = (t * 0x1040u) & 0x81C081C0u;
    uint32_t r = ptx::bf16x2_mul(x, sa);
    if (two_step) r = ptx::bf16x2_mul(r, sb);
    out[i] = r;
  }
}

// MXFP4 word in natural order -> 4 f16x2: the hardware e2m1x2 -> f16x2 conversion (exact),
// then one FP16 multiply by f2 = the block's 2^(E - 127 + k) (exact while the product stays
// on FP16's grid, see PackedHeader::w_prescale).
__device__ __forceinline__ void decode_mxfp4_word_f16(uint32_t w, uint32_t f2, uint32_t* out) {
  out[0] = ptx::f16x2_mul(ptx::cvt_f16x2_e2m1x2<0>(w), f2);
  out[1] = ptx::f16x2_mul(ptx::cvt_f16x2_e2m1x2<1>(w), f2);
  out[2] = ptx::f16x2_mul(ptx::cvt_f16x2_e2m1x2<2>(w), f2);
  out[3] = ptx::f16x2_mul(ptx::cvt_f16x2_e2m1x2<3>(w), f2);
}

// f16x2 of 2^(E - 127) * p for an E8M0 exponent E and a power of two p (FP32 2^(E-127) is
// exact, also the subnormal 2^-127 for E = 0; the product rounds once to FP16, to 0 far
// below FP16's range).
__device__ __forceinline__ uint32_t e8m0_f16x2(uint32_t E, float p) {
  const float v = __uint_as_float(E != 0u ? (E << 23) : 0x00400000u) * p;
  return ptx::cvt_f16x2_f32(v, v);
}

// bf16x2 factors applying 2^(E-127) to the subnormal-offset e2m1 value (see above).
__device__ __forceinline__ void mxfp4_factors(uint32_t E, uint32_t& sa, uint32_t& sb,
                                              bool& big) {
  big = E > 128u;
  const uint32_t a = big ? 0x7F00u : ((E + 126u) << 7);      // 2^127   or 2^(E-1)
  const uint32_t b = big ? ((E - 1u) << 7) : 0x3F80u;        // 2^(E-128) or 1
  sa = a | (a << 16);
  sb = b | (b << 16);
}

// bf16x2 of 2^(E-127) for an E8M0 exponent E < 255 (E = 0: the bf16 subnormal 2^-127).
__device__ __forceinline__ uint32_t e8m0_bf16x2(uint32_t E) {
  return (E != 0u ? (E << 7) : 0x0040u) * 0x00010001u;
}

// bf16x2 of (E4M3 value of byte b) * 2^118, exact: the significand (8 + m for a normal,
// m for a subnormal) shifted by the exponent is an integer below 2^18, and the value
// 2^(e-1) (8 + m) 2^109 = (1 + m/8) 2^(e-7) 2^118 has at most 4 significant bits.  NaN
// codes never get here (the repack refuses them).
__device__ __forceinline__ uint32_t e4m3_bf16x2_p118(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  const uint32_t sig = e != 0u ? ((8u | m) << (e - 1u)) : m;
  const float v = __uint2float_rn(sig) * 0x1p109f;
  const uint32_t h = (__float_as_uint(v) >> 16) | ((b & 0x80u) << 8);
  return h * 0x00010001u;
}

// MXFP4 word (FP8 nibble order) -> two 32-bit words of four e4m3 bytes each.
__device__ __forceinline__ void decode_e2m1_to_e4m3_word(uint32_t w, uint32_t& lo,
                                                         uint32_t& hi) {
  const uint32_t a = w & 0x0F0F0F0Fu;
  const uint32_t b = (w >> 4) & 0x0F0F0F0Fu;
  lo = ((a & 0x07070707u) << 2) | ((a & 0x08080808u) << 4);
  hi = ((b & 0x07070707u) << 2) | ((b & 0x08080808u) << 4);
}

// ------------------------------------------------------------------------ layout helpers
// Position of K-element e (0..7) of a word in the nibble order used for BF16 activations.
__host__ __device__ constexpr int nibble_pos_a16(int e) { return (e & 1) ? 4 + (e >> 1) : (e >> 1); }
// ... and for FP8 activations.
__host__ __device__ constexpr int nibble_pos_a8(int e) { return (e < 4) ? 2 * e : 2 * (e - 4) + 1; }

}  // namespace qgemm
