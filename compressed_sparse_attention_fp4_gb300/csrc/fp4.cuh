// fp4.cuh -- the FP4 format on the device: E2M1 values with one E4M3 scale
// per 16 channels (foosynaptic atlas "DeepSeek-V4.1-Flash 梗概", section 3.2,
// "FP4 main KV"; newsaint.id "DeepSeek-V4.1-Flash 2026: ...", section 8,
// FP4Quantizer: levels {0,.5,1,1.5,2,3,4,6}, scale = amax/6 limited to 448,
// no second-level scale).  Shared by the main-KV codec, the FP4 indexer-key
// write and the FP4 indexer scan (which quantizes its query the same way).
//
// Rounding (the reading this library implements):
//   s_code = E4M3 round-to-nearest-even, saturating, of amax/6;
//   magnitude code = nearest E2M1 level to |x|/s, ties to the even code,
//   saturating at 6; the sign bit of x is kept; s == 0 gives magnitude 0.
// Both roundings use the hardware RNE conversions.  amax/6 is formed with a
// correctly rounded fp32 division: amax has <= 8 significant bits, so amax/6
// is exact or non-terminating in binary and can never sit on an E4M3
// midpoint -- rounding it first to fp32 cannot change the E4M3 result.
// |x|/s is formed as r0 = |x|*rcp(s) plus one FMA residual correction: away
// from an E2M1 midpoint |x|/s is at least 2^-8 (relative) from it, far more
// than r0's error; on an exact midpoint the correction returns it exactly,
// so the conversion sees the exact tie and rounds it to the even code.
#pragma once

#include "common.cuh"

namespace csa2 {

__device__ inline uint32_t e2m1x2_rn(float hi, float lo) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xFF;
}

__device__ inline uint32_t f32_to_e4m3_rn(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return uint32_t(r) & 0xFF;
}

// |x| / s rounded so that RNE onto the E2M1 grid sees the exact decision.
__device__ inline float scaled_mag(float ax, float s, float rcp) {
  float r0 = ax * rcp;
  float e = __fmaf_rn(-r0, s, ax);
  return __fmaf_rn(rcp, e, r0);
}

// Scale code of a group with largest magnitude amax, its value s and the
// reciprocal used by scaled_mag (0 for a zero scale).
__device__ inline uint32_t fp4_group_scale(float amax, float& s, float& rcp) {
  const uint32_t sc = f32_to_e4m3_rn(__fdiv_rn(amax, 6.0f));
  s = e4m3_to_f32(sc);
  rcp = s > 0.0f ? __frcp_rn(s) : 0.0f;
  return sc;
}

// Packed nibbles of 8 consecutive bf16 channels (channel 2j in the low half
// of word j) under a group scale: channel 2j in the low nibble of byte j.
__device__ inline uint32_t fp4_pack8(const uint32_t (&w)[4], float s, float rcp) {
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] << 16, hi = w[i] & 0xFFFF0000u;
    const float m0 = scaled_mag(__uint_as_float(lo & 0x7FFFFFFFu), s, rcp);
    const float m1 = scaled_mag(__uint_as_float(hi & 0x7FFFFFFFu), s, rcp);
    const uint32_t byte = e2m1x2_rn(m1, m0) | ((lo >> 31) << 3) | ((hi >> 31) << 7);
    packed |= byte << (8 * i);
  }
  return packed;
}

__device__ inline float bf16x8_amax(const uint32_t (&w)[4]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    amax = fmaxf(amax, fmaxf(__uint_as_float((w[i] << 16) & 0x7FFFFFFFu), __uint_as_float(w[i] & 0x7FFF0000u)));
  return amax;
}

// One lane's half of a 16-channel group: v holds 8 consecutive bf16 channels;
// the group's other 8 channels sit in lane ^ 1 (both lanes must call this
// together).  Returns the 4 packed bytes of this lane's channels and sets
// *scale to the group's E4M3 scale code.
__device__ inline uint32_t fp4_quantize_half_group(uint4 v, uint32_t* scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float amax = bf16x8_amax(w);
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  float s, rcp;
  *scale = fp4_group_scale(amax, s, rcp);
  return fp4_pack8(w, s, rcp);
}

// A whole 16-channel group held by one thread (lo: channels 0..7, hi:
// channels 8..15): 8 packed bytes (lo word first) and the scale code.
__device__ inline uint2 fp4_quantize_group(uint4 lo, uint4 hi, uint32_t* scale) {
  const uint32_t a[4] = {lo.x, lo.y, lo.z, lo.w}, b[4] = {hi.x, hi.y, hi.z, hi.w};
  float s, rcp;
  *scale = fp4_group_scale(fmaxf(bf16x8_amax(a), bf16x8_amax(b)), s, rcp);
  return make_uint2(fp4_pack8(a, s, rcp), fp4_pack8(b, s, rcp));
}

// Eight E2M1 nibbles (nibble k of w = channel k) as eight E4M3 bytes worth
// 2^-6 times their values, in the channel order 0, 2, 4, 6 (ev) and 1, 3, 5, 7
// (od): a nibble's three magnitude bits m go to bits 2..4 of its byte and its
// sign to bit 7.  (m = 0..3 land on the E4M3 subnormals / first binade as 0,
// 2^-7, 2^-6, 1.5 * 2^-6 and m = 4..7 on 2^-5, 1.5 * 2^-5, 2^-4, 1.5 * 2^-4:
// exactly 2^-6 * {0, .5, 1, 1.5, 2, 3, 4, 6}.)  A dot product is the same in
// any channel order, so keys and query widened alike multiply correctly.
__device__ inline void e2m1x8_to_e4m3x8_scaled(uint32_t w, uint32_t& ev, uint32_t& od) {
  ev = ((w & 0x07070707u) << 2) | ((w & 0x08080808u) << 4);
  od = ((w >> 2) & 0x1C1C1C1Cu) | (w & 0x80808080u);
}

// Four E2M1 nibbles (low 16 bits of w) as signed bytes of twice their values
// (-12 .. 12: every level times 2 is an integer).
__device__ inline uint32_t e2m1x4_to_i8x4_twice(uint32_t w) {
  const uint32_t sel = w & 0x7777u;
  const uint32_t pos = __byte_perm(0x03020100u, 0x0C080604u, sel);   //  0  1  2  3 |  4  6  8  12
  const uint32_t neg = __byte_perm(0xFDFEFF00u, 0xF4F8FAFCu, sel);   // -0 -1 -2 -3 | -4 -6 -8 -12
  const uint32_t t = __byte_perm(w, 0u, 0x1100u);
  const uint32_t sgn = ((t & 0x00080008u) << 4) | (t & 0x80008000u);  // bit 7 of byte k: sign of nibble k
  const uint32_t mask = (sgn >> 7) * 0xFFu;
  return (pos & ~mask) | (neg & mask);
}

}  // namespace csa2
