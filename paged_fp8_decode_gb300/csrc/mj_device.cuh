// Device helpers shared by the kernels: number-format conversions, exp2,
// warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace mj {

// Two e4m3 codes (low byte first) -> two floats, exactly (every e4m3 value is
// an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xFFFFu),
                                             __NV_E4M3);
  __half2 hh;
  memcpy(&hh, &h, sizeof(hh));
  return __half22float2(hh);
}

// Four packed e4m3 codes of a 32-bit word (byte 0 first) -> four floats.
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float out[4]) {
  float2 a = e4m3x2_to_float2(w);
  float2 b = e4m3x2_to_float2(w >> 16);
  out[0] = a.x;
  out[1] = a.y;
  out[2] = b.x;
  out[3] = b.y;
}

// Widen four 6-bit e2m3 codes, one per byte (code in bits 0-5), to four e4m3
// codes whose value is the e2m3 value times 2^-6.
//
// An e2m3 code s|EE|MMM read as the e4m3 code s|00EE|MMM (the sign moved to
// bit 7, the exponent field zero-extended) has exponent E-7 instead of E-1
// for E>0, and subnormal step 2^-9 instead of 2^-3 for E=0: in both cases the
// value is scaled by exactly 2^-6. So the widening is one bit move per byte
// and is exact; the factor 64 is folded into the K/V scales.
__device__ __forceinline__ uint32_t e2m3x4_to_e4m3x4(uint32_t four_codes) {
  return (four_codes & 0x1F1F1F1Fu) | ((four_codes & 0x20202020u) << 2);
}

// Widen four 6-bit e3m2 codes (one per byte) to e4m3 codes worth 2^-4 times
// the e3m2 values: s|EEE|MM read as s|0EEE|MM0 has exponent E-7 instead of
// E-3 (subnormals: step 2^-8 instead of 2^-4), the same scaling by 2^-4 in
// both cases, so the move is exact.
__device__ __forceinline__ uint32_t e3m2x4_to_e4m3x4(uint32_t four_codes) {
  return ((four_codes & 0x1F1F1F1Fu) << 1) | ((four_codes & 0x20202020u) << 2);
}

// Widen four 4-bit e2m1 codes (one per byte) to e4m3 codes worth 2^-6 times
// the e2m1 values: s|EE|M read as s|00EE|M00 (exponent E-7 instead of E-1;
// the subnormal 0.5 becomes 2^-7), exact.
__device__ __forceinline__ uint32_t e2m1x4_to_e4m3x4(uint32_t four_codes) {
  return ((four_codes & 0x07070707u) << 2) | ((four_codes & 0x08080808u) << 4);
}

// Spread four 6-bit codes held in the low 24 bits of `g` (code i at bits
// [6i, 6i+6), the little-endian bitstream) into the four bytes of a word.
__device__ __forceinline__ uint32_t spread6x4(uint32_t g) {
  return (g & 0x3Fu) | ((g << 2) & 0x3F00u) | ((g << 4) & 0x3F0000u) | ((g << 6) & 0x3F000000u);
}

// Spread four 4-bit codes held in the low 16 bits of `h` (code i at bits
// [4i, 4i+4)) into the four bytes of a word.
__device__ __forceinline__ uint32_t spread4x4(uint32_t h) {
  return (h & 0xFu) | ((h << 4) & 0xF00u) | ((h << 8) & 0xF0000u) | ((h << 12) & 0xF000000u);
}


// 2^x with the hardware approximation (ex2.approx, relative error ~2^-22).
// exp2(-inf) = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  uint16_t u;
  memcpy(&u, &h, sizeof(u));
  return u;
}

__device__ __forceinline__ uint16_t float_to_f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

// the decode output element: bf16 or fp16, rounded to nearest even
__device__ __forceinline__ uint16_t float_to_out_bits(float x, int f16) {
  return f16 ? float_to_f16_bits(x) : float_to_bf16_bits(x);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t u) {
  return __uint_as_float(uint32_t(u) << 16);
}

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

}  // namespace mj
