// mxfp8.cuh -- device helpers for the MXFP8 format (OCP Microscaling): FP8
// E4M3 elements with one E8M0 scale byte 2^(b - 127) per 32 consecutive
// elements, as the page "SGLang and Miles Add Day-0 Support for Inkling"
// (section "Relative Logits Optimization", paragraph "MXFP8 Support") stores K
// and V.  A block's shared exponent is floor(log2(amax)) - 8 (8 = the
// exponent of E4M3's largest power of two), clamped to [-127, 127], -127 for
// an all-zero block; each element is x * 2^-e rounded to the nearest E4M3
// value (ties to even, the sign kept, saturating at 448).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace relattn {

// Two E4M3 codes, round-to-nearest-even with saturation: hi in bits 8..15, lo in 0..7.
__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^e as fp32 for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float pow2i(int e) {
  return e > -127 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Shared exponent of a block with largest magnitude amax.
__device__ __forceinline__ int mx_block_exponent(float amax) {
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);   // floor(log2 amax) + 127 for normals
  return ef == 0 ? -127 : max(-127, min(127, ef - 127 - 8));
}

// MXFP8 of 32 bf16 values (64 bytes at src, 16-byte aligned): the 32 codes in
// element order (c[i] holds elements 4i .. 4i+3, lowest byte first) and the
// shared exponent e.  x * 2^-e is exact in fp32 wherever the result can round
// to a non-zero code, so the codes are the exact round-to-nearest ones.
__device__ __forceinline__ void quantize_block32(const uint4 *src, uint32_t (&c)[8], int &e) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = src[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = __uint_as_float(ws[k] << 16);
      v[8 * i + 2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  e = mx_block_exponent(amax);
  const float inv = pow2i(-e);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    c[i] = e4m3x2(v[4 * i + 1] * inv, v[4 * i] * inv) | (e4m3x2(v[4 * i + 3] * inv, v[4 * i + 2] * inv) << 16);
}

// Four E4M3 codes (one 32-bit word, lowest byte = first element) times 2^e
// scale s, as four bf16 in two words (first element in the low half).  Exact:
// an E4M3 value has at most 4 significant bits, so the fp32 product keeps its
// low 16 bits zero and its top half is the bf16 value.
__device__ __forceinline__ void dequant4_bf16(uint32_t w, float s, uint32_t &o01, uint32_t &o23) {
  uint32_t h01, h23;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(w & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(w >> 16)));
  float f0, f1, f2, f3;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f0) : "h"((uint16_t)(h01 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(f1) : "h"((uint16_t)(h01 >> 16)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(f2) : "h"((uint16_t)(h23 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(f3) : "h"((uint16_t)(h23 >> 16)));
  o01 = (__float_as_uint(f0 * s) >> 16) | (__float_as_uint(f1 * s) & 0xffff0000u);
  o23 = (__float_as_uint(f2 * s) >> 16) | (__float_as_uint(f3 * s) & 0xffff0000u);
}

}  // namespace relattn
