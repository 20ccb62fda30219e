// mxq.cuh -- activations in MXFP4 "terms" for the block-scaled tensor-core path.
//
// A vector v (bf16 x, or fp32 act) is written as a sum of kTerms MXFP4 vectors: for each
// group of 32 elements, term 0 is v rounded to E2M1 under the group's own E8M0 scale (the
// smallest power of two that puts the group's largest magnitude at or below 6), term 1 the
// same rounding of what term 0 left over, and so on.  Each term gains about two bits, so
// four terms carry v to roughly 2^-8 of the group maximum: the same order as the bf16 input
// itself.  The weights' E2M1 codes and scales are the checkpoint's own bytes (README
// "kimi-k3-in-c", Part II section 4); only the activations are split.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace k3 {

constexpr int kTerms = 4;

// E8M0 exponent e (unbiased) of a group with largest magnitude amax: the smallest e with
// amax <= 6 * 2^e, clamped to the E8M0 range; amax == 0 gives e = 0.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (amax == 0.f || (b >> 23) == 0) return amax == 0.f ? 0 : -127;
  const int x = (int)((b >> 23) & 255u) - 127;  // amax = m * 2^x, m in [1, 2)
  int e = x - 2 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);  // m > 1.5 needs one more
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Round a (|a| <= 6) to the nearest E2M1 value, ties to the even code; returns the 4-bit
// code (bit 3 = sign) and the value it stands for.  Branch-free (lanes of a warp hold
// different magnitudes): the code counts the rounding boundaries at or below |a|, with
// < or <= at each midpoint so that a tie goes to the even code.
__device__ __forceinline__ uint32_t e2m1_rne(float a, float* val) {
  const float m = fabsf(a);
  const uint32_t c = (uint32_t)(m > 0.25f) + (uint32_t)(m >= 0.75f) + (uint32_t)(m > 1.25f) +
                     (uint32_t)(m >= 1.75f) + (uint32_t)(m > 2.5f) + (uint32_t)(m >= 3.5f) +
                     (uint32_t)(m > 5.f);
  // E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 by code
  const float v = c <= 4u ? 0.5f * (float)c : (c == 7u ? 6.f : (float)c - 2.f);
  const bool neg = __float_as_uint(a) >> 31;
  *val = neg ? -v : v;
  return c | (neg ? 8u : 0u);
}

// 2^e as a float for e in [-127, 127] (exact: 2^-127 is a subnormal).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00200000u);
}

// Warp-wide max of |r| in one reduction: the bit patterns of non-negative floats are in
// their numeric order.
__device__ __forceinline__ float warp_absmax(float r) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(r))));
}

// The 4-bit codes of this lane's group of 8 lanes (lanes 8g .. 8g+7), packed lane 8g first
// in the low nibble: one ballot per code bit, then each ballot's 8 bits spread to every
// fourth bit position.
__device__ __forceinline__ uint32_t pack_codes8(uint32_t code, int lane) {
  const int sh = lane & 24;
  uint32_t w = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t x = (__ballot_sync(0xffffffffu, (code >> k) & 1u) >> sh) & 0xFFu;
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    w |= x << k;
  }
  return w;
}

// One warp, one group of 32 elements (lane i holds element i): the kTerms terms.  On return
// every lane holds word (lane/8) of each term's 16 packed bytes (low nibble = even element)
// in words[t], and each term's E8M0 byte in sf[t].
__device__ __forceinline__ void mx_split_group(float v, uint32_t (&words)[kTerms],
                                               uint32_t (&sf)[kTerms]) {
  const int lane = threadIdx.x & 31;
  float r = v;
#pragma unroll
  for (int t = 0; t < kTerms; ++t) {
    const int e = mx_scale_exp(warp_absmax(r));
    float q;
    const uint32_t code = e2m1_rne(r * pow2f(-e), &q);
    r -= q * pow2f(e);
    words[t] = pack_codes8(code, lane);
    sf[t] = (uint32_t)(e + 127);
  }
}

// The same for TB independent groups at once (one value each per lane): the terms of all
// groups advance together, so their reductions and ballots interleave.
template <int TB>
__device__ __forceinline__ void mx_split_groups(const float (&v)[TB], uint32_t (&words)[TB][kTerms],
                                                uint32_t (&sf)[TB][kTerms]) {
  const int lane = threadIdx.x & 31;
  float r[TB];
#pragma unroll
  for (int b = 0; b < TB; ++b) r[b] = v[b];
#pragma unroll
  for (int t = 0; t < kTerms; ++t) {
    float amax[TB];
#pragma unroll
    for (int b = 0; b < TB; ++b) amax[b] = warp_absmax(r[b]);
    uint32_t code[TB];
#pragma unroll
    for (int b = 0; b < TB; ++b) {
      const int e = mx_scale_exp(amax[b]);
      float q;
      code[b] = e2m1_rne(r[b] * pow2f(-e), &q);
      r[b] -= q * pow2f(e);
      sf[b][t] = (uint32_t)(e + 127);
    }
#pragma unroll
    for (int b = 0; b < TB; ++b) words[b][t] = pack_codes8(code[b], lane);
  }
}

// Two values (|v| <= 6 after scaling) rounded to E2M1 by the hardware conversion (nearest,
// ties to the even code: the same rounding as e2m1_rne), as one byte: lo in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_rn(float hi, float lo) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// The values of an E2M1 byte's two codes (exact), low nibble first.
__device__ __forceinline__ float2 e2m1x2_values(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// One thread, one group of 32 elements r[0..31] (consumed): the kTerms terms, as 16 packed
// bytes each (words[t][i] holds elements 8i .. 8i+7, element 8i in the low nibble) and an
// E8M0 byte.  The same arithmetic as mx_split_group, without cross-lane work; element pairs
// are rounded by the hardware conversion.
__device__ __forceinline__ void mx_split_lane32(float (&r)[32], uint32_t (&words)[kTerms][4],
                                                uint32_t (&sf)[kTerms]) {
#pragma unroll
  for (int t = 0; t < kTerms; ++t) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(r[i]));
    const int e = mx_scale_exp(amax);
    const float down = pow2f(-e), up = pow2f(e);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const uint32_t b = e2m1x2_rn(r[i + 1] * down, r[i] * down);
      const float2 q = e2m1x2_values(b);
      r[i] -= q.x * up;
      r[i + 1] -= q.y * up;
      w[i >> 3] |= b << (4 * (i & 7));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) words[t][i] = w[i];
    sf[t] = (uint32_t)(e + 127);
  }
}

// Four lanes (a quad, t4 = lane % 4), one group of 32 elements: lane t4 holds elements
// 8 t4 .. 8 t4 + 7 in r (consumed).  The kTerms terms, with the arithmetic of mx_split_lane32
// (the group maximum over all 32, each element rounded alone): on return w[t] is lane t4's
// 4 bytes of term t's 16 code bytes (bytes 4 t4 .. 4 t4 + 3, element 8 t4 in the low nibble)
// and sf[t] the term's E8M0 byte (the same in the four lanes).  Every lane of the warp calls it.
__device__ __forceinline__ void mx_split_quad8(float (&r)[8], uint32_t (&w)[kTerms],
                                               uint32_t (&sf)[kTerms]) {
#pragma unroll
  for (int t = 0; t < kTerms; ++t) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(r[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int e = mx_scale_exp(amax);
    const float down = pow2f(-e), up = pow2f(e);
    uint32_t word = 0u;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const uint32_t b = e2m1x2_rn(r[i + 1] * down, r[i] * down);
      const float2 q = e2m1x2_values(b);
      r[i] -= q.x * up;
      r[i + 1] -= q.y * up;
      word |= b << (4 * i);
    }
    w[t] = word;
    sf[t] = (uint32_t)(e + 127);
  }
}

}  // namespace k3
