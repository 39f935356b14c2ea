// Per-element arithmetic of the activation quantiser, shared by every kernel
// that quantises (the standalone quantiser and the fused one- and two-token
// GEMM), so that all of them produce the same codes and scales.
//
// Per token n and 32-element block c: amax = max|x|, da = amax/127,
// xq = clamp(round_half_away(x/da), -127, 127); amax == 0 gives da = 0 and
// xq = 0 ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2 consumes this
// per-32 scale; the pages print no quantiser, so the division and the
// rounding are IEEE f32 and half-away).
#pragma once
#include "q6_internal.cuh"

namespace q6 {
namespace {

__device__ __forceinline__ int quant1(float x, float d) {
  if (d == 0.0f) return 0;
  const float r = roundf(__fdiv_rn(x, d));
  return (int)fminf(fmaxf(r, -127.0f), 127.0f);
}

// The code of x in a block with a normal scale d, given r = 1/d correctly
// rounded. With |x| <= amax and d = amax/127 rounded, |x / d| <= 127.00001,
// and q = x * r differs from the correctly rounded quotient x / d by at most
// 2^-15.6 (two roundings of relative size 2^-24 each, plus half an ulp of the
// quotient). So unless q lies within 2^-14 of a rounding tie both round to
// the same integer, by any rounding rule: the code is rint(q). Near a tie
// `near` is set and the caller takes the exact division.
__device__ __forceinline__ float qfast(float x, float r, bool& near) {
  const float q = x * r;
  const float n = rintf(q);
  near |= !(fabsf(q - n) < 0.5f - 0x1p-14f);
  return n;
}

// Eight elements of one block -> their codes as floats (exact integers), the
// fast way when possible and by the exact division otherwise.
__device__ __forceinline__ void quant8f(const float4 v0, const float4 v1, float d, float r,
                                        float (&n)[8]) {
  const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  bool near = !(d >= 0x1p-126f);  // zero or subnormal scale: the exact path
#pragma unroll
  for (int i = 0; i < 8; ++i) n[i] = qfast(x[i], r, near);
  if (near) {
#pragma unroll
    for (int i = 0; i < 8; ++i) n[i] = (float)quant1(x[i], d);
  }
}

// Codes (floats, -127..127) -> binary16 pairs, and -> int8 bytes through the
// binary16 bits of code + 1152 (0x64 above the byte code + 128).
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_q4(uint32_t h01, uint32_t h23) {
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  const __half2 a = __hadd2(*reinterpret_cast<const __half2*>(&h01), bias);
  const __half2 b = __hadd2(*reinterpret_cast<const __half2*>(&h23), bias);
  const uint32_t ua = *reinterpret_cast<const uint32_t*>(&a);
  const uint32_t ub = *reinterpret_cast<const uint32_t*>(&b);
  return __byte_perm(ua, ub, 0x6420) ^ 0x80808080u;
}

// Eight elements -> two words of int8 codes and four binary16 pairs.
__device__ __forceinline__ void quant8(const float4 v0, const float4 v1, float d, float r,
                                       uint2& q8, uint4& h8) {
  float n[8];
  quant8f(v0, v1, d, r, n);
  h8 = make_uint4(pack_h2(n[0], n[1]), pack_h2(n[2], n[3]), pack_h2(n[4], n[5]),
                  pack_h2(n[6], n[7]));
  q8 = make_uint2(pack_q4(h8.x, h8.y), pack_q4(h8.z, h8.w));
}

// Eight elements -> their binary16 codes only (the operand plane).
__device__ __forceinline__ void quant8h(const float4 v0, const float4 v1, float d, float r,
                                        uint4& h8) {
  float n[8];
  quant8f(v0, v1, d, r, n);
  h8 = make_uint4(pack_h2(n[0], n[1]), pack_h2(n[2], n[3]), pack_h2(n[4], n[5]),
                  pack_h2(n[6], n[7]));
}

// quant8, and the sum of the eight codes (an exact integer as a float).
__device__ __forceinline__ void quant8_sum(const float4 v0, const float4 v1, float d, float r,
                                           uint2& q8, uint4& h8, float& sum) {
  float n[8];
  quant8f(v0, v1, d, r, n);
  h8 = make_uint4(pack_h2(n[0], n[1]), pack_h2(n[2], n[3]), pack_h2(n[4], n[5]),
                  pack_h2(n[6], n[7]));
  q8 = make_uint2(pack_q4(h8.x, h8.y), pack_q4(h8.z, h8.w));
  sum = ((n[0] + n[1]) + (n[2] + n[3])) + ((n[4] + n[5]) + (n[6] + n[7]));
}

__device__ __forceinline__ float recip_or_zero(float d) {
  return d >= 0x1p-126f ? __frcp_rn(d) : 0.0f;
}

}  // namespace
}  // namespace q6
