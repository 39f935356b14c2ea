// Activation quantiser: f32 X[N][K] -> int8 Xq[N][K], f32 da[K/32][ldda] and
// the binary16 operand plane Xh[N][K] read by the tensor-core GEMM.
//
// Per token n and 32-element block c: amax = max|x|, da = amax/127,
// xq = clamp(round_half_away(x/da), -127, 127); amax == 0 gives da = 0 and
// xq = 0. The per-32 activation scale is the one the q6_K rescale consumes
// ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2); the pages print no
// quantiser, so the division and the rounding are IEEE f32 and half-away.
//
// HBM-bound: 4 bytes read and 3 written per element. Each thread owns four
// consecutive elements (one float4); eight threads of a warp form one block
// and reduce amax with three xor-shuffles.
#include "q6_internal.cuh"

namespace q6 {
namespace {

__device__ __forceinline__ int quant1(float x, float d) {
  if (d == 0.0f) return 0;
  const float r = roundf(__fdiv_rn(x, d));
  return (int)fminf(fmaxf(r, -127.0f), 127.0f);
}

__global__ void __launch_bounds__(256) q8_quantize_kernel(const float* __restrict__ X, int N, int K,
                                                          int ldx, int8_t* __restrict__ Xq,
                                                          float* __restrict__ da, int ldda,
                                                          __half* __restrict__ Xh) {
  const long long per_row = K >> 2;
  const long long total = (long long)N * per_row;  // a multiple of 64: whole warps stay active
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += stride) {
    const int n = (int)(g / per_row);
    const int j = (int)(g - (long long)n * per_row);  // float4 index in the row
    const float4 v = __ldg(reinterpret_cast<const float4*>(X + (size_t)n * ldx) + j);
    float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    const float d = __fdiv_rn(a, 127.0f);
    const int q0 = quant1(v.x, d), q1 = quant1(v.y, d), q2 = quant1(v.z, d), q3 = quant1(v.w, d);
    const uint32_t packed = (uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8) |
                            ((uint32_t)(q2 & 0xFF) << 16) | ((uint32_t)(q3 & 0xFF) << 24);
    reinterpret_cast<uint32_t*>(Xq + (size_t)n * K)[j] = packed;
    if (Xh != nullptr) {
      const __half2 h01 = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
      const __half2 h23 = __halves2half2(__int2half_rn(q2), __int2half_rn(q3));
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&h01);
      w.y = *reinterpret_cast<const uint32_t*>(&h23);
      reinterpret_cast<uint2*>(Xh + (size_t)n * K)[j] = w;
    }
    if ((j & 7) == 0) da[(size_t)(j >> 3) * ldda + n] = d;
  }
}

}  // namespace

cudaError_t launch_quantize(const float* X, int N, int K, int ldx, int8_t* Xq, float* da, int ldda,
                            __half* Xh, cudaStream_t s) {
  const long long total = (long long)N * (K / 4);
  long long blocks = (total + 255) / 256;
  const long long cap = 152LL * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  q8_quantize_kernel<<<(unsigned)blocks, 256, 0, s>>>(X, N, K, ldx, Xq, da, ldda, Xh);
  return cudaGetLastError();
}

}  // namespace q6
