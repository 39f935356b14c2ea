// Activation quantiser: f32 X[N][K] -> int8 Xq[N][K], f32 da[K/32][ldda] and
// the binary16 operand plane Xh[N][K] read by the tensor-core GEMM (either of
// Xq and Xh may be skipped).
//
// Per token n and 32-element block c: amax = max|x|, da = amax/127,
// xq = clamp(round_half_away(x/da), -127, 127); amax == 0 gives da = 0 and
// xq = 0. The per-32 activation scale is the one the q6_K rescale consumes
// ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2); the pages print no
// quantiser, so the division and the rounding are IEEE f32 and half-away.
// The kernels reach exactly those codes with one multiply by the reciprocal
// per element, falling back to the division next to rounding ties (qfast).
//
// HBM-bound: 4 bytes read and 3 written per element (plus 4 per 32 for da).
// Optionally (kSums) it also writes us = da * S per block, S the sum of the
// block's 32 codes (exact), the activation side of the q4_K min term
// ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2: the prepass packs
// the scale with the block sum), as the tf32 pair hi + lo the GEMM's min-term
// MMAs read: row n of us [N][q4_min_ld(K)] holds, per super-block b, the hi
// parts of its 8 blocks at 16 b .. 16 b + 7 and the lo parts at 16 b + 8 ..
// 16 b + 15, and 16 zeros after an odd super-block count.
#include "q6_quant.cuh"

namespace q6 {
namespace {

// Block c of token n: us = da * S as its hi/lo pair (and the padding of an
// odd super-block count, written by the last super-block's blocks).
__device__ __forceinline__ void store_us(float* __restrict__ us, int n, int K, int c, float v) {
  float hi, lo;
  tf32_split(v, hi, lo);
  const int b = c >> 3, i = c & 7, nsb = K >> 8;
  float* row = us + (size_t)n * q4_min_ld(K) + 16 * b;
  row[i] = hi;
  row[8 + i] = lo;
  if ((nsb & 1) && b == nsb - 1) {
    row[16 + i] = 0.0f;
    row[24 + i] = 0.0f;
  }
}

// Small inputs (a few tokens): each thread owns eight consecutive elements
// (two float4 loads issued together); four threads form one 32-element block
// and reduce amax with two xor-shuffles. K % 256 == 0 makes the group count a
// multiple of 32, so whole warps stay active.
template <bool kSums>
__global__ void __launch_bounds__(256) q8_quantize8_kernel(const float* __restrict__ X, int N, int K,
                                                           int ldx, int8_t* __restrict__ Xq,
                                                           float* __restrict__ da, int ldda,
                                                           __half* __restrict__ Xh,
                                                           float* __restrict__ us) {
  griddep_launch_dependents();  // the GEMM that reads these may start its prologue
  const long long per_row = K >> 3;  // eight-element groups per row
  const long long total = (long long)N * per_row;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += stride) {
    const int n = (int)(g / per_row);
    const int j = (int)(g - (long long)n * per_row);  // eight-element group in the row
    const float4* src = reinterpret_cast<const float4*>(X + (size_t)n * ldx) + 2 * j;
    const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
    float a = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                    fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const float d = __fdiv_rn(a, 127.0f);
    uint2 q8;
    uint4 h8;
    float sum = 0.0f;
    if (kSums) {
      quant8_sum(v0, v1, d, recip_or_zero(d), q8, h8, sum);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    } else {
      quant8(v0, v1, d, recip_or_zero(d), q8, h8);
    }
    if (Xq != nullptr) reinterpret_cast<uint2*>(Xq + (size_t)n * K)[j] = q8;
    if (Xh != nullptr) reinterpret_cast<uint4*>(Xh + (size_t)n * K)[j] = h8;
    if ((j & 3) == 0) {
      da[(size_t)(j >> 2) * ldda + n] = d;
      if (kSums) store_us(us, n, K, j >> 2, d * sum);
    }
  }
}

// Large inputs: each thread owns sixteen consecutive elements (four float4 loads issued
// together); two neighbouring lanes form one 32-element block and reduce amax
// with one xor-shuffle. Warps walk the rows' 16-element groups in lockstep
// (a lane past the end idles through the shuffle), so the shuffle always has
// the whole warp.
template <bool kSums>
__global__ void __launch_bounds__(256) q8_quantize_kernel(const float* __restrict__ X, int N, int K,
                                                          int ldx, int8_t* __restrict__ Xq,
                                                          float* __restrict__ da, int ldda,
                                                          __half* __restrict__ Xh,
                                                          float* __restrict__ us) {
  griddep_launch_dependents();  // the GEMM that reads these may start its prologue
  const long long per_row = K >> 4;                // sixteen-element groups per row (even)
  const long long total = (long long)N * per_row;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31;
  for (long long base = (long long)blockIdx.x * blockDim.x + (threadIdx.x - lane); base < total;
       base += stride) {
    const long long g = base + lane;
    const bool on = g < total;  // both lanes of a pair agree: total is even
    const int n = on ? (int)(g / per_row) : 0;
    const int j = on ? (int)(g - (long long)n * per_row) : 0;  // group in the row
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0, v2 = v0, v3 = v0;
    if (on) {
      const float4* src = reinterpret_cast<const float4*>(X + (size_t)n * ldx) + 4 * j;
      v0 = __ldg(src);
      v1 = __ldg(src + 1);
      v2 = __ldg(src + 2);
      v3 = __ldg(src + 3);
    }
    float a = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                    fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
    a = fmaxf(a, fmaxf(fmaxf(fmaxf(fabsf(v2.x), fabsf(v2.y)), fmaxf(fabsf(v2.z), fabsf(v2.w))),
                       fmaxf(fmaxf(fabsf(v3.x), fabsf(v3.y)), fmaxf(fabsf(v3.z), fabsf(v3.w)))));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    const float d = __fdiv_rn(a, 127.0f);
    const float r = recip_or_zero(d);
    uint2 qa, qb;
    uint4 ha, hb;
    float sum = 0.0f;
    if (kSums) {
      // every lane runs this (past the end on zeros), so the shuffle has the warp
      float s0, s1;
      quant8_sum(v0, v1, d, r, qa, ha, s0);
      quant8_sum(v2, v3, d, r, qb, hb, s1);
      sum = s0 + s1;
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    }
    if (!on) continue;
    if (!kSums) {
      quant8(v0, v1, d, r, qa, ha);
      quant8(v2, v3, d, r, qb, hb);
    }
    if (Xq != nullptr)
      reinterpret_cast<uint4*>(Xq + (size_t)n * K)[j] = make_uint4(qa.x, qa.y, qb.x, qb.y);
    if (Xh != nullptr) {
      uint4* h = reinterpret_cast<uint4*>(Xh + (size_t)n * K) + 2 * j;
      h[0] = ha;
      h[1] = hb;
    }
    if ((j & 1) == 0) {
      da[(size_t)(j >> 1) * ldda + n] = d;
      if (kSums) store_us(us, n, K, j >> 1, d * sum);
    }
  }
}

}  // namespace

// One pass. Prefill-sized inputs take the sixteen-element form with the grid
// capped at 32 blocks of 256 threads per SM (about two groups per thread),
// which measured fastest; a few tokens take the eight-element form, whose
// shorter per-thread chain and twice the threads finish sooner.
cudaError_t launch_quantize(const float* X, int N, int K, int ldx, int8_t* Xq, float* da, int ldda,
                            __half* Xh, float* us, cudaStream_t s) {
  const long long elems = (long long)N * K;
  if (elems < (1LL << 20)) {
    const long long blocks = (elems / 8 + 255) / 256;
    const unsigned grid = (unsigned)(blocks < 1 ? 1 : blocks);
    if (us)
      q8_quantize8_kernel<true><<<grid, 256, 0, s>>>(X, N, K, ldx, Xq, da, ldda, Xh, us);
    else
      q8_quantize8_kernel<false><<<grid, 256, 0, s>>>(X, N, K, ldx, Xq, da, ldda, Xh, nullptr);
    return cudaGetLastError();
  }
  long long blocks = (elems / 16 + 255) / 256;
  const long long cap = 152LL * 32;
  if (blocks > cap) blocks = cap;
  if (us)
    q8_quantize_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(X, N, K, ldx, Xq, da, ldda, Xh, us);
  else
    q8_quantize_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(X, N, K, ldx, Xq, da, ldda, Xh,
                                                               nullptr);
  return cudaGetLastError();
}

}  // namespace q6
