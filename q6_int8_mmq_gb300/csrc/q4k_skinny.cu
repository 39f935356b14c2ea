// q4_K x int8 GEMM for a few tokens: a weight-streaming kernel on the CUDA
// cores, bound by HBM (0.59 byte per weight: the 0.5-byte nibbles, the 6-bit
// scale and min bytes of each 32-element sub-block and the f32 (d, dmin) of
// each super-block).
//
// Math ("r18: Load-time B pre-expansion", Sec. 1 and 3.2; "r38 -- q6_K
// BT-style raw-byte mma kernel", Sec. 2.2): for sub-block c of token n,
//   Y += da[c] * d * sc[c] * P  -  dmin * m[c] * us[c],
// P = sum over the 32 elements of q * xq (q the raw nibble 0..15, exact
// with dp4a), us = da * (sum of the block's codes) from the quantiser.
//
// Row dot product: one warp per weight row; per step a warp covers four
// super-blocks, eight lanes per super-block. Lane (p, h) of a super-block
// reads the 16 nibble bytes at 32 p + 16 h of its 128: their low nibbles
// are elements 16 h .. 16 h + 15 of sub-block 2 p and their high nibbles the
// same elements of sub-block 2 p + 1, so each lane forms half of two
// sub-blocks' P with four dp4a each; the lane with h = 0 also subtracts the
// two sub-blocks' min terms. The loads of the next step are in flight while
// a step is computed (two register buffers used in turn), warps stride over
// the rows with the grid sized to one resident wave. Each token repeats its
// dot products and re-reads its activations for every row (from L1), so the
// time grows by about 6 us a token on 4096 x 11008 weights; beyond
// Q6_Q4K_DP4A_MAX_N tokens the warp-level f16 MMA kernel, which shares each
// activation fragment across 16 rows, is faster. The file also holds the
// fused kernel behind q4k_mmq_f32 (at its end), which quantises one or two
// f32 activation rows itself and then runs the same row dot products.
#include "q6_quant.cuh"

namespace q6 {
namespace {

constexpr int kWarps = 4;      // warps per CTA
constexpr int kMinBlocks = 8;  // resident CTAs per SM (64 registers per thread)

// c + sum over the four byte pairs of a (unsigned) times b (signed).
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One step of a row as a lane holds it: 16 nibble bytes, the two sub-blocks'
// scale and min bytes, and the super-block's (d, dmin).
struct Step {
  uint4 L;
  uint32_t sc, mn;  // bytes of sub-blocks 2p, 2p + 1 in bits 0-7, 8-15
  float2 dd;
};

// The dot products of weight row m with the N <= kMaxN activation rows,
// reduced across the warp; lane 0 writes Y[n][m]. The codes Xq [N][K] and
// scales da [K/32][ldda] come from global memory with the block sums us as the
// quantiser's hi/lo pairs [N][ldus], or (kSmem) from the fused kernel's
// shared-memory copy, whose block sums are us itself [N][K/32].
template <bool kPartials, int kMaxN, bool kSmem>
__device__ __forceinline__ void q4_row(const uint8_t* __restrict__ plane, const Q4Geom& g, int m,
                                       int M, int K, const int8_t* __restrict__ Xq,
                                       const float* __restrict__ da, int ldda,
                                       const float* __restrict__ us, int N,
                                       float* __restrict__ Y, int ldy,
                                       int32_t* __restrict__ partials) {
  const int lane = threadIdx.x & 31;
  const int nsb = K / 256, nc = K / 32, ldus = q4_min_ld(K);
  const int sbi = lane >> 3;            // super-block within the step
  const int p = (lane >> 1) & 3, h = lane & 1;
  const uint8_t* qs = plane + g.qs_off + (size_t)m * (K / 2);
  const uint8_t* scr = plane + g.sc_off + (size_t)m * nc;
  const uint8_t* mnr = plane + g.mn_off + (size_t)m * nc;
  const float2* ddr = reinterpret_cast<const float2*>(plane + g.ddm_off) + (size_t)m * nsb;
  float acc[kMaxN];
#pragma unroll
  for (int n = 0; n < kMaxN; ++n) acc[n] = 0.0f;

  auto load = [&](int sb, Step& r) {
    r.L = make_uint4(0, 0, 0, 0);
    r.sc = r.mn = 0;
    r.dd = make_float2(0.0f, 0.0f);
    if (sb < nsb) {
      r.L = __ldg(reinterpret_cast<const uint4*>(qs + (size_t)sb * 128 + 32 * p + 16 * h));
      r.sc = __ldg(reinterpret_cast<const uint16_t*>(scr + 8 * sb + 2 * p));
      r.mn = __ldg(reinterpret_cast<const uint16_t*>(mnr + 8 * sb + 2 * p));
      r.dd = __ldg(ddr + sb);
    }
  };
  auto step = [&](int sb, const Step& r) {
    // lanes of a super-block past the end compute nothing but still take
    // the (full-warp) shuffles of the debug partials
    const bool valid = sb < nsb;
    const int ca = 8 * sb + 2 * p;  // sub-blocks ca (low nibbles) and ca + 1 (high)
    const uint32_t Lw[4] = {r.L.x, r.L.y, r.L.z, r.L.w};
    const float sca = (float)(r.sc & 0xFF), scb = (float)(r.sc >> 8);
    const float mna = (float)(r.mn & 0xFF), mnb = (float)(r.mn >> 8);
#pragma unroll
    for (int n = 0; n < kMaxN; ++n) {
      if (n < N) {
        int pa = 0, pb = 0;
        if (valid) {
          const int8_t* xr = Xq + (size_t)n * K + 32 * ca + 16 * h;
          uint4 xa, xb;
          float daa, dab;
          if (kSmem) {
            xa = *reinterpret_cast<const uint4*>(xr);
            xb = *reinterpret_cast<const uint4*>(xr + 32);
            daa = da[(size_t)ca * ldda + n];
            dab = da[(size_t)(ca + 1) * ldda + n];
          } else {
            xa = __ldg(reinterpret_cast<const uint4*>(xr));
            xb = __ldg(reinterpret_cast<const uint4*>(xr + 32));
            daa = __ldg(da + (size_t)ca * ldda + n);
            dab = __ldg(da + (size_t)(ca + 1) * ldda + n);
          }
          const uint32_t Xa[4] = {xa.x, xa.y, xa.z, xa.w}, Xb[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            pa = dp4a_us(Lw[w] & 0x0F0F0F0Fu, Xa[w], pa);
            pb = dp4a_us((Lw[w] >> 4) & 0x0F0F0F0Fu, Xb[w], pb);
          }
          // sc * P is an integer below 2^21 in magnitude: exact in f32
          float v = r.dd.x * fmaf(dab, scb * (float)pb, daa * (sca * (float)pa));
          if (h == 0) {
            float ua, ub;
            if (kSmem) {
              ua = us[(size_t)n * nc + ca];
              ub = us[(size_t)n * nc + ca + 1];
            } else {
              // us of the two sub-blocks from their exact hi/lo pairs (the
              // two hi parts, and the two lo parts, are adjacent)
              const float* ur = us + (size_t)n * ldus + 16 * sb + 2 * p;
              const float2 hi = __ldg(reinterpret_cast<const float2*>(ur));
              const float2 lo = __ldg(reinterpret_cast<const float2*>(ur + 8));
              ua = hi.x + lo.x;
              ub = hi.y + lo.y;
            }
            v = fmaf(-r.dd.y, fmaf(mnb, ub, mna * ua), v);
          }
          acc[n] += v;
        }
        if (kPartials && partials) {
          // P of the two sub-blocks: this lane's half and its neighbour's
          const int fa = pa + __shfl_xor_sync(0xffffffffu, pa, 1);
          const int fb = pb + __shfl_xor_sync(0xffffffffu, pb, 1);
          if (valid && h == 0) {
            int32_t* pr = partials + ((size_t)n * M + m) * (size_t)nc + ca;
            pr[0] = fa;
            pr[1] = fb;
          }
        }
      }
    }
  };
  Step A, B;
  load(sbi, A);
  for (int g0 = 0; g0 < nsb; g0 += 8) {
    load(g0 + 4 + sbi, B);  // in flight during the step on A
    step(g0 + sbi, A);
    load(g0 + 8 + sbi, A);  // in flight during the step on B
    step(g0 + 4 + sbi, B);
  }
#pragma unroll
  for (int n = 0; n < kMaxN; ++n) {
    if (n < N) {
      float v = acc[n];
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) Y[(size_t)n * ldy + m] = v;
    }
  }
}

template <bool kPartials, int kMaxN>
__global__ void __launch_bounds__(kWarps * 32, kMinBlocks) q4k_skinny_kernel(
    const uint8_t* __restrict__ plane, Q4Geom g, int M, int K, const int8_t* __restrict__ Xq,
    const float* __restrict__ da, int ldda, const float* __restrict__ us, int N,
    float* __restrict__ Y, int ldy, int32_t* __restrict__ partials) {
  // No early griddep_launch_dependents() here: with eight CTAs per SM the
  // next few-token kernel's CTAs become resident beside this grid's tail,
  // which measured slower (one token 9.1 -> 9.7 us, two 13.9 -> 14.8 us).
  griddep_wait();  // launched as a dependent launch: global memory from here on
  const int warps = (int)gridDim.x * kWarps;
  for (int m = (threadIdx.x >> 5) * (int)gridDim.x + blockIdx.x; m < M; m += warps)
    q4_row<kPartials, kMaxN, false>(plane, g, m, M, K, Xq, da, ldda, us, N, Y, ldy, partials);
}

template <bool P, int kMaxN>
cudaError_t launch_bucket(const uint8_t* plane, const Q4Geom& g, int M, int K, const int8_t* Xq,
                          const float* da, int ldda, const float* us, int N, float* Y, int ldy,
                          int32_t* partials, cudaStream_t s) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q4k_skinny_kernel<P, kMaxN>,
                                                         kWarps * 32, 0)))
    return e;
  const unsigned blocks = (unsigned)(sms * (per_sm > 0 ? per_sm : 1));
  return launch_pdl(q4k_skinny_kernel<P, kMaxN>, dim3(blocks), dim3(kWarps * 32), 0, s, plane, g,
                    M, K, Xq, da, ldda, us, N, Y, ldy, partials);
}

template <int kMaxN>
cudaError_t launch_n(const uint8_t* plane, const Q4Geom& g, int M, int K, const int8_t* Xq,
                     const float* da, int ldda, const float* us, int N, float* Y, int ldy,
                     int32_t* partials, cudaStream_t s) {
  return partials ? launch_bucket<true, kMaxN>(plane, g, M, K, Xq, da, ldda, us, N, Y, ldy,
                                               partials, s)
                  : launch_bucket<false, kMaxN>(plane, g, M, K, Xq, da, ldda, us, N, Y, ldy,
                                                nullptr, s);
}

// One or two tokens straight from f32 activations, in one launch (the q4_K
// form of mmq_skinny_fused_kernel): a CTA of 32 warps per SM, rows to warps as
// in q4k_skinny_kernel. The CTA quantises the N rows of X into shared memory
// with the standalone quantiser's arithmetic (q6_quant.cuh: the codes, scales
// and block sums of q8_quantize_act_sums; us = da * S kept as the f32 value
// that the quantiser's hi/lo pair holds exactly), and after one barrier the
// warps form the same dot products from the staged codes, so Y is bit for bit
// that of the two calls. Every CTA quantises all of X, so no CTA waits on
// another and nothing else is launched.
constexpr int kFusedWarps = 32;
// The quantiser loop's full-mask shuffles need whole warps and the four
// threads of a 32-element block in one warp: the CTA is whole warps and
// N * K / 8 is a multiple of 32 (K % 256 == 0, checked in launch_fused).
static_assert((kFusedWarps * 32) % 32 == 0, "the fused CTA must be whole warps");

size_t fused_smem_bytes(int K, int kmax) {  // codes [kmax][K], da [K/32][kmax], us [kmax][K/32]
  return (size_t)kmax * K + 2 * (size_t)(K / 32) * kmax * 4;
}

template <int kMaxN>
__global__ void __launch_bounds__(kFusedWarps * 32, 1) q4k_skinny_fused_kernel(
    const uint8_t* __restrict__ plane, Q4Geom g, int M, int K, const float* __restrict__ X,
    int ldx, int N, float* __restrict__ Y, int ldy) {
  griddep_launch_dependents();  // the next dependent launch may start its prologue
  griddep_wait();  // launched as a dependent launch: global memory from here on
  extern __shared__ __align__(16) uint8_t fused_smem[];
  const int nc = K / 32;
  int8_t* xs = reinterpret_cast<int8_t*>(fused_smem);                     // codes [N][K]
  float* das = reinterpret_cast<float*>(fused_smem + (size_t)kMaxN * K);  // da [K/32][kMaxN]
  float* uss = das + (size_t)nc * kMaxN;                                  // us [N][K/32]
  {
    // eight elements per thread, four threads per 32-element block (as the
    // standalone few-token quantiser); N*K/8 is a multiple of 32, so every
    // warp runs the shuffles whole
    const int per_row = K >> 3;
    const int total = N * per_row;
    for (int gi = threadIdx.x; gi < total; gi += blockDim.x) {
      const int n = gi / per_row;
      const int j = gi - n * per_row;
      const float4* src = reinterpret_cast<const float4*>(X + (size_t)n * ldx) + 2 * j;
      const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
      float a = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                      fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
      const float d = __fdiv_rn(a, 127.0f);
      uint2 q8;
      uint4 h8;
      float sum;
      quant8_sum(v0, v1, d, recip_or_zero(d), q8, h8, sum);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      *reinterpret_cast<uint2*>(xs + (size_t)n * K + 8 * j) = q8;
      if ((j & 3) == 0) {
        das[(j >> 2) * kMaxN + n] = d;
        uss[(size_t)n * nc + (j >> 2)] = d * sum;
      }
    }
  }
  __syncthreads();
  const int warps = (int)gridDim.x * kFusedWarps;
  for (int m = (threadIdx.x >> 5) * (int)gridDim.x + blockIdx.x; m < M; m += warps)
    q4_row<false, kMaxN, true>(plane, g, m, M, K, xs, das, kMaxN, uss, N, Y, ldy, nullptr);
}

template <int kMaxN>
cudaError_t launch_fused(const uint8_t* plane, int M, int K, const float* X, int ldx, int N,
                         float* Y, int ldy, cudaStream_t s) {
  // the quantiser's full-mask shuffles need K / 8 to be a multiple of 32
  if (K % 256 != 0) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  return launch_pdl(q4k_skinny_fused_kernel<kMaxN>, dim3((unsigned)sms), dim3(kFusedWarps * 32),
                    fused_smem_bytes(K, kMaxN), s, plane, q4_geom(M, K), M, K, X, ldx, N, Y,
                    ldy);
}

// Two tokens of already quantised activations: the fused kernel's CTA shape
// and row loop, with the codes, scales and block sums copied into shared
// memory instead of formed there (us as the f32 sum of its hi/lo pair, which
// is exact). Each token's activations are then read from shared memory by
// every row instead of from L1, and the block sum of a sub-block is one word
// instead of two 8-byte pairs; the dot products and their order are those of
// q4k_skinny_kernel, so Y is the same bit for bit.
__global__ void __launch_bounds__(kFusedWarps * 32, 1) q4k_skinny_staged_kernel(
    const uint8_t* __restrict__ plane, Q4Geom g, int M, int K, const int8_t* __restrict__ Xq,
    const float* __restrict__ da, int ldda, const float* __restrict__ us, int N,
    float* __restrict__ Y, int ldy) {
  constexpr int kMaxN = 2;
  griddep_launch_dependents();  // the next dependent launch may start its prologue
  griddep_wait();  // launched as a dependent launch: global memory from here on
  extern __shared__ __align__(16) uint8_t fused_smem[];
  const int nc = K / 32, ldus = q4_min_ld(K);
  int8_t* xs = reinterpret_cast<int8_t*>(fused_smem);                     // codes [N][K]
  float* das = reinterpret_cast<float*>(fused_smem + (size_t)kMaxN * K);  // da [K/32][kMaxN]
  float* uss = das + (size_t)nc * kMaxN;                                  // us [N][K/32]
  for (int i = threadIdx.x; i < N * (K / 16); i += blockDim.x) {
    const int n = i / (K / 16), j = i - n * (K / 16);
    reinterpret_cast<uint4*>(xs + (size_t)n * K)[j] =
        __ldg(reinterpret_cast<const uint4*>(Xq + (size_t)n * K) + j);
  }
  for (int i = threadIdx.x; i < N * nc; i += blockDim.x) {
    const int n = i / nc, c = i - n * nc;
    const float* ur = us + (size_t)n * ldus + 16 * (c >> 3) + (c & 7);
    das[c * kMaxN + n] = __ldg(da + (size_t)c * ldda + n);
    uss[(size_t)n * nc + c] = __ldg(ur) + __ldg(ur + 8);
  }
  __syncthreads();
  const int warps = (int)gridDim.x * kFusedWarps;
  for (int m = (threadIdx.x >> 5) * (int)gridDim.x + blockIdx.x; m < M; m += warps)
    q4_row<false, kMaxN, true>(plane, g, m, M, K, xs, das, kMaxN, uss, N, Y, ldy, nullptr);
}

}  // namespace

cudaError_t q4k_skinny_prepare() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(q4k_skinny_fused_kernel<1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemMax)) ||
      (e = cudaFuncSetAttribute(q4k_skinny_staged_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemMax)))
    return e;
  return cudaFuncSetAttribute(q4k_skinny_fused_kernel<2>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemMax);
}

size_t q4k_skinny_fused_smem(int K, int N) { return fused_smem_bytes(K, N); }

cudaError_t launch_q4k_skinny_fused(const uint8_t* plane, int M, int K, const float* X, int ldx,
                                    int N, float* Y, int ldy, cudaStream_t s) {
  return N == 1 ? launch_fused<1>(plane, M, K, X, ldx, N, Y, ldy, s)
                : launch_fused<2>(plane, M, K, X, ldx, N, Y, ldy, s);
}

cudaError_t launch_q4k_skinny(const uint8_t* plane, int M, int K, const int8_t* Xq,
                              const float* da, int ldda, const float* us, int N, float* Y,
                              int ldy, int32_t* partials, cudaStream_t s) {
  const Q4Geom g = q4_geom(M, K);
  if (N <= 1) return launch_n<1>(plane, g, M, K, Xq, da, ldda, us, N, Y, ldy, partials, s);
  if (N == 2 && !partials && fused_smem_bytes(K, 2) <= (size_t)kFusedSmemMax) {
    // two tokens: the activations staged in shared memory once per CTA
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
    return launch_pdl(q4k_skinny_staged_kernel, dim3((unsigned)sms), dim3(kFusedWarps * 32),
                      fused_smem_bytes(K, 2), s, plane, g, M, K, Xq, da, ldda, us, N, Y, ldy);
  }
  if (N <= 2) return launch_n<2>(plane, g, M, K, Xq, da, ldda, us, N, Y, ldy, partials, s);
  if (N <= 4) return launch_n<4>(plane, g, M, K, Xq, da, ldda, us, N, Y, ldy, partials, s);
  static_assert(Q6_Q4K_DP4A_MAX_N <= 8, "the largest token bucket holds 8 tokens");
  return launch_n<8>(plane, g, M, K, Xq, da, ldda, us, N, Y, ldy, partials, s);
}

}  // namespace q6
