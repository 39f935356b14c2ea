// q6_K x int8 GEMM for one or two tokens: a weight-streaming kernel on the
// CUDA cores, bound by HBM (0.82 byte per weight: 210 bytes per 256 weights,
// plus the 16-byte padding of each d row). 3..16 tokens run on the
// tensor-core form in mmq_skinny_mma.cu. Measured on GB300 (ffn_down
// weights, us per launch, this form / the tensor form): 2 tokens 14.4 / 16.5,
// 3 tokens 18.1 / 16.5, 4 tokens 24.9 / 17.3; each token adds its own dp4a
// work, while the tensor form pays once for the weight conversion. The file
// also holds the fused kernel behind q6k_mmq_f32 (at its end), which
// quantises one or two f32 activation rows itself and then runs the same
// dot products.
//
// Math ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1-2.2): for each
// 16-element sub-block s the exact integer P = sum (q - 32) * xq is formed
// with dp4a, then Y += f32(d) * (da[chunk] * (sc[s] * P)) summed over the
// sub-blocks. The element map is the one of Sec. 3.2 (see pack.cu).
//
// Split form of the integer dot product: a code is q = lo + 16*hi (lo the
// ql nibble, hi the 2-bit qh field), so  sum (q - 32) x = sum (lo - 32) x +
// 16 * sum hi x.  lo - 32 as a signed byte is lo | 0xE0 (lo < 16), one LOP3
// per four codes; the qh fields are masked in place (a field at bits f, f+1
// gives 2^f * hi per byte) and the power of two is taken off the int32 sum
// with one shift. No code is ever assembled or re-centred, which halves the
// integer work per weight against building the 6-bit codes first.
//
// Row dot product: one warp per weight row; per iteration a warp covers four
// super-blocks, eight lanes per super-block. Lane (half, s4) of a super-block
// reads the 16 ql bytes at 16*s4 of its half and the 16 qh bytes at
// 16*(s4&1): the low nibbles give sub-block 8*half + s4, the high nibbles
// (same bytes) sub-block 8*half + s4 + 4; their 2-bit fields sit at bits
// 2*(s4>>1) and 2*(s4>>1) + 4 of the qh bytes.
//
// Streaming: warps stride over the rows, with the grid sized to one resident
// wave (4 warps per CTA, 64 registers, 8 CTAs per SM) so every warp starts at
// once and reads its row's qlh run in coalesced 768-byte steps; the loads of
// the next step are in flight while the current step is computed. Rows go to
// warps warp-index-major (rank = warp * gridDim + block), so consecutive
// rows land on consecutive CTAs and every SM gets the same number of rows
// to within one. Measured on GB300 and not kept: loading two to four steps
// ahead (more registers, fewer resident warps), a cp.async.bulk ring of whole
// rows, a per-warp cp.async ring in shared memory, L2 prefetches (per step,
// or of whole rows with cp.async.bulk.prefetch), a step-major order of the
// weight plane (no faster than row-major), one 8-byte load of the two
// sub-block scales with byte permutes (slower than two byte loads), more
// resident CTAs (10 or 12 per SM: 10.8 / 11.3 us against 9.2 for one token
// on 4096 x 11008; the 4096 rows already fit one wave of warps at 8).
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

// Exact P of a lane's two sub-blocks (split form, see the top of the file):
// pa = sum (q - 32) * xa over the low-nibble sub-block (qh field at bits
// fsh), pb the same over the high-nibble sub-block (field at fsh + 4), from
// its 16 ql bytes L, 16 qh bytes H and the 16 activation bytes of each.
__device__ __forceinline__ void dot_pair(const uint4 L, const uint4 H, int fsh, const uint4 xa,
                                         const uint4 xb, int& pa, int& pb) {
  const uint32_t Lw[4] = {L.x, L.y, L.z, L.w}, Hw[4] = {H.x, H.y, H.z, H.w};
  const uint32_t Xa[4] = {xa.x, xa.y, xa.z, xa.w}, Xb[4] = {xb.x, xb.y, xb.z, xb.w};
  const uint32_t mha = 0x03030303u << fsh, mhb = 0x30303030u << fsh;
  int la = 0, lb = 0, ha = 0, hb = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    la = __dp4a((int)((Lw[w] & 0x0F0F0F0Fu) | 0xE0E0E0E0u), (int)Xa[w], la);  // lo - 32
    lb = __dp4a((int)(((Lw[w] >> 4) & 0x0F0F0F0Fu) | 0xE0E0E0E0u), (int)Xb[w], lb);
    ha = __dp4a((int)(Hw[w] & mha), (int)Xa[w], ha);  // 2^fsh * hi: bytes <= 12
    hb = dp4a_us(Hw[w] & mhb, Xb[w], hb);             // 16 * 2^fsh * hi: bytes <= 192
  }
  pa = la + (ha << (4 - fsh));
  pb = lb + (hb >> fsh);  // an exact multiple of 2^fsh
}

// One lane's share of one step: sub-blocks sa = 8*half + s4 and sa + 4 of
// super-block sb, from its 16 ql bytes L and 16 qh bytes H, for every token.
// The codes Xq [N][K] and scales da come from global memory, or (kSmem) from
// the fused kernel's shared-memory copy.
template <bool kPartials, int kMaxN, bool kSmem = false>
__device__ __forceinline__ void step_dot(const uint4 L, const uint4 H, int sc_a, int sc_b,
                                         uint16_t dbits, int sb, int m, int M, int K,
                                         const int8_t* __restrict__ Xq,
                                         const float* __restrict__ da, int ldda, int N,
                                         int32_t* __restrict__ partials,
                                         int32_t* __restrict__ chunks, float (&acc)[kMaxN]) {
  const int lane = threadIdx.x & 31;
  const int half = (lane >> 2) & 1;
  const int s4 = lane & 3;
  const int fsh = 2 * (s4 >> 1);  // field of the low-nibble sub-block
  const int sa = 8 * half + s4;   // sub-block (0..15) of the low nibbles; sb_b = sa + 4
  const float d = __half2float(__ushort_as_half(dbits));
  const int ka = 256 * sb + 16 * sa;  // first element of sub-block a
  const int ca_blk = ka >> 5, cb_blk = (ka + 64) >> 5;
#pragma unroll
  for (int n = 0; n < kMaxN; ++n) {
    if (n < N) {
      const int8_t* xr = Xq + (size_t)n * K;
      uint4 xa, xb;
      float daa, dab;
      if (kSmem) {
        xa = *reinterpret_cast<const uint4*>(xr + ka);
        xb = *reinterpret_cast<const uint4*>(xr + ka + 64);
        daa = da[(size_t)ca_blk * ldda + n];
        dab = da[(size_t)cb_blk * ldda + n];
      } else {
        xa = __ldg(reinterpret_cast<const uint4*>(xr + ka));
        xb = __ldg(reinterpret_cast<const uint4*>(xr + ka + 64));
        daa = __ldg(da + (size_t)ca_blk * ldda + n);
        dab = __ldg(da + (size_t)cb_blk * ldda + n);
      }
      int pa, pb;
      dot_pair(L, H, fsh, xa, xb, pa, pb);
      // sc * P is an integer below 2^24 in magnitude: exact in f32
      acc[n] = fmaf(d, fmaf(dab, (float)(sc_b * pb), daa * (float)(sc_a * pa)), acc[n]);
      if (kPartials && partials) {
        // the sub-block partials P of this lane's two sub-blocks
        int32_t* pr = partials + ((size_t)n * M + m) * (size_t)(K / 16) + (size_t)sb * 16;
        pr[sa] = pa;
        pr[sa + 4] = pb;
      }
      if (kPartials && chunks) {
        // chunk sums sc*P over the chunk's two sub-blocks; the other
        // sub-block of each chunk is in lane ^ 1 (active together)
        const unsigned act = __activemask();
        const int ta = sc_a * pa, tb = sc_b * pb;
        const int sa2 = ta + __shfl_xor_sync(act, ta, 1);
        const int sb2 = tb + __shfl_xor_sync(act, tb, 1);
        if ((s4 & 1) == 0) {
          int32_t* pr = chunks + ((size_t)n * M + m) * (size_t)(K / 32) + (size_t)sb * 8;
          pr[sa >> 1] = sa2;
          pr[(sa + 4) >> 1] = sb2;
        }
      }
    }
  }
}

// Reduces each token's sum across the warp; lane 0 writes Y[n][m].
template <int kMaxN>
__device__ __forceinline__ void row_store(float (&acc)[kMaxN], int m, int N, float* __restrict__ Y,
                                          int ldy) {
  const int lane = threadIdx.x & 31;
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

// One step of a row as a lane holds it: 16 ql bytes, 16 qh bytes, the two
// sub-block scales and the super-block scale bits.
struct Step {
  uint4 L, H;
  int a, b;
  uint16_t d;
};

// The dot products of one weight row with the N <= kMaxN activation rows.
// Each step covers 4 super-blocks (768 bytes of codes per warp); the loads of
// step i + 1 are issued before the math of step i (a one-step software
// pipeline on two register buffers). The result is reduced across the warp
// and written by lane 0.
template <bool kPartials, int kMaxN, bool kSmem = false>
__device__ __forceinline__ void row_dot(const uint8_t* __restrict__ qlh_row,
                                        const int8_t* __restrict__ sc_row,
                                        const uint16_t* __restrict__ d_row, int m, int M, int K,
                                        const int8_t* __restrict__ Xq, const float* __restrict__ da,
                                        int ldda, int N, float* __restrict__ Y, int ldy,
                                        int32_t* __restrict__ partials,
                                        int32_t* __restrict__ chunks) {
  const int lane = threadIdx.x & 31;
  const int nsb = K / 256;
  const int sbi = lane >> 3;  // super-block within the step
  const int half = (lane >> 2) & 1;
  const int s4 = lane & 3;
  const int sa = 8 * half + s4;  // sub-block (0..15) of the low nibbles; sb_b = sa + 4

  float acc[kMaxN];
#pragma unroll
  for (int n = 0; n < kMaxN; ++n) acc[n] = 0.0f;

  auto load = [&](int sb, Step& r) {
    r.L = make_uint4(0, 0, 0, 0);
    r.H = r.L;
    r.a = r.b = 0;
    r.d = 0;
    if (sb < nsb) {
      const uint8_t* hb = qlh_row + (size_t)(2 * sb + half) * 96;
      r.L = __ldg(reinterpret_cast<const uint4*>(hb + 16 * s4));
      r.H = __ldg(reinterpret_cast<const uint4*>(hb + 64 + 16 * (s4 & 1)));
      r.a = __ldg(sc_row + 16 * sb + sa);
      r.b = __ldg(sc_row + 16 * sb + sa + 4);
      r.d = __ldg(d_row + sb);
    }
  };
  auto step = [&](int sb, const Step& r) {
    if (sb < nsb)
      step_dot<kPartials, kMaxN, kSmem>(r.L, r.H, r.a, r.b, r.d, sb, m, M, K, Xq, da, ldda, N,
                                        partials, chunks, acc);
  };
  // two step buffers used in turn, so no registers are copied between steps
  Step A, B;
  load(sbi, A);
  for (int g0 = 0; g0 < nsb; g0 += 8) {
    load(g0 + 4 + sbi, B);  // in flight during the step on A
    step(g0 + sbi, A);
    load(g0 + 8 + sbi, A);  // in flight during the step on B
    step(g0 + 4 + sbi, B);
  }
  row_store<kMaxN>(acc, m, N, Y, ldy);
}

// One warp per row, straight from global memory.
template <bool kPartials, int kMaxN>
__global__ void __launch_bounds__(kWarps * 32, kMinBlocks) mmq_skinny_kernel(
    const uint8_t* __restrict__ plane, PlaneGeom g, int M, int K, const int8_t* __restrict__ Xq,
    const float* __restrict__ da, int ldda, int N, float* __restrict__ Y, int ldy,
    int32_t* __restrict__ partials, int32_t* __restrict__ chunks) {
  // No early griddep_launch_dependents() here: with eight CTAs per SM the
  // next few-token kernel's CTAs become resident beside this grid's tail,
  // which measured slower (one token 9.1 -> 9.7 us, two 13.9 -> 14.8 us).
  griddep_wait();  // launched as a dependent launch: global memory from here on
  const int warps = (int)gridDim.x * kWarps;
  for (int m = (threadIdx.x >> 5) * (int)gridDim.x + blockIdx.x; m < M; m += warps)
    row_dot<kPartials, kMaxN>(
        plane + g.qlh_off + (size_t)m * g.qlh_row,
        reinterpret_cast<const int8_t*>(plane + g.sc_off) + (size_t)m * (K / 16),
        reinterpret_cast<const uint16_t*>(plane + g.d_off + (size_t)m * g.d_row), m, M, K, Xq, da,
        ldda, N, Y, ldy, partials, chunks);
}


// One or two tokens straight from f32 activations, in one launch: a CTA of
// 32 warps per SM, rows to warps as in mmq_skinny_kernel. Each warp requests
// the first two steps of its first row, the CTA then quantises the N rows of
// X into shared memory with the standalone quantiser's arithmetic
// (q6_quant.cuh: the same codes and scales as q8_quantize_act), and after one
// barrier the warps form the same dot products as mmq_skinny_kernel from the
// staged codes. Every CTA quantises all of X (N*K*4 bytes, from L2 after the
// first CTAs), so no CTA waits on another and nothing else is launched.
constexpr int kFusedWarps = 32;
// The quantiser loop below runs full-mask shuffles: every warp must run it
// whole and the four threads of a 32-element block must share a warp. Both
// hold because the CTA is whole warps and N * K / 8 is a multiple of 32
// (K % 256 == 0, checked in launch_fused).
static_assert((kFusedWarps * 32) % 32 == 0, "the fused CTA must be whole warps");

template <int kMaxN>
__global__ void __launch_bounds__(kFusedWarps * 32, 1) mmq_skinny_fused_kernel(
    const uint8_t* __restrict__ plane, PlaneGeom g, int M, int K, const float* __restrict__ X,
    int ldx, int N, float* __restrict__ Y, int ldy) {
  griddep_launch_dependents();  // the next dependent launch may start its prologue
  griddep_wait();  // launched as a dependent launch: global memory from here on
  extern __shared__ __align__(16) uint8_t fused_smem[];
  int8_t* xs = reinterpret_cast<int8_t*>(fused_smem);                     // codes [N][K]
  float* das = reinterpret_cast<float*>(fused_smem + (size_t)kMaxN * K);  // scales [K/32][kMaxN]
  const int lane = threadIdx.x & 31;
  const int nsb = K / 256;
  const int sbi = lane >> 3;
  const int half = (lane >> 2) & 1;
  const int s4 = lane & 3;
  const int sa = 8 * half + s4;
  const int warps = (int)gridDim.x * kFusedWarps;
  int m = (threadIdx.x >> 5) * (int)gridDim.x + blockIdx.x;

  const uint8_t* qlh_row = nullptr;
  const int8_t* sc_row = nullptr;
  const uint16_t* d_row = nullptr;
  auto row = [&](int mm) {
    qlh_row = plane + g.qlh_off + (size_t)mm * g.qlh_row;
    sc_row = reinterpret_cast<const int8_t*>(plane + g.sc_off) + (size_t)mm * (K / 16);
    d_row = reinterpret_cast<const uint16_t*>(plane + g.d_off + (size_t)mm * g.d_row);
  };
  auto load = [&](int sb, Step& r) {
    r.L = make_uint4(0, 0, 0, 0);
    r.H = r.L;
    r.a = r.b = 0;
    r.d = 0;
    if (sb < nsb) {
      const uint8_t* hb = qlh_row + (size_t)(2 * sb + half) * 96;
      r.L = __ldg(reinterpret_cast<const uint4*>(hb + 16 * s4));
      r.H = __ldg(reinterpret_cast<const uint4*>(hb + 64 + 16 * (s4 & 1)));
      r.a = __ldg(sc_row + 16 * sb + sa);
      r.b = __ldg(sc_row + 16 * sb + sa + 4);
      r.d = __ldg(d_row + sb);
    }
  };

  // the first row's first two steps are in flight while the codes are made
  Step A, B;
  if (m < M) {
    row(m);
    load(sbi, A);
    load(4 + sbi, B);
  }
  {
    // eight elements per thread, four threads per 32-element block (as the
    // standalone few-token quantiser); N*K/8 is a multiple of 32, so every
    // warp runs the shuffles whole. Without this loop the kernel takes 9.1
    // us for one token on the ffn_down weights (10.6 with it). Measured and
    // not kept: two groups per thread with their loads issued together
    // (spills: 11.3 us), the first two steps requested into L2 instead of
    // registers (10.8 us), sixteen elements per thread, one round for a
    // token (11.0 us; 10.7 with the L2 requests), and two or six further
    // steps requested into L2 before the quantisation (11.0 / 11.4 us).
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
      quant8(v0, v1, d, recip_or_zero(d), q8, h8);
      *reinterpret_cast<uint2*>(xs + (size_t)n * K + 8 * j) = q8;
      if ((j & 3) == 0) das[(j >> 2) * kMaxN + n] = d;
    }
  }
  __syncthreads();

  for (bool first = true; m < M; m += warps, first = false) {
    if (!first) {
      row(m);
      load(sbi, A);
      load(4 + sbi, B);
    }
    float acc[kMaxN];
#pragma unroll
    for (int n = 0; n < kMaxN; ++n) acc[n] = 0.0f;
    auto step = [&](int sb, const Step& r) {
      if (sb < nsb)
        step_dot<false, kMaxN, true>(r.L, r.H, r.a, r.b, r.d, sb, m, M, K, xs, das, kMaxN, N,
                                     nullptr, nullptr, acc);
    };
    // the first iteration of mmq_skinny_kernel's loop with both of its
    // loads already issued, then the same loop
    step(sbi, A);
    load(8 + sbi, A);
    step(4 + sbi, B);
    for (int g0 = 8; g0 < nsb; g0 += 8) {
      load(g0 + 4 + sbi, B);
      step(g0 + sbi, A);
      load(g0 + 8 + sbi, A);
      step(g0 + 4 + sbi, B);
    }
    row_store<kMaxN>(acc, m, N, Y, ldy);
  }
}

size_t fused_smem_bytes(int K, int kmax) { return (size_t)kmax * K + (size_t)(K / 32) * kmax * 4; }

// Two tokens of already quantised activations: the fused kernel's CTA shape
// and row loop, with the codes and scales copied into shared memory instead
// of formed there, so each token's activations are read from shared memory by
// every row instead of from L1. The dot products and their order are those of
// mmq_skinny_kernel, so Y is the same bit for bit.
__global__ void __launch_bounds__(kFusedWarps * 32, 1) mmq_skinny_staged_kernel(
    const uint8_t* __restrict__ plane, PlaneGeom g, int M, int K, const int8_t* __restrict__ Xq,
    const float* __restrict__ da, int ldda, int N, float* __restrict__ Y, int ldy) {
  constexpr int kMaxN = 2;
  griddep_launch_dependents();  // the next dependent launch may start its prologue
  griddep_wait();  // launched as a dependent launch: global memory from here on
  extern __shared__ __align__(16) uint8_t fused_smem[];
  int8_t* xs = reinterpret_cast<int8_t*>(fused_smem);                     // codes [N][K]
  float* das = reinterpret_cast<float*>(fused_smem + (size_t)kMaxN * K);  // scales [K/32][kMaxN]
  const int nc = K / 32;
  for (int i = threadIdx.x; i < N * (K / 16); i += blockDim.x) {
    const int n = i / (K / 16), j = i - n * (K / 16);
    reinterpret_cast<uint4*>(xs + (size_t)n * K)[j] =
        __ldg(reinterpret_cast<const uint4*>(Xq + (size_t)n * K) + j);
  }
  for (int i = threadIdx.x; i < N * nc; i += blockDim.x) {
    const int n = i / nc, c = i - n * nc;
    das[c * kMaxN + n] = __ldg(da + (size_t)c * ldda + n);
  }
  __syncthreads();
  const int warps = (int)gridDim.x * kFusedWarps;
  for (int m = (threadIdx.x >> 5) * (int)gridDim.x + blockIdx.x; m < M; m += warps)
    row_dot<false, kMaxN, true>(
        plane + g.qlh_off + (size_t)m * g.qlh_row,
        reinterpret_cast<const int8_t*>(plane + g.sc_off) + (size_t)m * (K / 16),
        reinterpret_cast<const uint16_t*>(plane + g.d_off + (size_t)m * g.d_row), m, M, K, xs,
        das, kMaxN, N, Y, ldy, nullptr, nullptr);
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
  return launch_pdl(mmq_skinny_fused_kernel<kMaxN>, dim3((unsigned)sms), dim3(kFusedWarps * 32),
                    fused_smem_bytes(K, kMaxN), s, plane, plane_geom(M, K), M, K, X, ldx, N, Y,
                    ldy);
}

}  // namespace

cudaError_t mmq_skinny_prepare() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(mmq_skinny_fused_kernel<1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemMax)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_fused_kernel<2>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemMax)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_staged_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemMax)))
    return e;
  return mmq_skinny_mma_prepare();
}

size_t mmq_skinny_fused_smem(int K, int N) { return fused_smem_bytes(K, N); }

cudaError_t launch_mmq_skinny_fused(const uint8_t* plane, int M, int K, const float* X, int ldx,
                                    int N, float* Y, int ldy, cudaStream_t s) {
  return N == 1 ? launch_fused<1>(plane, M, K, X, ldx, N, Y, ldy, s)
                : launch_fused<2>(plane, M, K, X, ldx, N, Y, ldy, s);
}

template <bool P, int kMaxN>
cudaError_t launch_bucket(const uint8_t* plane, const PlaneGeom& g, int M, int K, const int8_t* Xq,
                          const float* da, int ldda, int N, float* Y, int ldy, Debug dbg,
                          cudaStream_t s) {
  // one resident wave of blocks, warps striding over the rows (blocks with
  // no row return at once; the row order spreads the rows evenly over SMs)
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mmq_skinny_kernel<P, kMaxN>,
                                                         kWarps * 32, 0)))
    return e;
  const unsigned blocks = (unsigned)(sms * (per_sm > 0 ? per_sm : 1));
  return launch_pdl(mmq_skinny_kernel<P, kMaxN>, dim3(blocks), dim3(kWarps * 32), 0, s, plane, g,
                    M, K, Xq, da, ldda, N, Y, ldy, dbg.partials, dbg.chunk_sums);
}

cudaError_t launch_mmq_skinny(const uint8_t* plane, int M, int K, const int8_t* Xq, const float* da,
                              int ldda, int N, float* Y, int ldy, Debug dbg,
                              unsigned int* status, cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  // one or two tokens: the dp4a weight-streaming kernel (the debug partials
  // come from the same dot products); 3..16 tokens: the f16 tensor form with
  // TMA-staged weights (mmq_skinny_mma.cu), partials included
  if (N == 1)
    return dbg.any() ? launch_bucket<true, 1>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, dbg, s)
                     : launch_bucket<false, 1>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, dbg, s);
  if (N == 2 && !dbg.any() && fused_smem_bytes(K, 2) <= (size_t)kFusedSmemMax) {
    // two tokens: the activations staged in shared memory once per CTA (13.9
    // -> 13.3 us on 4096 x 11008)
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
    return launch_pdl(mmq_skinny_staged_kernel, dim3((unsigned)sms), dim3(kFusedWarps * 32),
                      fused_smem_bytes(K, 2), s, plane, g, M, K, Xq, da, ldda, N, Y, ldy);
  }
  if (N == 2)
    return dbg.any() ? launch_bucket<true, 2>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, dbg, s)
                     : launch_bucket<false, 2>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, dbg, s);
  return launch_mmq_skinny_mma(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s);
}

}  // namespace q6
