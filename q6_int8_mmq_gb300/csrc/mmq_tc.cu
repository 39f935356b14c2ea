// q6_K x int8 prefill GEMM on the 5th-generation tensor cores (sm_103a).
//
// What it computes ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1-2.4):
// for every token n, weight row m and 16-element sub-block s, the exact
// integer partial P = sum (q - 32) * xq, then
//     Y[n][m] += da[n][chunk] * (dsc[m][2c] * P_2c + dsc[m][2c+1] * P_2c+1)
// per 32-element chunk c, with dsc = f32(d) * sc (no dmin term). The pages run
// this as KSPLIT=2 pairs of int8 mma.sync m16n8k16 per chunk.
//
// sm_103a has no tcgen05 int8 MMA, so both operands are binary16 planes
// holding the small integers exactly (weights -32..31 from the unpack pass,
// activations -127..127 from the quantiser) and are multiplied by tcgen05.mma
// kind::f16 with f32 accumulation in TMEM: every sub-block sum is at most
// 16 * 32 * 127 = 65024 < 2^24, so the f32 partial is the integer partial
// exactly. One K=16 MMA per sub-block writes a fresh accumulator, so each
// sub-block keeps its own scale.
//
// CTA tile: 128 weight rows (MMA M, TMEM lanes) x 128 tokens (MMA N). Two
// shared-memory rings filled by TMA:
//   operand ring (5 stages x 64 of K): Xh and Wh tiles, 128 rows x 128 bytes
//          each, 128-byte swizzled; freed by the MMA (tcgen05.commit).
//   scale ring (6 stages x 128 of K): dsc [128 rows][8] and da [4][128];
//          freed by the epilogue.
// Warp roles (12 warps; warpgroup 0 gives registers to warpgroups 1-2):
//   0      TMA producer for both rings.
//   1      TMEM allocation (512 columns); lane 0 issues the MMAs: per chunk two
//          K=16 MMAs (sub-blocks 2c, 2c+1) into one of two TMEM buffers of
//          2 x 128 columns, then tcgen05.commit to that buffer's barrier.
//   2-3    idle (their registers go to the epilogue).
//   4-11   epilogue: warp w owns TMEM lanes 32(w%4).. and 64 token columns.
//          Per chunk it loads the two sub-block partials of its columns in
//          two halves of 32 columns, software-pipelined across chunks (the
//          load of one half overlaps the math of the other), releases the
//          TMEM buffer as soon as both halves are in registers, and
//          accumulates Y in registers: acc += da * (dsc0 * P0 + dsc1 * P1).
// Every mbarrier wait is bounded (see q6_internal.cuh).
#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int BM = 128, BN = 128;
constexpr int KB = 64, SB = 5;   // operand ring: K per stage, stages
constexpr int KS = 128, SS = 6;  // scale ring
constexpr int kThreads = 384;                 // launched with 168 registers per thread
constexpr int kCtlRegs = 40, kEpiRegs = 232;  // 128 * 40 + 256 * 232 == 384 * 168
static_assert(128 * kCtlRegs + 256 * kEpiRegs <= kThreads * 168, "register split");
constexpr int kEpiWarp0 = 4, kNumEpiWarps = 8;

constexpr int kOpX = 0, kOpW = BN * 128, kOpStage = kOpW + BM * 128;
constexpr int kScDsc = 0, kScDa = BM * 8 * 4, kScStage = kScDa + 4 * BN * 4;
constexpr int kRingS = SB * kOpStage;  // the scale ring follows the operand ring
constexpr int kRingsBytes = kRingS + SS * kScStage;
static_assert(kOpStage % 1024 == 0, "operand stages must keep 1024-byte alignment");
static_assert(kScStage % 128 == 0, "scale stages must keep 128-byte alignment");
constexpr int kTmemCols = 512;

enum : uint32_t { kSiteSEmpty = 1, kSiteSFull = 2, kSiteBEmpty = 3, kSiteBFull = 4,
                  kSiteTFull = 6, kSiteTEmpty = 7, kSiteDrain = 8 };

struct Bars {
  uint64_t s_full[SS], s_empty[SS];
  uint64_t b_full[SB], b_empty[SB];
  uint64_t tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kRingsBytes + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "shared memory budget");

// acc[j] += da[j] * (s0 * P0[j] + s1 * P1[j]) for 32 columns (16 pairs).
__device__ __forceinline__ void rescale32(float2 (&acc)[16], const uint32_t (&p0)[32],
                                          const uint32_t (&p1)[32], float2 s0v, float2 s1v,
                                          const float* __restrict__ dq) {
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 a4 = reinterpret_cast<const float4*>(dq)[v];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = 4 * v + 2 * e;
      float2 t = __fmul2_rn(s0v, make_float2(__uint_as_float(p0[j]), __uint_as_float(p0[j + 1])));
      t = __ffma2_rn(s1v, make_float2(__uint_as_float(p1[j]), __uint_as_float(p1[j + 1])), t);
      const float2 dav = e ? make_float2(a4.z, a4.w) : make_float2(a4.x, a4.y);
      acc[2 * v + e] = __ffma2_rn(dav, t, acc[2 * v + e]);
    }
  }
}

template <bool kPartials>
__device__ __forceinline__ void dump_partials(int32_t* __restrict__ partials, int M, int K, int N,
                                              int m, int n_first, size_t sub,
                                              const uint32_t (&p0)[32], const uint32_t (&p1)[32]) {
  if (kPartials) {
    if (m < M) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int n = n_first + j;
        if (n < N) {
          int32_t* pr = partials + ((size_t)n * M + m) * (size_t)(K / 16) + sub;
          pr[0] = (int32_t)__uint_as_float(p0[j]);
          pr[1] = (int32_t)__uint_as_float(p1[j]);
        }
      }
    }
    __syncwarp();
  }
}

template <bool kPartials>
__global__ void __launch_bounds__(kThreads, 1)
    mmq_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ CUtensorMap tmDa, const __grid_constant__ CUtensorMap tmDsc,
                  int M, int K, int N, float* __restrict__ Y, int ldy,
                  int32_t* __restrict__ partials, unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kRingsBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int ns = K / KS;   // scale-ring steps (half super-blocks)
  const int nb = K / KB;   // operand-ring steps
  const int nc = K / 32;   // chunks
  volatile int* abort_flag = &bars->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SS; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], kNumEpiWarps);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&bars->b_full[s], 1);
      mbar_init(&bars->b_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->tfull[b], 1);
      mbar_init(&bars->tempty[b], kNumEpiWarps);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmDa);
    tma_prefetch_desc(&tmDsc);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < kEpiWarp0) {
    // --------------------------------------------------- warpgroup 0: control --
    regs_dealloc<kCtlRegs>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer --
      if (lane == 0) {
        constexpr uint32_t kTxS = BM * 8 * 4 + 4 * BN * 4;
        constexpr uint32_t kTxB = (BN + BM) * 128;
        int s_issued = 0, b_issued = 0;
        bool ok = true;
        for (int ks = 0; ks < ns && ok; ++ks) {
          const int ss = ks % SS;
          ok = mbar_wait_bounded(&bars->s_empty[ss], ((ks / SS) & 1) ^ 1, abort_flag, status,
                                 kSiteSEmpty);
          if (!ok) break;
          uint8_t* st = smem + kRingS + ss * kScStage;
          mbar_arrive_expect_tx(&bars->s_full[ss], kTxS);
          tma_load_2d(st + kScDsc, &tmDsc, &bars->s_full[ss], ks * 8, m0);
          tma_load_2d(st + kScDa, &tmDa, &bars->s_full[ss], n0, ks * 4);
          s_issued = ks + 1;
          for (int h = 0; h < 2; ++h) {
            const int kb = 2 * ks + h, sb = kb % SB;
            ok = mbar_wait_bounded(&bars->b_empty[sb], ((kb / SB) & 1) ^ 1, abort_flag, status,
                                   kSiteBEmpty);
            if (!ok) break;
            uint8_t* bt = smem + sb * kOpStage;
            mbar_arrive_expect_tx(&bars->b_full[sb], kTxB);
            tma_load_2d(bt + kOpX, &tmX, &bars->b_full[sb], kb * KB, n0);
            tma_load_2d(bt + kOpW, &tmW, &bars->b_full[sb], kb * KB, m0);
            b_issued = kb + 1;
          }
        }
        if (!ok) {
          // Let copies already issued land before the CTA exits.
          volatile int no_abort = 0;
          for (int k = (s_issued > SS ? s_issued - SS : 0); k < s_issued; ++k)
            mbar_wait_bounded(&bars->s_full[k % SS], (k / SS) & 1, &no_abort, status, kSiteSFull);
          for (int k = (b_issued > SB ? b_issued - SB : 0); k < b_issued; ++k)
            mbar_wait_bounded(&bars->b_full[k % SB], (k / SB) & 1, &no_abort, status, kSiteBFull);
        }
      }
    } else if (warp == 1) {
      // --------------------------------------------------------------- MMA --
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
        int cc = 0;
        bool ok = true;
        for (int kb = 0; kb < nb && ok; ++kb) {
          const int sb = kb % SB;
          if (!mbar_wait_bounded(&bars->b_full[sb], (kb / SB) & 1, abort_flag, status, kSiteBFull))
            break;
          tc_fence_after();
          const uint8_t* bt = smem + sb * kOpStage;
          const uint32_t w_base = smem_u32(bt + kOpW), x_base = smem_u32(bt + kOpX);
          for (int q = 0; q < 2; ++q, ++cc) {
            const int b = cc & 1;
            const uint32_t use = (uint32_t)(cc >> 1);
            if (!mbar_wait_bounded(&bars->tempty[b], (use & 1) ^ 1, abort_flag, status,
                                   kSiteTEmpty)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t koff = (uint32_t)((2 * q + h) * 32);  // sub-block within the stage
              umma_f16(tmem + (uint32_t)(b * 256 + h * 128), sw128_kmajor_desc(w_base + koff),
                       sw128_kmajor_desc(x_base + koff), idesc, 0u);
            }
            umma_commit(&bars->tfull[b]);
          }
          if (ok) umma_commit(&bars->b_empty[sb]);
        }
        // Every MMA must be finished before TMEM is released.
        umma_commit(&bars->drain);
        volatile int no_abort = 0;
        mbar_wait_bounded(&bars->drain, 0, &no_abort, status, kSiteDrain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ warpgroups 1-2: epilogue --
    regs_alloc<kEpiRegs>();
    const int ew = warp - kEpiWarp0;  // 0..7
    const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
    const int colh = ew >> 2;         // token columns 64*colh .. +63
    const int row = 32 * quarter + lane;
    const int m = m0 + row;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(64 * colh);
    float2 accA[16], accB[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) accA[j] = accB[j] = make_float2(0.0f, 0.0f);
    uint32_t pA0[32], pA1[32], pB0[32], pB1[32];
    bool ok = mbar_wait_warp(&bars->tfull[0], 0, abort_flag, status, kSiteTFull);
    if (ok) {
      tc_fence_after();
      tmem_ld32(lane_addr, pA0);
      tmem_ld32(lane_addr + 128u, pA1);
      tmem_wait_ld2(pA0, pA1);
    }
    // Outer loop: one scale stage (four 32-element chunks); inner loop unrolled,
    // so the TMEM buffer (chunk & 1), the barrier parities and the scale
    // selection are compile-time constants.
    for (int ks = 0; ks < ns && ok; ++ks) {
      const int ss = ks % SS;
      if (!mbar_wait_warp(&bars->s_full[ss], (ks / SS) & 1, abort_flag, status, kSiteSFull)) break;
      const uint8_t* st = smem + kRingS + ss * kScStage;
      const float* sda = reinterpret_cast<const float*>(st + kScDa) + 64 * colh;
      const float4 d0 = reinterpret_cast<const float4*>(st + kScDsc + row * 32)[0];
      const float4 d1 = reinterpret_cast<const float4*>(st + kScDsc + row * 32)[1];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = 4 * ks + q;
        const uint32_t b = (uint32_t)(q & 1);
        const float s0 = q == 0 ? d0.x : q == 1 ? d0.z : q == 2 ? d1.x : d1.z;
        const float s1 = q == 0 ? d0.y : q == 1 ? d0.w : q == 2 ? d1.y : d1.w;
        const float2 s0v = make_float2(s0, s0), s1v = make_float2(s1, s1);
        const float* dq = sda + q * 128;
        // second half of this chunk in flight while the first half is scaled
        tmem_ld32(lane_addr + b * 256u + 32u, pB0);
        tmem_ld32(lane_addr + b * 256u + 160u, pB1);
        rescale32(accA, pA0, pA1, s0v, s1v, dq);
        dump_partials<kPartials>(partials, M, K, N, m, n0 + 64 * colh, (size_t)c * 2, pA0, pA1);
        tmem_wait_ld2(pB0, pB1);
        // both halves are in registers: the TMEM buffer can take chunk c + 2
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tempty[b]);
        // First half of the next chunk in flight while the second half is
        // scaled. The loads are unconditional (after the last chunk they
        // re-read the other buffer, which no MMA writes any more): keeping the
        // async loads and their wait out of branches lets them overlap the math.
        if ((q < 3 || c + 1 < nc) &&
            !mbar_wait_warp(&bars->tfull[b ^ 1u], (uint32_t)(((q + 1) >> 1) & 1), abort_flag, status,
                            kSiteTFull))
          ok = false;
        tc_fence_after();
        tmem_ld32(lane_addr + (b ^ 1u) * 256u, pA0);
        tmem_ld32(lane_addr + (b ^ 1u) * 256u + 128u, pA1);
        rescale32(accB, pB0, pB1, s0v, s1v, dq + 32);
        dump_partials<kPartials>(partials, M, K, N, m, n0 + 64 * colh + 32, (size_t)c * 2, pB0, pB1);
        tmem_wait_ld2(pA0, pA1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_empty[ss]);
    }
    if (m < M) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = n0 + 64 * colh + 2 * j;
        if (n < N) Y[(size_t)n * ldy + m] = accA[j].x;
        if (n + 1 < N) Y[(size_t)(n + 1) * ldy + m] = accA[j].y;
        if (n + 32 < N) Y[(size_t)(n + 32) * ldy + m] = accB[j].x;
        if (n + 33 < N) Y[(size_t)(n + 33) * ldy + m] = accB[j].y;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool P>
cudaError_t launch_one(const TcMaps& maps, int M, int K, int N, float* Y, int ldy, int32_t* partials,
                       unsigned int* status, cudaStream_t s) {
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  mmq_tc_kernel<P><<<grid, kThreads, kSmemBytes, s>>>(maps.x, maps.w, maps.da, maps.dsc, M, K, N, Y,
                                                     ldy, partials, status);
  return cudaGetLastError();
}

}  // namespace

size_t mmq_tc_smem_bytes() { return kSmemBytes; }

// Raises the dynamic shared-memory limit of both instantiations; once per device.
cudaError_t mmq_tc_prepare() {
  cudaError_t e = cudaFuncSetAttribute(mmq_tc_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mmq_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmemBytes);
}

cudaError_t launch_mmq_tc(const TcMaps& maps, int M, int K, int N, float* Y, int ldy,
                          int32_t* partials, unsigned int* status, cudaStream_t s) {
  return partials ? launch_one<true>(maps, M, K, N, Y, ldy, partials, status, s)
                  : launch_one<false>(maps, M, K, N, Y, ldy, nullptr, status, s);
}

}  // namespace q6
