// q6_K x int8 prefill GEMM on the 5th-generation tensor cores (sm_103a).
//
// What it computes ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1-2.4):
// for every token n, weight row m and 16-element sub-block s, the exact
// integer partial P = sum (q - 32) * xq, then
//     Y[n][m] += da[n][chunk] * (dsc[m][2c] * P_2c + dsc[m][2c+1] * P_2c+1)
// per 32-element chunk c, with dsc = f32(d) * sc (no dmin term). The pages run
// this as KSPLIT=2 pairs of int8 mma.sync m16n8k16 per chunk.
//
// Here, sm_103a offers no tcgen05 int8 MMA, so both operands are staged as
// binary16 holding the small integers exactly (weights -32..31, activations
// -127..127) and multiplied by tcgen05.mma kind::f16 with f32 accumulation in
// TMEM: every sub-block sum is at most 16 * 32 * 127 = 65024 < 2^24, so the
// f32 partial equals the integer partial exactly. One K=16 MMA per sub-block
// writes a fresh accumulator, so each sub-block keeps its own scale.
//
// CTA tile: 128 weight rows (MMA M, TMEM lanes) x 128 tokens (MMA N), K staged
// 128 at a time (one half super-block) in a 2-stage mbarrier ring.
//   warp 0      TMA producer: Xh tile (two 64-wide 128B-swizzled boxes), the
//               weight source (96-byte qlh rows, or 128-byte W_exp rows), the
//               da slice [4 chunks][128 tokens], the dsc slice [128 rows][8].
//   warp 1      allocates 512 TMEM columns; lane 0 issues the MMAs: per chunk
//               two MMAs (sub-blocks 2c, 2c+1) into one of two TMEM buffers of
//               2 x 128 columns, then tcgen05.commit to the buffer's barrier.
//   warps 2-5   unpack the weight source into the binary16 operand tile in the
//               128B-swizzled K-major layout (raw: ql nibble | qh field << 4,
//               minus 32; W_exp: int8 -> f16), fence to the async proxy.
//   warps 6-13  epilogue: tcgen05.ld both sub-block partials of a chunk, scale
//               with dsc (per row, this thread's lane) and da (per column),
//               accumulate Y in registers, release the TMEM buffer.
// Every mbarrier wait is bounded (see q6_internal.cuh).
#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int BM = 128, BN = 128, BK = 128, STAGES = 2;
constexpr int kThreads = 448;
constexpr int kConvWarp0 = 2, kNumConvWarps = 4;
constexpr int kEpiWarp0 = 6, kNumEpiWarps = 8;
constexpr int kConvThreads = kNumConvWarps * 32;

constexpr int kXOff = 0;                      // Xh tile: 2 x [128 rows][128 B], swizzled
constexpr int kAOff = kXOff + BN * BK * 2;    // weight operand: same layout
constexpr int kWOff = kAOff + BM * BK * 2;    // weight source (qlh 96 B or W_exp 128 B per row)
constexpr int kDaOff = kWOff + BM * BK;       // da [4][128] f32
constexpr int kDscOff = kDaOff + 4 * BN * 4;  // dsc [128][8] f32
constexpr int kStageBytes = kDscOff + BM * 8 * 4;
static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
constexpr int kTmemCols = 512;

enum : uint32_t { kSiteEmpty = 1, kSiteFull = 2, kSiteConv = 3, kSiteTFull = 4, kSiteTEmpty = 5,
                  kSiteDrain = 6 };

struct Bars {
  uint64_t full[STAGES], conv[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)STAGES * kStageBytes + sizeof(Bars);

// Four 6-bit codes -> two binary16 pairs holding code - 32 exactly:
// bytes 0x64cc are the f16 value 1024 + cc; subtracting 1056 leaves cc - 32.
__device__ __forceinline__ void codes_to_f16(uint32_t code, uint32_t& lo, uint32_t& hi) {
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6420));  // 1056
  uint32_t a = __byte_perm(code, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(code, 0x64646464u, 0x4342);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}
// Four int8 values -> two binary16 pairs: flipping bit 7 gives v + 128 as an
// unsigned byte, 0x64xx is 1024 + that, and subtracting 1152 leaves v.
__device__ __forceinline__ void i8_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

template <bool kWexp, bool kPartials>
__global__ void __launch_bounds__(kThreads, 1)
    mmq_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ CUtensorMap tmDa, const __grid_constant__ CUtensorMap tmDsc,
                  int M, int K, int N, float* __restrict__ Y, int ldy,
                  int32_t* __restrict__ partials, unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int nk = K / BK;
  volatile int* abort_flag = &bars->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->conv[s], kConvThreads);
      mbar_init(&bars->empty[s], 1 + kNumEpiWarps);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      constexpr uint32_t kTx = BN * BK * 2 + (kWexp ? BM * BK : BM * 96) + 4 * BN * 4 + BM * 8 * 4;
      int issued = 0;
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % STAGES;
        const uint32_t ph = (kt / STAGES) & 1;
        if (!mbar_wait_bounded(&bars->empty[s], ph ^ 1, abort_flag, status, kSiteEmpty)) break;
        uint8_t* st = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&bars->full[s], kTx);
        tma_load_2d(st + kXOff, &tmX, &bars->full[s], kt * BK, n0);
        tma_load_2d(st + kXOff + BN * 128, &tmX, &bars->full[s], kt * BK + 64, n0);
        if (kWexp)
          tma_load_2d(st + kWOff, &tmW, &bars->full[s], kt * BK, m0);
        else
          tma_load_2d(st + kWOff, &tmW, &bars->full[s], kt * 96, m0);
        tma_load_2d(st + kDaOff, &tmDa, &bars->full[s], n0, kt * 4);
        tma_load_2d(st + kDscOff, &tmDsc, &bars->full[s], kt * 8, m0);
        issued = kt + 1;
      }
      if (*abort_flag) {
        // Let the copies already issued land before the CTA exits.
        for (int kt = (issued > STAGES ? issued - STAGES : 0); kt < issued; ++kt) {
          volatile int no_abort = 0;
          mbar_wait_bounded(&bars->full[kt % STAGES], (kt / STAGES) & 1, &no_abort, status,
                            kSiteFull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      int cc = 0;
      bool ok = true;
      for (int kt = 0; kt < nk && ok; ++kt) {
        const int s = kt % STAGES;
        const uint32_t ph = (kt / STAGES) & 1;
        ok = mbar_wait_bounded(&bars->full[s], ph, abort_flag, status, kSiteFull) &&
             mbar_wait_bounded(&bars->conv[s], ph, abort_flag, status, kSiteConv);
        if (!ok) break;
        tc_fence_after();
        const uint8_t* st = smem + s * kStageBytes;
        const uint32_t a_base = smem_u32(st + kAOff), b_base = smem_u32(st + kXOff);
        for (int q = 0; q < 4; ++q, ++cc) {
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
            const int j = 2 * q + h;  // sub-block within the stage
            const uint32_t koff = (uint32_t)((j >> 2) * (BN * 128) + (j & 3) * 32);
            umma_f16(tmem + (uint32_t)(b * 256 + h * 128), sw128_kmajor_desc(a_base + koff),
                     sw128_kmajor_desc(b_base + koff), idesc, 0u);
          }
          umma_commit(&bars->tfull[b]);
        }
        if (ok) umma_commit(&bars->empty[s]);
      }
      // Every MMA must be finished before TMEM is released.
      umma_commit(&bars->drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(&bars->drain, 0, &no_abort, status, kSiteDrain);
    }
    __syncwarp();
  } else if (warp < kEpiWarp0) {
    // -------------------------------------------------------------- unpack --
    const int ct = threadIdx.x - kConvWarp0 * 32;  // 0..127
    for (int kt = 0; kt < nk; ++kt) {
      const int s = kt % STAGES;
      const uint32_t ph = (kt / STAGES) & 1;
      if (!mbar_wait_bounded(&bars->full[s], ph, abort_flag, status, kSiteFull)) break;
      uint8_t* st = smem + s * kStageBytes;
      const uint8_t* wsrc = st + kWOff;
      uint8_t* aop = st + kAOff;
#pragma unroll 2
      for (int it = 0; it < (BM * 8) / kConvThreads; ++it) {
        const int item = it * kConvThreads + ct;
        const int r = item >> 3, g = item & 7;  // row, 16-element group of the half block
        uint32_t o[8];
        if (kWexp) {
          const uint4 v = *reinterpret_cast<const uint4*>(wsrc + r * 128 + g * 16);
          i8_to_f16(v.x, o[0], o[1]);
          i8_to_f16(v.y, o[2], o[3]);
          i8_to_f16(v.z, o[4], o[5]);
          i8_to_f16(v.w, o[6], o[7]);
        } else {
          // elements 16g .. 16g+15 of the half: ql bytes 16(g&3).., nibble g>>2;
          // qh bytes 16(g&1).., 2-bit field (g>>1)&3.
          const uint4 L = *reinterpret_cast<const uint4*>(wsrc + r * 96 + 16 * (g & 3));
          const uint4 H = *reinterpret_cast<const uint4*>(wsrc + r * 96 + 64 + 16 * (g & 1));
          const int nsh = 4 * (g >> 2), fsh = 2 * ((g >> 1) & 3);
          const uint32_t Lw[4] = {L.x, L.y, L.z, L.w}, Hw[4] = {H.x, H.y, H.z, H.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t code =
                ((Lw[w] >> nsh) & 0x0F0F0F0Fu) | (((Hw[w] >> fsh) & 0x03030303u) << 4);
            codes_to_f16(code, o[2 * w], o[2 * w + 1]);
          }
        }
        // 16 elements = 16B chunks 2(g&3), 2(g&3)+1 of 64-wide k-block g>>2, swizzled.
        uint8_t* row = aop + (g >> 2) * (BM * 128) + r * 128;
        const int c0 = 2 * (g & 3);
        *reinterpret_cast<uint4*>(row + ((c0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) =
            make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->conv[s]);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - kEpiWarp0;   // 0..7
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31
    const int colh = ew >> 2;          // token columns 64*colh .. +63
    const int row = 32 * quarter + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    float2 acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = make_float2(0.0f, 0.0f);
    int cc = 0;
    bool ok = true;
    for (int kt = 0; kt < nk && ok; ++kt) {
      const int s = kt % STAGES;
      const uint32_t ph = (kt / STAGES) & 1;
      if (!mbar_wait_warp(&bars->full[s], ph, abort_flag, status, kSiteFull)) break;
      const uint8_t* st = smem + s * kStageBytes;
      const float* sda = reinterpret_cast<const float*>(st + kDaOff);
      const float4 d0 = reinterpret_cast<const float4*>(st + kDscOff + row * 32)[0];
      const float4 d1 = reinterpret_cast<const float4*>(st + kDscOff + row * 32)[1];
      const float dscv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
      for (int q = 0; q < 4; ++q, ++cc) {
        const int b = cc & 1;
        const uint32_t use = (uint32_t)(cc >> 1);
        if (!mbar_wait_warp(&bars->tfull[b], use & 1, abort_flag, status, kSiteTFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float s0 = (q == 0) ? dscv[0] : (q == 1) ? dscv[2] : (q == 2) ? dscv[4] : dscv[6];
        const float s1 = (q == 0) ? dscv[1] : (q == 1) ? dscv[3] : (q == 2) ? dscv[5] : dscv[7];
        const float2 s0v = make_float2(s0, s0), s1v = make_float2(s1, s1);
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          const int col = 64 * colh + 16 * sl;
          uint32_t p0[16], p1[16];
          tmem_ld2x16(lane_addr + (uint32_t)(b * 256 + col), lane_addr + (uint32_t)(b * 256 + 128 + col),
                      p0, p1);
          const float4* dap = reinterpret_cast<const float4*>(sda + q * 128 + col);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float4 a4 = dap[v];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = 4 * v + 2 * e;
              const float2 pa = make_float2(__uint_as_float(p0[j]), __uint_as_float(p0[j + 1]));
              const float2 pb = make_float2(__uint_as_float(p1[j]), __uint_as_float(p1[j + 1]));
              float2 t = __fmul2_rn(s0v, pa);
              t = __ffma2_rn(s1v, pb, t);
              const float2 dav = e ? make_float2(a4.z, a4.w) : make_float2(a4.x, a4.y);
              acc[8 * sl + 2 * v + e] = __ffma2_rn(dav, t, acc[8 * sl + 2 * v + e]);
            }
          }
          if (kPartials) {
            const int m = m0 + row;
            if (m < M) {
              const size_t sub = (size_t)kt * 8 + 2 * q;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = n0 + col + j;
                if (n < N) {
                  int32_t* pr = partials + ((size_t)n * M + m) * (size_t)(K / 16) + sub;
                  pr[0] = (int32_t)__uint_as_float(p0[j]);
                  pr[1] = (int32_t)__uint_as_float(p1[j]);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tempty[b]);
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&bars->empty[s]);
    }
    const int m = m0 + row;
    if (m < M) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int n = n0 + 64 * colh + 2 * j;
        if (n < N) Y[(size_t)n * ldy + m] = acc[j].x;
        if (n + 1 < N) Y[(size_t)(n + 1) * ldy + m] = acc[j].y;
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

template <bool W, bool P>
cudaError_t launch_one(const TcMaps& maps, int M, int K, int N, float* Y, int ldy, int32_t* partials,
                       unsigned int* status, cudaStream_t s) {
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  mmq_tc_kernel<W, P><<<grid, kThreads, kSmemBytes, s>>>(maps.x, maps.w, maps.da, maps.dsc, M, K, N,
                                                        Y, ldy, partials, status);
  return cudaGetLastError();
}

}  // namespace

size_t mmq_tc_smem_bytes() { return kSmemBytes; }

// Raises the dynamic shared-memory limit of every instantiation; once per device.
cudaError_t mmq_tc_prepare() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(mmq_tc_kernel<false, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)))
    return e;
  if ((e = cudaFuncSetAttribute(mmq_tc_kernel<false, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)))
    return e;
  if ((e = cudaFuncSetAttribute(mmq_tc_kernel<true, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)))
    return e;
  return cudaFuncSetAttribute(mmq_tc_kernel<true, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

cudaError_t launch_mmq_tc(const TcMaps& maps, bool wexp, int M, int K, int N, float* Y, int ldy,
                          int32_t* partials, unsigned int* status, cudaStream_t s) {
  if (wexp)
    return partials ? launch_one<true, true>(maps, M, K, N, Y, ldy, partials, status, s)
                    : launch_one<true, false>(maps, M, K, N, Y, ldy, nullptr, status, s);
  return partials ? launch_one<false, true>(maps, M, K, N, Y, ldy, partials, status, s)
                  : launch_one<false, false>(maps, M, K, N, Y, ldy, nullptr, status, s);
}

}  // namespace q6
