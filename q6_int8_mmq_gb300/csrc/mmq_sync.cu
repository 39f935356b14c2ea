// q6_K x int8 GEMM on the legacy warp-level tensor path (mma.sync), the
// pages' own route, kept as a measured comparison point for the tcgen05
// kernel on sm_103a.
//
// What it computes is the same as the tensor-core kernel; how follows the
// pages ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.2-2.4; "r53 --
// q6_K bundle: W_exp pre-expansion plane", Sec. 2.3): the weights come from
// the pre-expanded centered-int8 W_exp plane, the activations from Xq, and
// one exact int32 partial P per 16-element sub-block is formed with
// mma.sync.m16n8k16.s8. The scale sc is folded in integers per 32-element
// chunk, S = sc[2c] * P[2c] + sc[2c+1] * P[2c+1] (|S| < 2^24), and the
// rescale is the same two-level f32 form: Sb += da * S per chunk,
// Y += d * Sb per super-block.
//
// CTA tile 128 weight rows x 64 tokens, 8 warps of 32 x 32; one super-block
// (256 of K) per shared-memory stage, two stages filled by cp.async (rows
// padded to 272 bytes so every ldmatrix phase is free of bank conflicts).
#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int SBM = 128, SBN = 64, SKB = 256, RS = SKB + 16;
constexpr int kStW = 0, kStX = kStW + SBM * RS, kStSc = kStX + SBN * RS;
constexpr int kStDa = kStSc + SBM * 16, kStD = kStDa + 8 * SBN * 4;
constexpr int kStage = kStD + SBM * 4;
constexpr int kSyncSmem = 2 * kStage;
static_assert(kStage % 16 == 0, "stage alignment");

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = smem_u32(dst);
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A (16x16 s8, row) * B (16x8 s8, col), fresh int32 accumulator.
__device__ __forceinline__ void mma_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
      "{%7, %7, %7, %7};"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "r"(0));
}

// One super-block's operands and scales into stage `st` (zero-filled outside
// the matrix).
__device__ __forceinline__ void load_stage(uint8_t* st, const int8_t* __restrict__ wexp,
                                           const int8_t* __restrict__ scp,
                                           const float* __restrict__ dT, int ldm,
                                           const int8_t* __restrict__ Xq,
                                           const float* __restrict__ da, int ldda, int M, int K,
                                           int N, int m0, int n0, int sb) {
  const int tid = threadIdx.x;
  for (int p = tid; p < SBM * 16; p += 256) {  // W: 128 rows x 16 pieces
    const int r = p >> 4, c = p & 15, m = m0 + r;
    const bool ok = m < M;
    cp_async16(st + kStW + r * RS + 16 * c, wexp + (size_t)(ok ? m : 0) * K + sb * SKB + 16 * c, ok);
  }
  for (int p = tid; p < SBN * 16; p += 256) {  // X: 64 tokens x 16 pieces
    const int r = p >> 4, c = p & 15, n = n0 + r;
    const bool ok = n < N;
    cp_async16(st + kStX + r * RS + 16 * c, Xq + (size_t)(ok ? n : 0) * K + sb * SKB + 16 * c, ok);
  }
  // scales: sc (128 rows x 16 bytes), da (8 chunks x 64 tokens), d (128 rows)
  constexpr int kPSc = SBM, kPDa = 8 * (SBN / 4), kPD = SBM / 4;
  for (int p = tid; p < kPSc + kPDa + kPD; p += 256) {
    if (p < kPSc) {
      const int m = m0 + p;
      const bool ok = m < M;
      cp_async16(st + kStSc + p * 16, scp + (size_t)(ok ? m : 0) * (K / 16) + sb * 16, ok);
    } else if (p < kPSc + kPDa) {
      const int q = p - kPSc, c = q / (SBN / 4), j = q % (SBN / 4), n = n0 + 4 * j;
      const bool ok = n < ldda;
      cp_async16(st + kStDa + (c * SBN + 4 * j) * 4, da + (size_t)(8 * sb + c) * ldda + (ok ? n : 0),
                 ok);
    } else {
      const int q = p - kPSc - kPDa, m = m0 + 4 * q;
      const bool ok = m < ldm;
      cp_async16(st + kStD + 16 * q, dT + (size_t)sb * ldm + (ok ? m : 0), ok);
    }
  }
}

template <bool kPartials>
__global__ void __launch_bounds__(256, 1)
    mmq_sync_kernel(const int8_t* __restrict__ wexp, const int8_t* __restrict__ scp,
                    const float* __restrict__ dT, int ldm, int M, int K,
                    const int8_t* __restrict__ Xq, const float* __restrict__ da, int ldda, int N,
                    float* __restrict__ Y, int ldy, int32_t* __restrict__ partials,
                    int32_t* __restrict__ chunks) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp & 3, wn = warp >> 2;  // 32-row x 32-token warp tile
  const int g = lane >> 2, t = lane & 3;    // mma fragment coordinates
  const int m0 = blockIdx.y * SBM, n0 = blockIdx.x * SBN;
  const int nsb = K / SKB, nc = K / 32;

  float acc[2][4][4], sbacc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.0f;

  load_stage(smem, wexp, scp, dT, ldm, Xq, da, ldda, M, K, N, m0, n0, 0);
  cp_async_commit();
  for (int sb = 0; sb < nsb; ++sb) {
    uint8_t* st = smem + (sb & 1) * kStage;
    if (sb + 1 < nsb)
      load_stage(smem + ((sb + 1) & 1) * kStage, wexp, scp, dT, ldm, Xq, da, ldda, M, K, N, m0,
                 n0, sb + 1);
    cp_async_commit();
    cp_async_wait<1>();  // this super-block's group has landed
    __syncthreads();
    const uint32_t wbase = smem_u32(st + kStW), xbase = smem_u32(st + kStX);
    const int8_t* sc_s = reinterpret_cast<const int8_t*>(st + kStSc);
    const float* da_s = reinterpret_cast<const float*>(st + kStDa);
    const float* d_s = reinterpret_cast<const float*>(st + kStD);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      int P[2][2][4][4];  // [sub-block][m16][n8][element]
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int koff = 32 * c + 16 * h;
        uint32_t a[2][2], b[4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
          ldsm_x2(wbase + (uint32_t)((wm * 32 + mi * 16 + (lane & 15)) * RS + koff), a[mi][0],
                  a[mi][1]);
        ldsm_x4(xbase + (uint32_t)((wn * 32 + (lane >> 3) * 8 + (lane & 7)) * RS + koff), b[0], b[1],
                b[2], b[3]);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int ni = 0; ni < 4; ++ni) mma_s8(P[h][mi][ni], a[mi][0], a[mi][1], b[ni]);
      }
      // S = sc * P over the chunk's two sub-blocks (exact), then Sb += da * S
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int row = wm * 32 + mi * 16 + g + 8 * half;
          const int sa = sc_s[row * 16 + 2 * c], sbv = sc_s[row * 16 + 2 * c + 1];
#pragma unroll
          for (int ni = 0; ni < 4; ++ni) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int e = 2 * half + e2;
              const int tok = wn * 32 + ni * 8 + 2 * t + e2;
              const int S = sa * P[0][mi][ni][e] + sbv * P[1][mi][ni][e];
              const float dav = da_s[c * SBN + tok];
              sbacc[mi][ni][e] = (c == 0) ? dav * (float)S : fmaf(dav, (float)S, sbacc[mi][ni][e]);
              if (kPartials) {
                const int n = n0 + tok, m = m0 + row;
                if (n < N && m < M) {
                  const size_t nm = (size_t)n * M + m;
                  if (chunks) chunks[nm * (size_t)nc + 8 * sb + c] = S;
                  if (partials) {
                    // P of the chunk's two sub-blocks 2c, 2c + 1
                    partials[nm * (size_t)(2 * nc) + 16 * sb + 2 * c] = P[0][mi][ni][e];
                    partials[nm * (size_t)(2 * nc) + 16 * sb + 2 * c + 1] = P[1][mi][ni][e];
                  }
                }
              }
            }
          }
        }
      }
    }
    // Y += d * Sb for this super-block
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float dv = d_s[wm * 32 + mi * 16 + g + 8 * half];
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2)
            acc[mi][ni][2 * half + e2] = fmaf(dv, sbacc[mi][ni][2 * half + e2], acc[mi][ni][2 * half + e2]);
      }
    __syncthreads();  // the stage may be refilled
  }
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = m0 + wm * 32 + mi * 16 + g + 8 * (e >> 1);
        const int n = n0 + wn * 32 + ni * 8 + 2 * t + (e & 1);
        if (m < M && n < N) Y[(size_t)n * ldy + m] = acc[mi][ni][e];
      }
}

}  // namespace

cudaError_t mmq_sync_prepare() {
  cudaError_t e = cudaFuncSetAttribute(mmq_sync_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSyncSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mmq_sync_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSyncSmem);
}

cudaError_t launch_mmq_sync(const uint8_t* plane, const int8_t* wexp, int M, int K,
                            const int8_t* Xq, const float* da, int ldda, int N, float* Y, int ldy,
                            Debug dbg, cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  const int8_t* scp = reinterpret_cast<const int8_t*>(plane + g.sc_off);
  const float* dT = reinterpret_cast<const float*>(plane + g.dt_off);
  dim3 grid((unsigned)((N + SBN - 1) / SBN), (unsigned)((M + SBM - 1) / SBM));
  if (dbg.any())
    mmq_sync_kernel<true><<<grid, 256, kSyncSmem, s>>>(wexp, scp, dT, g.ldm, M, K, Xq, da, ldda, N,
                                                       Y, ldy, dbg.partials, dbg.chunk_sums);
  else
    mmq_sync_kernel<false><<<grid, 256, kSyncSmem, s>>>(wexp, scp, dT, g.ldm, M, K, Xq, da, ldda,
                                                        N, Y, ldy, nullptr, nullptr);
  return cudaGetLastError();
}

}  // namespace q6
