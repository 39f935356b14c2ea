// q6_K x int8 GEMM for a few tokens (N <= 16) on the warp-level int8 tensor
// path: the weights are streamed from the packed plane once (HBM-bound, 0.82
// byte per weight), and the products run as mma.sync.m16n8k16.s8 so that one
// activation word serves sixteen weight rows instead of one.
//
// Math ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1-2.4): per
// 16-element sub-block s the exact integer P = sum (q - 32) * xq comes from one
// MMA (A = 16 weight rows x 16 codes, B = 16 activations x 8 tokens); per
// 32-element chunk the scale is folded in integers, S = sc[2c] * P[2c] +
// sc[2c+1] * P[2c+1] (|S| < 2^24), and Y += (d * da) * S in f32.
//
// Layout: a CTA of 8 warps owns 16 weight rows; warp w takes super-blocks
// w, w + 8, ... of the rows (the eight warps read neighbouring super-blocks of
// the same rows at the same time) and the partial sums of the eight warps are
// added in shared memory at the end. Lane (g, t) = (lane / 4, lane % 4) holds
// the MMA fragments of rows g and g + 8 at codes 4t .. 4t + 3 of each
// sub-block, which it builds from 4-byte words of the qlh run ("r41 -- q6_K
// B-expand widened to uint4 group loads", Sec. 3.2 element map): within a
// 128-element half, sub-block s (0..7) takes the low (s < 4) or high nibbles
// of ql word s % 4 at byte 16 (s % 4) + 4t, and the 2-bit field s / 2 of qh
// word s % 2 at byte 64 + 16 (s % 2) + 4t. The next super-block's words are
// loaded while the current one is computed.
#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int kWarps = 8;  // warps per CTA (the K split of a row tile)

__device__ __forceinline__ uint32_t ldg32(const uint8_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// Bytes (code - 32) mod 256 of four 6-bit codes (code + 96 never carries out of
// its byte; adding 128 more flips bit 7).
__device__ __forceinline__ uint32_t centered(uint32_t code) {
  return (code + 0x60606060u) ^ 0x80808080u;
}

// Codes 4t .. 4t + 3 of sub-block s (0..7) of a half, as centered int8.
__device__ __forceinline__ uint32_t codes_of(const uint32_t (&ql)[4], const uint32_t (&qh)[2], int s) {
  const uint32_t lo = (s < 4 ? ql[s] : ql[s - 4] >> 4) & 0x0F0F0F0Fu;
  const uint32_t hi = ((qh[s & 1] >> (2 * (s >> 1))) & 0x03030303u) << 4;
  return centered(lo | hi);
}

// D = A (16x16 s8, row) * B (16x8 s8, col), int32, fresh accumulator.
__device__ __forceinline__ void mma16816(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
      "{%7, %7, %7, %7};"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "r"(0));
}

// One lane's share of a super-block of its two rows: ql / qh words of both
// halves, the 16 sub-block scales and d.
struct SbWords {
  uint32_t ql[2][2][4];  // [row][half][word]
  uint32_t qh[2][2][2];
  uint4 sc[2];
  uint16_t d[2];
};

__device__ __forceinline__ void load_sb(SbWords& w, const uint8_t* const (&q)[2],
                                        const int8_t* const (&sc)[2], const uint16_t* const (&d)[2],
                                        int sb, int t) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint8_t* hb = q[r] + (size_t)sb * 192 + 96 * h + 4 * t;
#pragma unroll
      for (int j = 0; j < 4; ++j) w.ql[r][h][j] = ldg32(hb + 16 * j);
      w.qh[r][h][0] = ldg32(hb + 64);
      w.qh[r][h][1] = ldg32(hb + 80);
    }
    w.sc[r] = __ldg(reinterpret_cast<const uint4*>(sc[r] + 16 * sb));
    w.d[r] = __ldg(d[r] + sb);
  }
}

__device__ __forceinline__ int sc_byte(const uint4 v, int i) {
  const uint32_t w = i < 4 ? v.x : i < 8 ? v.y : i < 12 ? v.z : v.w;
  return (int)(int8_t)(w >> (8 * (i & 3)));
}

template <int kNT, bool kPartials>
__global__ void __launch_bounds__(kWarps * 32, 2) mmq_skinny_mma_kernel(
    const uint8_t* __restrict__ plane, PlaneGeom g, int M, int K, const int8_t* __restrict__ Xq,
    const float* __restrict__ da, int ldda, int N, float* __restrict__ Y, int ldy,
    int32_t* __restrict__ partials) {
  __shared__ float red[kWarps][16][17];  // [warp][row][token] partial sums
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, t = lane & 3;
  const int nsb = K / 256, nc = K / 32;
  const int ntiles = (M + 15) / 16;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int m0 = 16 * tile;
    int rows[2];
    const uint8_t* q[2];
    const int8_t* scp[2];
    const uint16_t* dp[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      rows[r] = m0 + gq + 8 * r;
      const int rr = rows[r] < M ? rows[r] : M - 1;  // a row past the end reads row M-1, unused
      q[r] = plane + g.qlh_off + (size_t)rr * g.qlh_row;
      scp[r] = reinterpret_cast<const int8_t*>(plane + g.sc_off) + (size_t)rr * (K / 16);
      dp[r] = reinterpret_cast<const uint16_t*>(plane + g.d_off + (size_t)rr * g.d_row);
    }
    float acc[2][2 * kNT];  // [row][2 nt + j]: tokens 8 nt + 2t + j
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int i = 0; i < 2 * kNT; ++i) acc[r][i] = 0.0f;

    SbWords cur, nxt;
    if (warp < nsb) load_sb(cur, q, scp, dp, warp, t);
    for (int sb = warp; sb < nsb; sb += kWarps) {
      if (sb + kWarps < nsb) load_sb(nxt, q, scp, dp, sb + kWarps, t);  // in flight meanwhile
      const float dr[2] = {__half2float(__ushort_as_half(cur.d[0])),
                           __half2float(__ushort_as_half(cur.d[1]))};
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        int S[2][2 * kNT];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int i = 0; i < 2 * kNT; ++i) S[r][i] = 0;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int s16 = 2 * c8 + e, h = s16 >> 3, s = s16 & 7;
          const uint32_t a0 = codes_of(cur.ql[0][h], cur.qh[0][h], s);
          const uint32_t a1 = codes_of(cur.ql[1][h], cur.qh[1][h], s);
          const int sc0 = sc_byte(cur.sc[0], s16), sc1 = sc_byte(cur.sc[1], s16);
          const int k0 = 256 * sb + 16 * s16 + 4 * t;
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int tok = 8 * nt + gq;
            const uint32_t b =
                tok < N ? __ldg(reinterpret_cast<const unsigned int*>(Xq + (size_t)tok * K + k0)) : 0u;
            int d[4];
            mma16816(d, a0, a1, b);
            S[0][2 * nt] += sc0 * d[0];
            S[0][2 * nt + 1] += sc0 * d[1];
            S[1][2 * nt] += sc1 * d[2];
            S[1][2 * nt + 1] += sc1 * d[3];
          }
        }
        const int c = 8 * sb + c8;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int tok = 8 * nt + 2 * t + j;
            if (tok < N) {
              const float dav = __ldg(da + (size_t)c * ldda + tok);
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                acc[r][2 * nt + j] = fmaf(dr[r] * dav, (float)S[r][2 * nt + j], acc[r][2 * nt + j]);
                if (kPartials && rows[r] < M)
                  partials[((size_t)tok * M + rows[r]) * (size_t)nc + c] = S[r][2 * nt + j];
              }
            }
          }
      }
      cur = nxt;
    }
    // the eight warps' partial sums of the tile, added in a fixed order
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) red[warp][gq + 8 * r][8 * nt + 2 * t + j] = acc[r][2 * nt + j];
    __syncthreads();
    {
      const int row = threadIdx.x >> 4, tok = threadIdx.x & 15;
      if (tok < N && tok < 8 * kNT && m0 + row < M) {
        float y = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) y += red[w][row][tok];
        Y[(size_t)tok * ldy + m0 + row] = y;
      }
    }
    __syncthreads();
  }
}

template <int kNT, bool P>
cudaError_t launch_nt(const uint8_t* plane, const PlaneGeom& g, int M, int K, const int8_t* Xq,
                      const float* da, int ldda, int N, float* Y, int ldy, int32_t* partials,
                      cudaStream_t s) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mmq_skinny_mma_kernel<kNT, P>,
                                                         kWarps * 32, 0)))
    return e;
  const long long tiles = (M + 15) / 16, cap = (long long)sms * (per_sm > 0 ? per_sm : 1);
  const unsigned blocks = (unsigned)(tiles < cap ? tiles : cap);
  mmq_skinny_mma_kernel<kNT, P><<<blocks, kWarps * 32, 0, s>>>(plane, g, M, K, Xq, da, ldda, N, Y,
                                                               ldy, partials);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mmq_skinny_mma(const uint8_t* plane, int M, int K, const int8_t* Xq,
                                  const float* da, int ldda, int N, float* Y, int ldy,
                                  int32_t* partials, cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  if (N <= 8)
    return partials ? launch_nt<1, true>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, partials, s)
                    : launch_nt<1, false>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, nullptr, s);
  return partials ? launch_nt<2, true>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, partials, s)
                  : launch_nt<2, false>(plane, g, M, K, Xq, da, ldda, N, Y, ldy, nullptr, s);
}

}  // namespace q6
