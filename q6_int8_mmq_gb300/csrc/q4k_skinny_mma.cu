// q4_K x int8 GEMM for a few tokens (3 <= N <= 16) on the warp-level f16
// tensor path, with the nibbles and activations streamed into shared memory
// by TMA. HBM-bound by design: every weight byte is read once (0.59 byte per
// weight: the 0.5-byte nibbles, the 6-bit scale and min bytes of each
// 32-element sub-block and the f32 (d, dmin) of each super-block).
//
// Math ("r18: Load-time B pre-expansion", Sec. 1 and 3.2; "r38 -- q6_K
// BT-style raw-byte mma kernel", Sec. 2.2): for sub-block c of token n,
//   Y += d * (da[c] * (sc[c] * P))  -  dmin * (m[c] * us[c]),
// P = sum over the 32 elements of q * xq (q the raw nibble 0..15), formed on
// the tensor cores: two m16n8k16 MMAs chained through the accumulator, each
// over 16 of the elements. The products and sums are small integers, exact
// in f16 x f16 -> f32 (every partial sum is at most 15 * 127 * 32 < 2^24),
// and so is sc * P (< 63 * 15 * 127 * 32). us = da * (sum of the block's
// codes) comes from the quantiser as an exact hi/lo pair of f32.
//
// Code conversion: a lane's four nibbles of a 16-element group sit in one
// 32-bit word (low nibbles for sub-block 2p, high for 2p + 1 of the group of
// 32 bytes p); one byte permute places the exponent byte 0x64 above each
// nibble (1024 + q as binary16) and one f16x2 subtraction of 1024 leaves q.
//
// MMA mapping: m16n8k16 with A = 16 weight rows x 16 elements and B = 16
// elements x 8 tokens, both in the same order of the 16 elements: lane
// (g, t) = (lane / 4, lane % 4) holds elements 4t .. 4t + 3 of the group, the
// pairs (4t, 4t+2) in k-slots (2t, 2t+1) and (4t+1, 4t+3) in (2t+8, 2t+9).
// In the super-block's 128 nibble bytes, group e (0, 1) of sub-block c is the
// 16 bytes at 32 (c / 2) + 16 e, low nibbles for even c, high for odd, so a
// lane's word of it is at 32 (c / 2) + 16 e + 4t; its activation word is at
// byte 32 c + 16 e + 4t of the super-block's 256 codes.
//
// Work: CTA u takes R consecutive weight rows (R = ceil(M / SMs) up to 32)
// and all of K. A producer thread streams stages of 8 super-blocks through a
// ring of 2 or 3 stages (as many as shared memory holds) with 2D TMA loads:
// the nibbles of the R rows (each stage row 1040 bytes: 1024 plus 16 of the
// next stage, so that the 8 rows of a fragment fall on different banks), the
// stage's 2048 activation bytes of every token as two boxes of 1040-byte
// token rows, the activation scales of the stage's 64 sub-blocks and the
// block-sum pairs (528-byte token rows). The sub-block scale and min bytes
// and (d, dmin) are not TMA-able (their rows are K/32 bytes long, not a
// multiple of 16 when K/256 is odd): the producer warp's lanes copy them into
// the stage with 8-byte cp.async, whose completion arrives on the stage's
// full barrier next to the TMA bytes. Consumer warp (s, g) of 16 takes
// super-block s of every stage for rows 16g .. 16g + 15 of the unit, and the
// eight super-block warps' sums of a row are added in shared memory at the
// end (fixed order). Every mbarrier wait is bounded (q6_internal.cuh).
#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int kSbs = 8;                   // super-blocks per stage
constexpr int kCW = 2 * kSbs;             // consumer warps: super-block x row group of 16
constexpr int kThreads = 32 * (kCW + 1);  // + one producer warp
constexpr int kMaxNS = 3;                 // ring stages (2 or 3, by the shared-memory budget)
constexpr int kMaxR = 32;                 // rows per unit (two MMA row groups)
constexpr int kQPitch = 1040;             // bytes per row of a nibble stage (130 x 8)
constexpr int kXPitch = 1040;             // bytes per token row of an activation half-stage
constexpr int kUPitch = 528;              // bytes per token row of a block-sum stage (132 f32)
// bytes per row of a scale stage: 8 super-blocks x (sc 8 | m 8 | (d, dmin) 8),
// padded so that the 8 rows of a fragment fall on different banks
constexpr int kMPitch = 200;
constexpr int kSmemBudget = 227 * 1024;
constexpr int kRedBytes = kSbs * kMaxR * 16 * 4;

enum : uint32_t { kSiteEmpty = 23, kSiteFull = 24 };

struct Geo {  // byte offsets of one stage's regions and the stage size, for R rows, XR tokens
  int x0, x1, da, us, meta, stage;
};
__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }
__host__ __device__ inline Geo stage_geo(int R, int XR) {
  Geo g;
  g.x0 = align128(R * kQPitch);
  g.x1 = align128(g.x0 + XR * kXPitch);
  g.da = align128(g.x1 + XR * kXPitch);
  g.us = align128(g.da + 8 * kSbs * XR * 4);  // da of the stage's 64 sub-blocks x XR tokens
  g.meta = align128(g.us + XR * kUPitch);
  g.stage = align128(g.meta + R * kMPitch);
  return g;
}
size_t smem_bytes(int R, int XR, int ns) {
  return 1024 + (size_t)ns * stage_geo(R, XR).stage + kRedBytes + 256;
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// Nibbles (0..15, one per byte) of bytes (kOdd, kOdd + 2) of `nib` as the
// binary16 pair q: 1024 + q (exponent byte 0x64 above each) minus 1024.
template <int kOdd>
__device__ __forceinline__ uint32_t q_pair(uint32_t nib) {
  return hsub2u(__byte_perm(nib, 0x64u, kOdd ? 0x4341u : 0x4240u), kH2_1024);
}

__device__ __forceinline__ float byte_of(uint2 v, int c) {  // unsigned byte c of 8
  return (float)(((c < 4 ? v.x : v.y) >> (8 * (c & 3))) & 0xFFu);
}

// An 8-byte copy global -> shared; the copies of a thread complete in the
// background and are tracked by cp_async_arrive.
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
// One arrival on `bar` once all of this thread's earlier cp.async copies have
// landed (counted in the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void bar_consumers() {  // the kCW consumer warps only
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kCW) : "memory");
}

template <int kNT, bool kPartials>
__global__ void __launch_bounds__(kThreads, 1)
    q4k_skinny_mma_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmU, const uint8_t* __restrict__ plane,
                          Q4Geom pg, int M, int K, int N, int R, int units, int ns, int dcols,
                          float* __restrict__ Y, int ldy, int32_t* __restrict__ partials,
                          unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int XR = 8 * kNT;  // token rows of an activation stage
  const Geo geo = stage_geo(R, XR);
  float* red = reinterpret_cast<float*>(smem + (size_t)ns * geo.stage);  // [kSbs][kMaxR][16]
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + kRedBytes);
  uint64_t* empty = full + kMaxNS;
  int* abort_word = reinterpret_cast<int*>(empty + kMaxNS);
  volatile int* abort_flag = abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = K / 256, nst = (nsb + kSbs - 1) / kSbs, nc = K / 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1 + 32);  // the TMA thread + the producer lanes' copies
      mbar_init(&empty[s], kCW);
    }
    *abort_word = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kCW) {
    // ----------------------------------------------------------- producer --
    // lane 0 issues the TMA loads; every lane copies a share of the stage's
    // scale entries (row, super-block) and arrives on the full barrier when
    // its copies have landed
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmU);
    }
    const uint32_t tx = (uint32_t)R * kQPitch + 2u * (uint32_t)N * kXPitch +
                        (uint32_t)(8 * kSbs) * (uint32_t)dcols * 4u + (uint32_t)N * kUPitch;
    const uint8_t* scp = plane + pg.sc_off;
    const uint8_t* mnp = plane + pg.mn_off;
    const uint8_t* ddp = plane + pg.ddm_off;
    int gs = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      for (int st = 0; st < nst; ++st, ++gs) {
        const int slot = gs % ns;
        if (!(ok = mbar_wait_warp(&empty[slot], ((gs / ns) & 1) ^ 1, abort_flag, status,
                                  kSiteEmpty)))
          break;
        uint8_t* b = smem + (size_t)slot * geo.stage;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[slot], tx);
          tma_load_2d(b, &tmQ, &full[slot], 128 * st, u * R);
          // the stage's 2048 activation bytes of each token, as two boxes of
          // 1024 (+16) bytes per token row
          tma_load_2d(b + geo.x0, &tmX, &full[slot], 256 * st, 0);
          tma_load_2d(b + geo.x1, &tmX, &full[slot], 256 * st + 128, 0);
          // the activation scales of the stage's 64 sub-blocks, [sub-block][dcols]
          tma_load_2d(b + geo.da, &tmA, &full[slot], 0, 64 * st);
          // the block-sum pairs of the stage's 8 super-blocks, [token][132]
          tma_load_2d(b + geo.us, &tmU, &full[slot], 128 * st, 0);
        }
        // entries past M or past the last super-block are not copied (the
        // consumers do not read them)
        for (int j = lane; j < kSbs * R; j += 32) {
          const int row = j / kSbs, sbl = j - row * kSbs, sb = kSbs * st + sbl;
          const int m = u * R + row;
          if (m < M && sb < nsb) {
            uint8_t* dst = b + geo.meta + row * kMPitch + 24 * sbl;
            cp_async8(dst, scp + (size_t)m * nc + 8 * sb);
            cp_async8(dst + 8, mnp + (size_t)m * nc + 8 * sb);
            cp_async8(dst + 16, ddp + ((size_t)m * nsb + sb) * 8);
          }
        }
        cp_async_arrive(&full[slot]);
      }
    }
    cp_async_wait_all();
    if (!ok && lane == 0) {
      // let the copies already issued land before the CTA exits
      volatile int no_abort = 0;
      for (int k = (gs > ns ? gs - ns : 0); k < gs; ++k)
        mbar_wait_bounded(&full[k % ns], (k / ns) & 1, &no_abort, status, kSiteFull);
    }
    return;
  }

  // --------------------------------------------------------------- consumers --
  // warp (sbw, rg): super-block sbw of every stage, rows 16 rg .. 16 rg + 15 of the unit
  const int sbw = warp % kSbs, rg = warp / kSbs;
  const int gq = lane >> 2, t = lane & 3;
  const int ra = 16 * rg + gq, rb = ra + 8;  // this lane's two rows (unit-relative)
  const bool in_a = ra < R, in_b = rb < R, active = 16 * rg < R;
  int gs = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int r0 = u * R;
    const bool have_a = in_a && r0 + ra < M, have_b = in_b && r0 + rb < M;
    float acc[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
    for (int st = 0; st < nst; ++st, ++gs) {
      const int slot = gs % ns;
      if (ok) ok = mbar_wait_warp(&full[slot], (gs / ns) & 1, abort_flag, status, kSiteFull);
      const int sb = kSbs * st + sbw;
      if (ok && active && sb < nsb) {
        const uint8_t* b = smem + (size_t)slot * geo.stage;
        // rows past R are not in the stage (their bytes belong to the next region)
        const uint8_t* qa = b + (size_t)ra * kQPitch + 128 * sbw + 4 * t;
        const uint8_t* qb = b + (size_t)rb * kQPitch + 128 * sbw + 4 * t;
        const uint8_t* xs = b + (sbw < 4 ? geo.x0 : geo.x1) + 256 * (sbw & 3) + 4 * t;
        const float* sda = reinterpret_cast<const float*>(b + geo.da) + (size_t)(8 * sbw) * dcols;
        // this super-block's entries of rows ra, rb: sc, m, (d, dmin)
        const uint8_t* ent_a = b + geo.meta + ra * kMPitch + 24 * sbw;
        const uint8_t* ent_b = b + geo.meta + rb * kMPitch + 24 * sbw;
        const uint2 zero2 = make_uint2(0u, 0u);
        const uint2 sca = have_a ? *reinterpret_cast<const uint2*>(ent_a) : zero2;
        const uint2 scb = have_b ? *reinterpret_cast<const uint2*>(ent_b) : zero2;
        auto load_x = [&](int c8, uint32_t (&xw)[2][kNT]) {
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
              xw[e][nt] = lds32(xs + (size_t)(8 * nt + gq) * kXPitch + 32 * c8 + 16 * e);
        };
        float sbs[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sbs[nt][i] = 0.0f;
        uint32_t w[2][2];  // nibble words [row][group e] of the current pair of sub-blocks
        uint32_t xcur[2][kNT], xnxt[2][kNT];
        load_x(0, xcur);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          if ((c8 & 1) == 0) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              w[0][e] = in_a ? lds32(qa + 16 * c8 + 16 * e) : 0u;
              w[1][e] = in_b ? lds32(qb + 16 * c8 + 16 * e) : 0u;
            }
          }
          if (c8 < 7) load_x(c8 + 1, xnxt);
          float P[kNT][4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t na = ((c8 & 1) ? w[0][e] >> 4 : w[0][e]) & 0x0F0F0F0Fu;
            const uint32_t nb = ((c8 & 1) ? w[1][e] >> 4 : w[1][e]) & 0x0F0F0F0Fu;
            const uint32_t a[4] = {q_pair<0>(na), q_pair<0>(nb), q_pair<1>(na), q_pair<1>(nb)};
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
              const uint32_t wb = xcur[e][nt] ^ 0x80808080u;
              if (e == 0) {
                const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_f16(P[nt], a, x_pair<0>(wb), x_pair<1>(wb), z);
              } else {
                const float c[4] = {P[nt][0], P[nt][1], P[nt][2], P[nt][3]};
                mma_f16(P[nt], a, x_pair<0>(wb), x_pair<1>(wb), c);
              }
            }
          }
          const float sa = byte_of(sca, c8), sbv = byte_of(scb, c8);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int t0 = 8 * nt + 2 * t;
            if (kPartials && partials) {
              // P of sub-block 8 sb + c8 (an exact integer in f32)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int rl = (i < 2) ? ra : rb, tk = t0 + (i & 1);
                if (rl < R && r0 + rl < M && tk < N)
                  partials[((size_t)tk * M + r0 + rl) * (size_t)nc + 8 * sb + c8] =
                      (int32_t)P[nt][i];
              }
            }
            const float d0 = t0 < N ? sda[c8 * dcols + t0] : 0.0f;
            const float d1 = t0 + 1 < N ? sda[c8 * dcols + t0 + 1] : 0.0f;
            // sc * P is exact in f32 (< 2^24)
            sbs[nt][0] = fmaf(d0, sa * P[nt][0], sbs[nt][0]);
            sbs[nt][1] = fmaf(d1, sa * P[nt][1], sbs[nt][1]);
            sbs[nt][2] = fmaf(d0, sbv * P[nt][2], sbs[nt][2]);
            sbs[nt][3] = fmaf(d1, sbv * P[nt][3], sbs[nt][3]);
          }
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) xcur[e][nt] = xnxt[e][nt];
        }
        // the min term of the super-block: sum over its 8 sub-blocks of
        // m * us, with us = hi + lo from the quantiser's pairs (exact); then
        // Y += d * sbs - dmin * (that sum)
        const uint2 mna = have_a ? *reinterpret_cast<const uint2*>(ent_a + 8) : zero2;
        const uint2 mnb = have_b ? *reinterpret_cast<const uint2*>(ent_b + 8) : zero2;
        const float2 zf = make_float2(0.0f, 0.0f);
        const float2 dda = have_a ? *reinterpret_cast<const float2*>(ent_a + 16) : zf;
        const float2 ddb = have_b ? *reinterpret_cast<const float2*>(ent_b + 16) : zf;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float* ur = reinterpret_cast<const float*>(
                b + geo.us + (size_t)(8 * nt + 2 * t + j) * kUPitch + 64 * sbw);
            const float4 h0 = *reinterpret_cast<const float4*>(ur);
            const float4 h1 = *reinterpret_cast<const float4*>(ur + 4);
            const float4 l0 = *reinterpret_cast<const float4*>(ur + 8);
            const float4 l1 = *reinterpret_cast<const float4*>(ur + 12);
            const float uu[8] = {h0.x + l0.x, h0.y + l0.y, h0.z + l0.z, h0.w + l0.w,
                                 h1.x + l1.x, h1.y + l1.y, h1.z + l1.z, h1.w + l1.w};
            float sa = 0.0f, sb2 = 0.0f;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              sa = fmaf(byte_of(mna, c8), uu[c8], sa);
              sb2 = fmaf(byte_of(mnb, c8), uu[c8], sb2);
            }
            acc[nt][j] = fmaf(-dda.y, sa, fmaf(dda.x, sbs[nt][j], acc[nt][j]));
            acc[nt][2 + j] = fmaf(-ddb.y, sb2, fmaf(ddb.x, sbs[nt][2 + j], acc[nt][2 + j]));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // the eight super-block warps' sums of each row, added in a fixed order
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = (i < 2) ? ra : rb, tk = 8 * nt + 2 * t + (i & 1);
        red[(sbw * kMaxR + row) * 16 + tk] = acc[nt][i];
      }
    bar_consumers();
    if (ok) {
      for (int i = threadIdx.x; i < 16 * R; i += 32 * kCW) {
        const int tk = i / R, row = i - tk * R;
        if (tk < N && tk < 8 * kNT && r0 + row < M) {
          float y = 0.0f;
#pragma unroll
          for (int w8 = 0; w8 < kSbs; ++w8) y += red[(w8 * kMaxR + row) * 16 + tk];
          Y[(size_t)tk * ldy + r0 + row] = y;
        }
      }
    }
    bar_consumers();
  }
}

template <int kNT, bool P>
cudaError_t launch_nt(const uint8_t* plane, int M, int K, const int8_t* Xq, const float* da,
                      int ldda, const float* us, int N, float* Y, int ldy, int32_t* partials,
                      unsigned int* status, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  // R rows per unit, at most kMaxR, units in whole waves over the SMs
  const long long waves = ((long long)M + (long long)kMaxR * sms - 1) / ((long long)kMaxR * sms);
  const int R = (int)(((long long)M + waves * sms - 1) / (waves * sms));
  const int units = (M + R - 1) / R;
  const Q4Geom g = q4_geom(M, K);
  // the scales of the N tokens: dcols columns of the [K/32][ldda] plane (a
  // token group of a larger call starts at a column that is a multiple of
  // 16, so the box never reaches past the plane's rows)
  const int dcols = (N + 3) & ~3;
  const int ldus = q4_min_ld(K);
  CUtensorMap mq, mx, ma, mu;
  // the activation and block-sum boxes hold the N token rows (the rows past
  // N in shared memory are never stored from)
  if (skinny_tensor_map(&mq, false, plane + g.qs_off, (uint64_t)K / 16, (uint64_t)M,
                        (uint64_t)K / 2, kQPitch / 8, (uint32_t)R) != CUDA_SUCCESS ||
      skinny_tensor_map(&mx, false, Xq, (uint64_t)K / 8, (uint64_t)N, (uint64_t)K, kXPitch / 8,
                        (uint32_t)N) != CUDA_SUCCESS ||
      skinny_tensor_map(&ma, true, da, (uint64_t)dcols, (uint64_t)K / 32, (uint64_t)ldda * 4,
                        (uint32_t)dcols, 8 * kSbs) != CUDA_SUCCESS ||
      skinny_tensor_map(&mu, true, us, (uint64_t)ldus, (uint64_t)N, (uint64_t)ldus * 4,
                        kUPitch / 4, (uint32_t)N) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int ns = smem_bytes(R, 8 * kNT, 3) <= (size_t)kSmemBudget ? 3 : 2;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  q4k_skinny_mma_kernel<kNT, P><<<grid, kThreads, smem_bytes(R, 8 * kNT, ns), s>>>(
      mq, mx, ma, mu, plane, g, M, K, N, R, units, ns, dcols, Y, ldy, partials, status);
  return cudaGetLastError();
}

}  // namespace

// Raises the dynamic shared-memory limit of every instantiation.
cudaError_t q4k_skinny_mma_prepare() {
  const int bytes = kSmemBudget;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(q4k_skinny_mma_kernel<1, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(q4k_skinny_mma_kernel<1, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(q4k_skinny_mma_kernel<2, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)))
    return e;
  return cudaFuncSetAttribute(q4k_skinny_mma_kernel<2, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_q4k_skinny_mma(const uint8_t* plane, int M, int K, const int8_t* Xq,
                                  const float* da, int ldda, const float* us, int N, float* Y,
                                  int ldy, int32_t* partials, unsigned int* status,
                                  cudaStream_t s) {
  if (N <= 8)
    return partials ? launch_nt<1, true>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, partials,
                                         status, s)
                    : launch_nt<1, false>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, nullptr,
                                          status, s);
  return partials ? launch_nt<2, true>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, partials,
                                       status, s)
                  : launch_nt<2, false>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, nullptr,
                                        status, s);
}

}  // namespace q6
