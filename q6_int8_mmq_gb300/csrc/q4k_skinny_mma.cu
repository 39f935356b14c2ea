// q4_K x int8 GEMM for a few tokens (3 <= N <= 32) on the warp-level f16
// tensor path, with the nibbles and activations streamed into shared memory
// by TMA. HBM-bound by design: every weight byte is read once (0.59 byte per
// weight: the 0.5-byte nibbles, the 6-bit scale and min bytes of each
// 32-element sub-block and the f32 (d, dmin) of each super-block).
//
// Math ("r18: Load-time B pre-expansion", Sec. 1 and 3.2; "r38 -- q6_K
// BT-style raw-byte mma kernel", Sec. 2.2): for sub-block c of token n,
//   Y += d * (da[c] * (sc[c] * P))  -  dmin * (m[c] * us[c]),
// P = sum over the 32 elements of q * xq (q the raw nibble 0..15), formed on
// the tensor cores: two m16n8k16 f16 MMAs chained through the accumulator,
// each over 16 of the elements. us = da * (sum of the block's codes) comes
// from the quantiser as a hi/lo pair of f32.
//
// Nibbles as binary16 subnormals: a masked nibble word is the operand itself.
// In a 32-bit word of nibble bytes, bits 0-3 and 16-19 (the low nibbles of
// bytes 0 and 2) read as an f16 pair are q * 2^-24; bits 4-7 and 20-23 (the
// high nibbles) are q * 2^-20; bytes 1 and 3 take one shift by 8 first. So a
// pair of codes costs one logic operation. The activations (-127..127) become
// 1024 + (x + 128) - 1152 (a byte permute and an f16x2 subtraction). Every
// product and partial sum is an exact multiple of 2^-24 (or 2^-20) below 2^24
// of them, so P comes out scaled by a power of two and exact; the sub-block
// scale is applied as sc (even sub-blocks) or sc / 16 (odd), both exact, and
// d as d * 2^24.
//
// The min term per super-block is a small contraction, sum over its 8
// sub-blocks of m * us, run as two tf32 m16n8k8 MMAs (A = m of 16 rows, exact
// in tf32; B = the hi, then the lo part of us of 8 tokens) into the same
// fragment layout as the accumulators.
//
// MMA mapping: m16n8k16 with A = 16 weight rows x 16 elements and B = 16
// elements x 8 tokens, both in the same order: lane (g, t) = (lane / 4,
// lane % 4) holds bytes 8t .. 8t + 7 of the sub-block's 32 (nibble bytes of
// its pair of sub-blocks, activation bytes of the sub-block), the first 4 for
// the first MMA, the next 4 for the second; of each 4, bytes (0, 2) go to
// k-slots (2t, 2t+1) and bytes (1, 3) to (2t+8, 2t+9). In the super-block's
// 128 nibble bytes the pair of sub-blocks (2p, 2p+1) is the 32 bytes at 32 p
// (low nibbles sub-block 2p, high 2p + 1); its activation codes are the 32
// bytes at 32 c of the super-block's 256.
//
// Work: CTA u takes R consecutive weight rows (R = ceil(M / SMs) up to 32)
// and all of K. A producer thread streams stages of 8 super-blocks through a
// ring of 2 or 3 stages (as many as shared memory holds) with 2D TMA loads:
// the nibbles of the R rows (each stage row 1056 bytes: 1024 plus 32 of the
// next stage, so that the 8-byte loads of a fragment's rows fall on
// different banks), the stage's 2048 activation bytes of every token as two
// boxes of 1056-byte token rows, the activation scales of the stage's 64
// sub-blocks and the block-sum pairs (528-byte token rows). The sub-block
// scale and min bytes and (d, dmin) are not TMA-able (their rows are K/32
// bytes long, not a multiple of 16 when K/256 is odd): the producer warp's
// lanes copy them into the stage with 8-byte cp.async, whose completion
// arrives on the stage's full barrier next to the TMA bytes. Consumer warp
// (s, g) of 16 takes super-block s of every stage for rows 16g .. 16g + 15 of
// the unit, and the eight super-block warps' sums of a row are added in
// shared memory at the end (fixed order). For 17..32 tokens a stage holds 4
// super-blocks for 8 consumer warps, each with all four 8-token tiles (see
// Shape below). Every mbarrier wait is bounded (q6_internal.cuh).
#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int kMaxNS = 3;                 // ring stages (2 or 3, by the shared-memory budget)
constexpr int kMaxR = 32;                 // rows per unit (two MMA row groups)
constexpr int kXPitch = 1056;             // bytes per token row of an activation box (132 x 8)
constexpr int kSmemBudget = 227 * 1024;

// The stage shape for kNT token tiles of 8. Up to 16 tokens a stage holds 8
// super-blocks for 16 consumer warps (super-block x row group); for 17..32
// tokens (kNT = 3 or 4) it holds 4 super-blocks for 8 consumer warps, each forming
// the MMAs of all four token tiles on one weight fragment (the activation
// rows of 8 super-blocks for 32 tokens would not fit twice in shared memory).
// Row pitches are 32 bytes past a multiple of 128 (nibbles), 4 words past a
// multiple of 32 words (block sums) and 26 words apart modulo 32 (scales), so
// that the 8 rows of a fragment fall on different banks.
template <int kNT>
struct Shape {
  static constexpr int kSbs = kNT <= 2 ? 8 : 4;     // super-blocks per stage
  static constexpr int kCW = 2 * kSbs;              // consumer warps
  static constexpr int kThreads = 32 * (kCW + 1);   // + one producer warp
  static constexpr int kQPitch = 128 * kSbs + 32;   // bytes per row of a nibble stage (1056 / 544)
  static constexpr int kUPitch = (16 * kSbs + 4) * 4;  // bytes per token row of block sums (528 / 272)
  // bytes per row of a scale stage: kSbs x (sc 8 | m 8 | (d, dmin) 8) + 8
  static constexpr int kMPitch = 24 * kSbs + 8;     // 200 / 104
  static constexpr int kXBoxes = kSbs / 4;          // activation boxes of 1024 (+32) bytes a token
  static constexpr int kRedTok = kNT <= 2 ? 16 : 8 * kNT;  // token columns of the final sums
  // the final sums [kSbs][kRedTok][kRedPitch]: rows contiguous with a pitch of
  // 36 words, so that the fragment stores (8 rows x 4 token pairs) and the
  // row-order reads of the final addition are free of bank conflicts
  static constexpr int kRedPitch = kMaxR + 4;
  static constexpr int kRedBytes = kSbs * kRedTok * kRedPitch * 4;
};

enum : uint32_t { kSiteEmpty = 23, kSiteFull = 24 };

struct Geo {  // byte offsets of one stage's regions and the stage size, for R rows, XR tokens
  int x0, x1, da, us, meta, stage;
};
__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }
template <int kNT>
__host__ __device__ inline Geo stage_geo(int R) {
  using S = Shape<kNT>;
  constexpr int XR = 8 * kNT;  // token rows of an activation stage
  Geo g;
  g.x0 = align128(R * S::kQPitch);
  g.x1 = S::kXBoxes == 2 ? align128(g.x0 + XR * kXPitch) : g.x0;
  g.da = align128(g.x1 + XR * kXPitch);
  g.us = align128(g.da + 8 * S::kSbs * XR * 4);  // da of the stage's sub-blocks x XR tokens
  g.meta = align128(g.us + XR * S::kUPitch);
  g.stage = align128(g.meta + R * S::kMPitch);
  return g;
}
template <int kNT>
size_t smem_bytes(int R, int ns) {
  return 1024 + (size_t)ns * stage_geo<kNT>(R).stage + Shape<kNT>::kRedBytes + 256;
}

__device__ __forceinline__ uint2 lds64(const uint8_t* p) {
  return *reinterpret_cast<const uint2*>(p);
}

__device__ __forceinline__ float byte_of(uint2 v, int c) {  // unsigned byte c of 8
  return (float)(((c < 4 ? v.x : v.y) >> (8 * (c & 3))) & 0xFFu);
}
// Sub-block scale c of 8 as the factor of its MMA result: sc for even c, sc /
// 16 for odd (whose codes enter the MMA 16 times larger). Exact: the byte
// goes into the mantissa of 2^23 (or 2^19) and that power is subtracted.
__device__ __forceinline__ float scale_of(uint2 v, int c) {
  const uint32_t byte = ((c < 4 ? v.x : v.y) >> (8 * (c & 3))) & 0xFFu;
  return (c & 1) ? __uint_as_float(0x49000000u | byte) - 524288.0f
                 : __uint_as_float(0x4B000000u | byte) - 8388608.0f;
}

// D = A (16x8 tf32, row) * B (8x8 tf32, col) + C, f32 accumulation.
__device__ __forceinline__ void mma_tf32_m16n8k8(float (&d)[4], const uint32_t (&a)[4],
                                                 uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
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

template <int kCW>
__device__ __forceinline__ void bar_consumers() {  // the kCW consumer warps only
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kCW) : "memory");
}

template <int kNT, bool kPartials>
__global__ void __launch_bounds__(Shape<kNT>::kThreads, 1)
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
  using S = Shape<kNT>;
  constexpr int kSbs = S::kSbs, kCW = S::kCW, kRedTok = S::kRedTok;
  constexpr int kQPitch = S::kQPitch, kUPitch = S::kUPitch, kMPitch = S::kMPitch;
  const Geo geo = stage_geo<kNT>(R);
  float* red = reinterpret_cast<float*>(smem + (size_t)ns * geo.stage);  // [kSbs][kRedTok][kRedPitch]
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + S::kRedBytes);
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
  griddep_launch_dependents();  // the next dependent launch may start its prologue
  griddep_wait();  // launched as a dependent launch: global memory from here on

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
    const uint32_t tx = (uint32_t)R * kQPitch + (uint32_t)S::kXBoxes * (uint32_t)N * kXPitch +
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
          // x coordinates in 8-byte (nibbles, activations) or 4-byte (block
          // sums) units, each a multiple of 16 bytes
          tma_load_2d(b, &tmQ, &full[slot], 16 * kSbs * st, u * R);
          // the stage's 256 * kSbs activation bytes of each token, as boxes of
          // 1024 (+32) bytes per token row
          tma_load_2d(b + geo.x0, &tmX, &full[slot], 32 * kSbs * st, 0);
          if (S::kXBoxes == 2) tma_load_2d(b + geo.x1, &tmX, &full[slot], 32 * kSbs * st + 128, 0);
          // the activation scales of the stage's sub-blocks, [sub-block][dcols]
          tma_load_2d(b + geo.da, &tmA, &full[slot], 0, 8 * kSbs * st);
          // the block-sum pairs of the stage's super-blocks, [token][16 kSbs + 4]
          tma_load_2d(b + geo.us, &tmU, &full[slot], 16 * kSbs * st, 0);
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
        const uint8_t* qa = b + (size_t)ra * kQPitch + 128 * sbw + 8 * t;
        const uint8_t* qb = b + (size_t)rb * kQPitch + 128 * sbw + 8 * t;
        const uint8_t* xs = b + (sbw < 4 ? geo.x0 : geo.x1) + 256 * (sbw & 3) + 8 * t;
        const float* sda = reinterpret_cast<const float*>(b + geo.da) + (size_t)(8 * sbw) * dcols;
        // this super-block's entries of rows ra, rb: sc, m, (d, dmin)
        const uint8_t* ent_a = b + geo.meta + ra * kMPitch + 24 * sbw;
        const uint8_t* ent_b = b + geo.meta + rb * kMPitch + 24 * sbw;
        const uint2 zero2 = make_uint2(0u, 0u);
        const uint2 sca = have_a ? *reinterpret_cast<const uint2*>(ent_a) : zero2;
        const uint2 scb = have_b ? *reinterpret_cast<const uint2*>(ent_b) : zero2;
        float2 sbs[kNT][2];  // [token tile][row a, b]: tokens (t0, t0 + 1)
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          sbs[nt][0] = make_float2(0.0f, 0.0f);
          sbs[nt][1] = make_float2(0.0f, 0.0f);
        }
        uint2 wa = zero2, wb2 = zero2;  // nibble bytes 8t .. 8t + 7 of the current pair of sub-blocks
        uint2 xcur[kNT], xnxt[kNT];     // activation bytes 8t .. 8t + 7 of a sub-block, per token tile
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          xcur[nt] = lds64(xs + (size_t)(8 * nt + gq) * kXPitch);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          constexpr uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u;
          const bool odd = c8 & 1;
          if (!odd) {
            if (in_a) wa = lds64(qa + 16 * c8);
            if (in_b) wb2 = lds64(qb + 16 * c8);
          }
          if (c8 < 7) {
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
              xnxt[nt] = lds64(xs + (size_t)(8 * nt + gq) * kXPitch + 32 * (c8 + 1));
          }
          float P[kNT][4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t va = e ? wa.y : wa.x, vb = e ? wb2.y : wb2.x;
            const uint32_t mask = odd ? kHi : kLo;
            // bytes (0, 2) and (1, 3) of the words: binary16 subnormals
            // q * 2^-24 (low nibbles) or q * 2^-20 (high nibbles)
            const uint32_t a[4] = {va & mask, vb & mask, (va >> 8) & mask, (vb >> 8) & mask};
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
              const uint32_t xw = (e ? xcur[nt].y : xcur[nt].x) ^ 0x80808080u;
              if (e == 0) {
                const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_f16(P[nt], a, x_pair<0>(xw), x_pair<1>(xw), z);
              } else {
                const float c[4] = {P[nt][0], P[nt][1], P[nt][2], P[nt][3]};
                mma_f16(P[nt], a, x_pair<0>(xw), x_pair<1>(xw), c);
              }
            }
          }
          // P[] = P * 2^-24 (even sub-blocks) or P * 2^-20 (odd), exact; the
          // scales are taken as sc or sc / 16 so that every S is sc * P * 2^-24
          const float sa = scale_of(sca, c8), sbv = scale_of(scb, c8);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int t0 = 8 * nt + 2 * t;
            if (kPartials && partials) {
              // P of sub-block 8 sb + c8 (an exact integer)
              const float up = odd ? 1048576.0f : 16777216.0f;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int rl = (i < 2) ? ra : rb, tk = t0 + (i & 1);
                if (rl < R && r0 + rl < M && tk < N)
                  partials[((size_t)tk * M + r0 + rl) * (size_t)nc + 8 * sb + c8] =
                      (int32_t)(P[nt][i] * up);
              }
            }
            // the scales of tokens t0, t0 + 1 (columns past N hold values
            // that only tokens past N use); S then da * S, two tokens at once
            const float2 d01 = *reinterpret_cast<const float2*>(sda + c8 * dcols + t0);
            sbs[nt][0] = __ffma2_rn(
                d01, __fmul2_rn(make_float2(sa, sa), make_float2(P[nt][0], P[nt][1])), sbs[nt][0]);
            sbs[nt][1] = __ffma2_rn(
                d01, __fmul2_rn(make_float2(sbv, sbv), make_float2(P[nt][2], P[nt][3])), sbs[nt][1]);
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) xcur[nt] = xnxt[nt];
        }
        // the min term of the super-block, sum over its 8 sub-blocks of
        // m * us, as two tf32 MMAs (k = the 8 sub-blocks) on the hi and lo
        // parts of us; m (6 bits) is exact in tf32 and so is hi, lo keeps its
        // top 11 bits (us within 2^-21 |us|). Then Y += d * sbs - dmin * that.
        const uint2 mna = have_a ? *reinterpret_cast<const uint2*>(ent_a + 8) : zero2;
        const uint2 mnb = have_b ? *reinterpret_cast<const uint2*>(ent_b + 8) : zero2;
        const float2 zf = make_float2(0.0f, 0.0f);
        const float2 dda = have_a ? *reinterpret_cast<const float2*>(ent_a + 16) : zf;
        const float2 ddb = have_b ? *reinterpret_cast<const float2*>(ent_b + 16) : zf;
        // A (16 rows x 8 sub-blocks): rows g, g + 8 at sub-blocks t, t + 4
        const uint32_t am[4] = {__float_as_uint(byte_of(mna, t)), __float_as_uint(byte_of(mnb, t)),
                                __float_as_uint(byte_of(mna, t + 4)),
                                __float_as_uint(byte_of(mnb, t + 4))};
        const float da2 = dda.x * 16777216.0f, db2 = ddb.x * 16777216.0f;  // d * 2^24
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          // B (8 sub-blocks x 8 tokens): token 8 nt + g at sub-blocks t, t + 4
          const float* ur =
              reinterpret_cast<const float*>(b + geo.us + (size_t)(8 * nt + gq) * kUPitch) +
              16 * sbw;
          const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          float mn4[4];
          mma_tf32_m16n8k8(mn4, am, __float_as_uint(ur[t]), __float_as_uint(ur[t + 4]), z);
          const float c[4] = {mn4[0], mn4[1], mn4[2], mn4[3]};
          mma_tf32_m16n8k8(mn4, am, __float_as_uint(ur[8 + t]), __float_as_uint(ur[12 + t]), c);
          acc[nt][0] = fmaf(-dda.y, mn4[0], fmaf(da2, sbs[nt][0].x, acc[nt][0]));
          acc[nt][1] = fmaf(-dda.y, mn4[1], fmaf(da2, sbs[nt][0].y, acc[nt][1]));
          acc[nt][2] = fmaf(-ddb.y, mn4[2], fmaf(db2, sbs[nt][1].x, acc[nt][2]));
          acc[nt][3] = fmaf(-ddb.y, mn4[3], fmaf(db2, sbs[nt][1].y, acc[nt][3]));
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
        red[(sbw * kRedTok + tk) * S::kRedPitch + row] = acc[nt][i];
      }
    bar_consumers<kCW>();
    if (ok) {
      for (int i = threadIdx.x; i < kRedTok * R; i += 32 * kCW) {
        const int tk = i / R, row = i - tk * R;
        if (tk < N && tk < 8 * kNT && r0 + row < M) {
          float y = 0.0f;
#pragma unroll
          for (int w8 = 0; w8 < kSbs; ++w8) y += red[(w8 * kRedTok + tk) * S::kRedPitch + row];
          Y[(size_t)tk * ldy + r0 + row] = y;
        }
      }
    }
    bar_consumers<kCW>();
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
  using S = Shape<kNT>;
  // the scales of the N tokens: dcols columns of the [K/32][ldda] plane (a
  // token group of a larger call starts at a column that is a multiple of
  // 4, so the box never reaches past the plane's rows)
  const int dcols = (N + 3) & ~3;
  const int ldus = q4_min_ld(K);
  CUtensorMap mq, mx, ma, mu;
  // the activation and block-sum boxes hold the N token rows (the rows past
  // N in shared memory are never stored from)
  if (skinny_tensor_map(&mq, false, plane + g.qs_off, (uint64_t)K / 16, (uint64_t)M,
                        (uint64_t)K / 2, S::kQPitch / 8, (uint32_t)R) != CUDA_SUCCESS ||
      skinny_tensor_map(&mx, false, Xq, (uint64_t)K / 8, (uint64_t)N, (uint64_t)K, kXPitch / 8,
                        (uint32_t)N) != CUDA_SUCCESS ||
      skinny_tensor_map(&ma, true, da, (uint64_t)dcols, (uint64_t)K / 32, (uint64_t)ldda * 4,
                        (uint32_t)dcols, 8 * S::kSbs) != CUDA_SUCCESS ||
      skinny_tensor_map(&mu, true, us, (uint64_t)ldus, (uint64_t)N, (uint64_t)ldus * 4,
                        S::kUPitch / 4, (uint32_t)N) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int ns = smem_bytes<kNT>(R, 3) <= (size_t)kSmemBudget ? 3 : 2;
  if (smem_bytes<kNT>(R, ns) > (size_t)kSmemBudget) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  return launch_pdl(q4k_skinny_mma_kernel<kNT, P>, dim3(grid), dim3(S::kThreads),
                    smem_bytes<kNT>(R, ns), s, mq, mx, ma, mu, plane, g, M, K, N, R, units, ns,
                    dcols, Y, ldy, partials, status);
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
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(q4k_skinny_mma_kernel<2, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(q4k_skinny_mma_kernel<4, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(q4k_skinny_mma_kernel<3, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(q4k_skinny_mma_kernel<3, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)))
    return e;
  return cudaFuncSetAttribute(q4k_skinny_mma_kernel<4, true>,
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
  if (N <= 16)
    return partials ? launch_nt<2, true>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, partials,
                                         status, s)
                    : launch_nt<2, false>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, nullptr,
                                          status, s);
  if (N > 32) return cudaErrorInvalidValue;
  if (N <= 24)  // 17..24 tokens on three token tiles
    return partials ? launch_nt<3, true>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, partials,
                                         status, s)
                    : launch_nt<3, false>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, nullptr,
                                          status, s);
  return partials ? launch_nt<4, true>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, partials,
                                       status, s)
                  : launch_nt<4, false>(plane, M, K, Xq, da, ldda, us, N, Y, ldy, nullptr,
                                        status, s);
}

}  // namespace q6
