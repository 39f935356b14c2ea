// q6_K x int8 GEMM for a few tokens (3 <= N <= 32) on the warp-level f16
// tensor path, with the weights streamed into shared memory by TMA. HBM-bound
// by design: every weight byte is read once (0.82 byte per weight).
//
// Math ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1-2.4): per
// 16-element sub-block s the exact integer P = sum (q - 32) * xq is formed on
// the tensor cores, per 32-element chunk the sub-block scales are applied,
// S = sc[2c] * P[2c] + sc[2c+1] * P[2c+1], and Y += d * (da * S) in f32.
//
// Why f16 and not int8 MMA: on this GPU an int8 mma.sync.m16n8k16 takes about
// 16 cycles per SM and an f16 one about 2 (measured), and the sub-block scale
// needs one MMA per 16 codes. The products are exact in f16 with f32
// accumulation: codes (q - 32) and activations (-127..127) are small
// integers, and every partial sum of a sub-block is at most 16 * 32 * 127.
// Each lane assembles its four 6-bit codes of a sub-block in one 32-bit word
// (ql nibbles | qh field << 4) and turns byte pairs into binary16 pairs with
// one byte permute (exponent byte 0x64 above each code: 1024 + code) and one
// f16x2 subtraction of 1056.
//
// MMA mapping: m16n8k16, A = 16 weight rows x 16 codes, B = 16 codes x 8
// tokens, both with the same order of the 16 codes: lane (g, t) = (lane / 4,
// lane % 4) holds codes 4t .. 4t + 3 of the sub-block, as the pairs (4t, 4t+2)
// in k-slots (2t, 2t+1) and (4t+1, 4t+3) in k-slots (2t+8, 2t+9). Those four
// codes sit in the same byte positions of one ql word and one qh word (the
// element map of Sec. 3.2, "r41 -- q6_K B-expand widened to uint4 group
// loads"): in half h of a super-block's 192-byte qlh run (64 ql bytes, then
// 32 qh bytes, per half), sub-block j (0..7) takes the low (j < 4) or high
// nibbles of the ql word at byte 96 h + 16 (j % 4) + 4t and the 2-bit field
// j / 2 of the qh word at byte 96 h + 64 + 16 (j % 2) + 4t.
//
// Work: CTA u takes R consecutive weight rows (R = ceil(M / SMs) up to 32,
// so every SM gets the same number of rows to within one) and all of K. A
// producer thread streams stages of 8 super-blocks of those rows through a
// ring of 2 or 3 stages (as many as shared memory holds) with 2D TMA loads:
// qlh, sc and d of the rows, the stage's 2048 activation bytes of every
// token as two boxes of 1040-byte token rows, and the activation scales of
// the stage's 64 chunks. Each row of a qlh stage box is
// 1552 bytes (1536 plus 16 of the next stage) and each activation row 1040,
// so that the 8 rows of a fragment fall on different shared-memory banks. Consumer warp (s, g)
// of 16 takes super-block s of every stage for rows 16g .. 16g + 15 of the
// unit (16 warps, four per scheduler, hide the MMA and shared-memory
// latencies), and the eight super-block warps' sums of a row are added in
// shared memory at the end (fixed order). For 17..32 tokens a stage holds
// 4 super-blocks (one activation box a token) for 8 consumer warps, each with
// all four 8-token tiles (see Shape below).
// Every mbarrier wait is bounded (see q6_internal.cuh).
#include <cudaTypedefs.h>

#include <mutex>

#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int kMaxNS = 3;                // ring stages (2 or 3, by the shared-memory budget)
constexpr int kMaxR = 32;                // rows per unit (two MMA row groups)
constexpr int kDPitch = 16;              // bytes per row of a d stage (2 x 8)
constexpr int kXPitch = 1040;            // bytes per token row of an activation box (130 x 8)
constexpr int kSmemBudget = 227 * 1024;

// The stage shape for kNT token tiles of 8. Up to 16 tokens a stage holds 8
// super-blocks and 16 consumer warps (super-block x row group) take them.
// For 17..32 tokens (kNT = 3 or 4) the activation rows of 8 super-blocks would not
// fit twice in shared memory, so a stage holds 4 super-blocks for 8 consumer
// warps, each of which forms the MMAs of all four token tiles on one weight
// fragment (more registers a warp: 9 warps a CTA instead of 17).
template <int kNT>
struct Shape {
  static constexpr int kSbs = kNT <= 2 ? 8 : 4;     // super-blocks per stage
  static constexpr int kCW = 2 * kSbs;              // consumer warps
  static constexpr int kThreads = 32 * (kCW + 1);   // + one producer warp
  static constexpr int kQPitch = 192 * kSbs + 16;   // bytes per row of a qlh stage (1552 / 784)
  static constexpr int kScPitch = 16 * kSbs + 16;   // bytes per row of an sc stage (144 / 80)
  static constexpr int kXBoxes = kSbs / 4;          // activation boxes of 1024 (+16) bytes a token
  static constexpr int kRedTok = kNT <= 2 ? 16 : 8 * kNT;  // token columns of the final sums
  // the final sums [kSbs][kRedTok][kRedPitch]: rows contiguous with a pitch of
  // 36 words, so that the fragment stores (8 rows x 4 token pairs) and the
  // row-order reads of the final addition are free of bank conflicts
  static constexpr int kRedPitch = kMaxR + 4;
  static constexpr int kRedBytes = kSbs * kRedTok * kRedPitch * 4;
};

enum : uint32_t { kSiteEmpty = 21, kSiteFull = 22 };

struct Geo {  // byte offsets of one stage's regions and the stage size, for R rows, XR tokens
  int sc, d, x0, x1, da, stage;
};
__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }
template <int kNT>
__host__ __device__ inline Geo stage_geo(int R) {
  using S = Shape<kNT>;
  constexpr int XR = 8 * kNT;  // token rows of an activation stage
  Geo g;
  g.sc = align128(R * S::kQPitch);
  g.d = align128(g.sc + R * S::kScPitch);
  g.x0 = align128(g.d + R * kDPitch);
  g.x1 = S::kXBoxes == 2 ? align128(g.x0 + XR * kXPitch) : g.x0;
  g.da = align128(g.x1 + XR * kXPitch);
  g.stage = align128(g.da + 8 * S::kSbs * XR * 4);  // da of the stage's chunks x XR tokens
  return g;
}
template <int kNT>
size_t smem_bytes(int R, int ns) {
  return 1024 + (size_t)ns * stage_geo<kNT>(R).stage + Shape<kNT>::kRedBytes + 256;
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

constexpr uint32_t kH2_1056 = 0x64206420u;  // (1056, 1056) as f16x2

// The four 6-bit codes (one per byte) of sub-block j (0..7 of a half) at this
// lane's positions: the low (j < 4) or high nibbles of ql word w and the
// 2-bit field j / 2 of qh word q, moved to bits 4-5.
__device__ __forceinline__ uint32_t codes(uint32_t w, uint32_t q, int j) {
  const uint32_t lo = (j < 4 ? w : w >> 4) & 0x0F0F0F0Fu;
  const int f = j >> 1;
  const uint32_t hi = (f < 2 ? q << (4 - 2 * f) : q >> (2 * f - 4)) & 0x30303030u;
  return lo | hi;
}
// Codes of bytes (kOdd, kOdd + 2) of `code` as the binary16 pair code - 32:
// 1024 + code (exponent byte 0x64 placed above each code byte) minus 1056.
template <int kOdd>
__device__ __forceinline__ uint32_t code_pair(uint32_t code) {
  const uint32_t v = __byte_perm(code, 0x64u, kOdd ? 0x4341u : 0x4240u);
  return hsub2u(v, kH2_1056);
}

__device__ __forceinline__ float sc_of(const uint4& v, int s) {  // signed byte s of 16
  const uint32_t w = s < 4 ? v.x : s < 8 ? v.y : s < 12 ? v.z : v.w;
  return (float)(int)(int8_t)(w >> (8 * (s & 3)));
}

template <int kCW>
__device__ __forceinline__ void bar_consumers() {  // the kCW consumer warps only
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kCW) : "memory");
}

template <int kNT, bool kPartials>
__global__ void __launch_bounds__(Shape<kNT>::kThreads, 1)
    mmq_skinny_mma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmS,
                          const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmA, int M, int K, int N, int R, int units,
                          int ns, int ldda, float* __restrict__ Y, int ldy, int32_t* __restrict__ partials,
                          int32_t* __restrict__ chunks, unsigned int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using S = Shape<kNT>;
  constexpr int kSbs = S::kSbs, kCW = S::kCW, kRedTok = S::kRedTok;
  const Geo geo = stage_geo<kNT>(R);
  float* red = reinterpret_cast<float*>(smem + (size_t)ns * geo.stage);  // [kSbs][kRedTok][kRedPitch]
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + S::kRedBytes);
  uint64_t* empty = full + kMaxNS;
  int* abort_word = reinterpret_cast<int*>(empty + kMaxNS);
  volatile int* abort_flag = abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = K / 256, nst = (nsb + kSbs - 1) / kSbs, nc = K / 32, ns16 = K / 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmS);
      tma_prefetch_desc(&tmD);
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmA);
      const uint32_t tx = (uint32_t)R * (S::kQPitch + S::kScPitch + kDPitch) +
                          (uint32_t)S::kXBoxes * (uint32_t)N * kXPitch +
                          (uint32_t)(8 * kSbs) * (uint32_t)ldda * 4u;
      int gs = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        for (int st = 0; st < nst; ++st, ++gs) {
          const int slot = gs % ns;
          if (!(ok = mbar_wait_bounded(&empty[slot], ((gs / ns) & 1) ^ 1, abort_flag, status,
                                       kSiteEmpty)))
            break;
          uint8_t* b = smem + (size_t)slot * geo.stage;
          mbar_arrive_expect_tx(&full[slot], tx);
          // x coordinates in 8-byte units, each a multiple of two (16 bytes)
          tma_load_2d(b, &tmQ, &full[slot], 24 * kSbs * st, u * R);
          tma_load_2d(b + geo.sc, &tmS, &full[slot], 2 * kSbs * st, u * R);
          // d: 16 bytes (8 super-blocks) from the even 8-byte unit at or
          // below the stage's first super-block; the stage's own d values
          // sit at byte 2 * (kSbs * st % 8) of each row
          tma_load_2d(b + geo.d, &tmD, &full[slot], (kSbs * st / 4) & ~1, u * R);
          // the stage's 256 * kSbs activation bytes of each token, as boxes
          // of 1024 (+16) bytes per token row
          tma_load_2d(b + geo.x0, &tmX, &full[slot], 32 * kSbs * st, 0);
          if (S::kXBoxes == 2) tma_load_2d(b + geo.x1, &tmX, &full[slot], 32 * kSbs * st + 128, 0);
          // the activation scales of the stage's 8 * kSbs chunks, [chunk][ldda]
          tma_load_2d(b + geo.da, &tmA, &full[slot], 0, 8 * kSbs * st);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits
        volatile int no_abort = 0;
        for (int k = (gs > ns ? gs - ns : 0); k < gs; ++k)
          mbar_wait_bounded(&full[k % ns], (k / ns) & 1, &no_abort, status, kSiteFull);
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers --
  // warp (sbw, g): super-block sbw of every stage, rows 16g .. 16g + 15 of the unit
  const int sbw = warp % kSbs, g = warp / kSbs;
  const int gq = lane >> 2, t = lane & 3;
  const int ra = 16 * g + gq, rb = ra + 8;  // this lane's two rows (unit-relative)
  const bool have_a = ra < R, have_b = rb < R, active = 16 * g < R;
  int gs = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int r0 = u * R;
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
        // this lane's ql / qh words of rows ra, rb in the current half block
        // (chunks 0-3 read half 0, chunks 4-7 half 1): [row][word]
        uint32_t ql[2][4], qh[2][2];
        const uint8_t* pa = b + (size_t)ra * S::kQPitch + 192 * sbw + 4 * t;
        const uint8_t* pb = b + (size_t)rb * S::kQPitch + 192 * sbw + 4 * t;
        auto load_half = [&](int h) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            ql[0][j] = have_a ? lds32(pa + 96 * h + 16 * j) : 0u;
            ql[1][j] = have_b ? lds32(pb + 96 * h + 16 * j) : 0u;
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            qh[0][j] = have_a ? lds32(pa + 96 * h + 64 + 16 * j) : 0u;
            qh[1][j] = have_b ? lds32(pb + 96 * h + 64 + 16 * j) : 0u;
          }
        };
        const uint4 sca4 = have_a ? *reinterpret_cast<const uint4*>(b + geo.sc + (size_t)ra * S::kScPitch + 16 * sbw)
                                  : make_uint4(0, 0, 0, 0);
        const uint4 scb4 = have_b ? *reinterpret_cast<const uint4*>(b + geo.sc + (size_t)rb * S::kScPitch + 16 * sbw)
                                  : make_uint4(0, 0, 0, 0);
        const int dsb = 2 * ((kSbs * st) % 8 + sbw);  // byte of this super-block's d
        const float d_a = have_a ? __half2float(*reinterpret_cast<const __half*>(
                                       b + geo.d + (size_t)ra * kDPitch + dsb))
                                 : 0.0f;
        const float d_b = have_b ? __half2float(*reinterpret_cast<const __half*>(
                                       b + geo.d + (size_t)rb * kDPitch + dsb))
                                 : 0.0f;
        // f32 pairs over the tokens (t0, t0 + 1) of a lane: [token tile][row a, b]
        float2 sbs[kNT][2];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) sbs[nt][0] = sbs[nt][1] = make_float2(0.0f, 0.0f);

        // activation words of a chunk (two sub-blocks, each token group) from
        // the stage's activation boxes (tokens past N were filled with 0),
        // read one chunk ahead of their use
        const uint8_t* xs = b + (sbw < 4 ? geo.x0 : geo.x1) + 256 * (sbw & 3) + 4 * t;
        auto load_x = [&](int c8, uint32_t (&xw)[2][kNT]) {
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
              xw[e][nt] = lds32(xs + (size_t)(8 * nt + gq) * kXPitch + 32 * c8 + 16 * e);
        };
        uint32_t xcur[2][kNT], xnxt[2][kNT];
        load_x(0, xcur);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const int c = 8 * sb + c8;  // chunk
          if (c8 == 0 || c8 == 4) load_half(c8 >> 2);
          if (c8 < 7) load_x(c8 + 1, xnxt);
          float2 S[kNT][2];
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) S[nt][0] = S[nt][1] = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int s16 = 2 * c8 + e, j = s16 & 7;
            uint32_t a[4];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const uint32_t code = codes(ql[rr][j & 3], qh[rr][j & 1], j);
              a[rr] = code_pair<0>(code);      // codes 4t, 4t + 2
              a[2 + rr] = code_pair<1>(code);  // codes 4t + 1, 4t + 3
            }
            const float sa = sc_of(sca4, s16), sbv = sc_of(scb4, s16);
            const float2 sa2 = make_float2(sa, sa), sb2 = make_float2(sbv, sbv);
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
              const uint32_t wb = xcur[e][nt] ^ 0x80808080u;
              const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
              float P[4];
              mma_f16(P, a, x_pair<0>(wb), x_pair<1>(wb), z);
              if (kPartials && partials) {
                // P of sub-block 16 sb + s16 (an exact integer in f32)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int rl = (i < 2) ? ra : rb, tk = 8 * nt + 2 * t + (i & 1);
                  if (rl < R && r0 + rl < M && tk < N)
                    partials[((size_t)tk * M + r0 + rl) * (size_t)ns16 + 16 * sb + s16] =
                        (int32_t)P[i];
                }
              }
              // sc * P and their sum over the chunk are exact in f32 (< 2^24);
              // one two-lane FMA per row (each lane rounds as fmaf does)
              S[nt][0] = __ffma2_rn(sa2, make_float2(P[0], P[1]), S[nt][0]);
              S[nt][1] = __ffma2_rn(sb2, make_float2(P[2], P[3]), S[nt][1]);
            }
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int t0 = 8 * nt + 2 * t;
            // da of tokens (t0, t0 + 1): the stage's da rows have ldda (a
            // multiple of 4) columns and 8 * kNT >= ldda, so the pair stays in
            // the region; a column at or past N carries whatever the plane
            // holds there and only reaches lanes of tokens that are never stored
            const float2 d01 = *reinterpret_cast<const float2*>(
                reinterpret_cast<const float*>(b + geo.da) + (8 * sbw + c8) * ldda + t0);
            sbs[nt][0] = __ffma2_rn(d01, S[nt][0], sbs[nt][0]);
            sbs[nt][1] = __ffma2_rn(d01, S[nt][1], sbs[nt][1]);
            if (kPartials && chunks) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int rl = (i < 2) ? ra : rb, tk = t0 + (i & 1);
                const float2 v = S[nt][i >> 1];
                if (rl < R && r0 + rl < M && tk < N)
                  chunks[((size_t)tk * M + r0 + rl) * (size_t)nc + c] = (int32_t)((i & 1) ? v.y : v.x);
              }
            }
          }
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) xcur[e][nt] = xnxt[e][nt];
        }
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          acc[nt][0] = fmaf(d_a, sbs[nt][0].x, acc[nt][0]);
          acc[nt][1] = fmaf(d_a, sbs[nt][0].y, acc[nt][1]);
          acc[nt][2] = fmaf(d_b, sbs[nt][1].x, acc[nt][2]);
          acc[nt][3] = fmaf(d_b, sbs[nt][1].y, acc[nt][3]);
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
          for (int w = 0; w < kSbs; ++w) y += red[(w * kRedTok + tk) * S::kRedPitch + row];
          Y[(size_t)tk * ldy + r0 + row] = y;
        }
      }
    }
    bar_consumers<kCW>();
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;
std::once_flag g_encode_once;

CUresult encode(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode_fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode_fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int kNT, bool P>
cudaError_t launch_nt(const uint8_t* plane, int M, int K, const int8_t* Xq, const float* da,
                      int ldda, int N, float* Y, int ldy, Debug dbg, unsigned int* status,
                      cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  // R rows per unit, at most kMaxR, units in whole waves over the SMs
  const long long waves = ((long long)M + (long long)kMaxR * sms - 1) / ((long long)kMaxR * sms);
  const int R = (int)(((long long)M + waves * sms - 1) / (waves * sms));
  const int units = (M + R - 1) / R;
  const PlaneGeom g = plane_geom(M, K);
  using S = Shape<kNT>;
  // the scales of the N tokens: dcols columns of the [K/32][ldda] plane (a
  // token group of a larger call starts at a column that is a multiple of
  // 4, so the box never reaches past the plane's rows)
  const int dcols = (N + 3) & ~3;
  CUtensorMap mq, ms, md, mx, ma;
  if (!g_encode_fn) return cudaErrorInitializationError;
  // the activation boxes hold the N token rows (the rows past N in shared
  // memory are never stored from)
  if (encode(&mq, plane + g.qlh_off, g.qlh_row / 8, (uint64_t)M, g.qlh_row, S::kQPitch / 8,
             (uint32_t)R) != CUDA_SUCCESS ||
      encode(&ms, plane + g.sc_off, (uint64_t)K / 128, (uint64_t)M, (uint64_t)K / 16,
             S::kScPitch / 8, (uint32_t)R) != CUDA_SUCCESS ||
      encode(&md, plane + g.d_off, g.d_row / 8, (uint64_t)M, g.d_row, kDPitch / 8, (uint32_t)R) !=
          CUDA_SUCCESS ||
      encode(&mx, Xq, (uint64_t)K / 8, (uint64_t)N, (uint64_t)K, kXPitch / 8, (uint32_t)N) !=
          CUDA_SUCCESS ||
      encode_f32(&ma, da, (uint64_t)dcols, (uint64_t)K / 32, (uint64_t)ldda * 4, (uint32_t)dcols,
                 8 * S::kSbs) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int ns = smem_bytes<kNT>(R, 3) <= (size_t)kSmemBudget ? 3 : 2;
  if (smem_bytes<kNT>(R, ns) > (size_t)kSmemBudget) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  return launch_pdl(mmq_skinny_mma_kernel<kNT, P>, dim3(grid), dim3(S::kThreads),
                    smem_bytes<kNT>(R, ns), s, mq, ms, md, mx, ma, M, K, N, R, units, ns,
                    dcols, Y, ldy, dbg.partials, dbg.chunk_sums, status);
}

}  // namespace

CUresult skinny_tensor_map(CUtensorMap* map, bool f32, const void* base, uint64_t inner,
                           uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                           uint32_t box_outer) {
  if (!g_encode_fn) return CUDA_ERROR_NOT_INITIALIZED;
  return f32 ? encode_f32(map, base, inner, outer, row_bytes, box_inner, box_outer)
             : encode(map, base, inner, outer, row_bytes, box_inner, box_outer);
}

// Raises the dynamic shared-memory limit of every instantiation and looks up
// the tensor-map encoder; once per device.
cudaError_t mmq_skinny_mma_prepare() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode_fn) return cudaErrorInitializationError;
  const int bytes = kSmemBudget;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(mmq_skinny_mma_kernel<1, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_mma_kernel<1, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_mma_kernel<2, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_mma_kernel<2, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_mma_kernel<4, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_mma_kernel<3, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) ||
      (e = cudaFuncSetAttribute(mmq_skinny_mma_kernel<3, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)))
    return e;
  return cudaFuncSetAttribute(mmq_skinny_mma_kernel<4, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_mmq_skinny_mma(const uint8_t* plane, int M, int K, const int8_t* Xq,
                                  const float* da, int ldda, int N, float* Y, int ldy,
                                  Debug dbg, unsigned int* status, cudaStream_t s) {
  if (N <= 8)
    return dbg.any() ? launch_nt<1, true>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s)
                     : launch_nt<1, false>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s);
  if (N <= 16)
    return dbg.any() ? launch_nt<2, true>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s)
                     : launch_nt<2, false>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s);
  if (N > 32) return cudaErrorInvalidValue;
  // 17..24 tokens on three token tiles (22.9 us against 26.9 on four, 4096 x 11008)
  if (N <= 24)
    return dbg.any() ? launch_nt<3, true>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s)
                     : launch_nt<3, false>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s);
  return dbg.any() ? launch_nt<4, true>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s)
                   : launch_nt<4, false>(plane, M, K, Xq, da, ldda, N, Y, ldy, dbg, status, s);
}

}  // namespace q6
