// q6_K x int8 prefill GEMM on the 5th-generation tensor cores (sm_103a).
//
// What it computes ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1-2.4):
//     Y[n][m] = sum over super-blocks b of d[m][b] *
//               sum over 32-element chunks c of b of da[n][c] * S[n][m][c],
//     S[n][m][c] = sum over the chunk's two 16-element sub-blocks s of
//                  sc[m][s] * P[n][m][s],   P = sum (q - 32) * xq,
// with no dmin term. The pages form P per sub-block with int8 mma.sync and
// rescale each with d * sc and da in f32 (KSPLIT=2 pairs per chunk).
//
// sm_103a has no tcgen05 int8 MMA. Here the integer chunk sum S is formed
// exactly on the kind::f16 tensor cores with f32 accumulation in TMEM: the
// activations are the binary16 plane of xq (-127..127), and the weights are
// the two binary16 planes W_hi = 16*floor(sc/16)*(q-32) and
// W_lo = (sc mod 16)*(q-32) (see expand.cu), so W_hi + W_lo = sc*(q-32) with
// both parts exact. Per chunk, four K=16 MMAs (hi and lo of each sub-block)
// accumulate into one fresh TMEM accumulator. Every partial sum along the way
// is an integer of magnitude at most 32 * 128 * 32 * 127 = 16,646,144 < 2^24,
// so the f32 accumulator holds S exactly. Folding sc into the operand leaves
// one f32 word per (n, m, chunk) for the epilogue instead of two, at twice the
// MMA work (the tensor pipe has the room; the CUDA-core rescale is the
// bottleneck of the per-sub-block form).
//
// Tile: 128 tokens (MMA M, TMEM lanes) x 128 weight rows (MMA N, TMEM
// columns). Tokens on the lanes make da a per-thread scalar; d is per column
// and constant over a super-block, so the epilogue keeps two f32 register
// accumulators per (n, m):  Sb += da * S  per chunk, and  Y += d * Sb  per
// super-block (one FFMA2 per two words per chunk, plus 1/8 of that).
//
// Persistent CTAs (one per SM) walk work units u = blockIdx.x, += gridDim.x.
// A unit is a tile t -> (weight band t / NT, token tile t % NT), so CTAs
// running at the same time share weight bands and read every activation
// tile; when the last round of tiles would leave more than half of the SMs
// idle, each of its tiles becomes two units over the two halves of its
// super-blocks, which add into Y after a small kernel has zeroed those tiles.
// Shared-memory rings filled by TMA run continuously across units:
//   operand ring (4 stages x 64 of K): Xh, W_hi, W_lo tiles, 128 rows x 128 B
//          each, 128-byte swizzled; freed by the epilogue once it has seen
//          the commit of the stage's MMAs.
//   scale ring (3 stages x one super-block): da [8 chunks][128 tokens] and
//          d [128 rows]; freed by the epilogue.
// TMEM: two slots of two 128-column accumulator buffers; operand stage g (two
// chunks) uses slot g % 2. The MMAs of a stage signal the epilogue with one
// tcgen05.commit on an mbarrier; the epilogue hands the slot back with a
// hardware named barrier (below).
// Warp roles (12 warps; warpgroup 0 gives registers to warpgroups 1-2):
//   0      TMA producer for both rings.
//   1      TMEM allocation (512 columns).
//   1-2    issuer warp w owns TMEM slot w - 1 and walks every other operand
//          stage; its lane 0 issues the stage's MMAs and the commit.
//   3      idle (its registers go to the epilogue).
//   4-11   epilogue: warp w owns TMEM lanes 32(w%4).. (32 tokens) and 64
//          weight-row columns. Per chunk it loads its 64 words and does the
//          math; the slot is handed back as soon as the stage's second chunk
//          is in registers.
// Every mbarrier wait is bounded (see q6_internal.cuh).
//
// q4_K ("r18: Load-time B pre-expansion", Sec. 1 and 3.2; "r38 -- q6_K
// BT-style raw-byte mma kernel", Sec. 2.2) uses the same pipeline with one
// operand plane sc * q (at most 945, exact in binary16: two MMAs per chunk)
// and a second term, - sum over chunks of (da * S) * (dmin * m). Done in the
// epilogue, that term costs one FMA per (token, row, chunk) with dmin * m
// broadcast to every lane from shared memory, 4 bytes per wavefront: more
// shared-memory wavefronts than the tensor pipe has cycles. Here it is a
// contraction over the K/32 chunks on the tensor cores instead: after a
// unit's chunk stages come its min stages (min_stages below), kind::tf32
// MMAs of the hi/lo pairs of us = da * S and mv = dmin * m into a TMEM
// buffer that the epilogue subtracts from Y, one word per (token, row) per
// pair of super-blocks.
#include "q6_quant.cuh"

namespace q6 {
namespace {

constexpr int BT = 128, BW = 128;  // tokens, weight rows per tile
constexpr int KB = 64, SB = 4;     // operand ring: K per stage, stages (one super-block)
constexpr int SS = 3;              // scale ring stages (one super-block each)
constexpr int kThreads = 384;      // launched with 168 registers per thread
constexpr int kCtlRegs = 24, kEpiRegs = 240;  // 128 * 24 + 256 * 240 == 384 * 168
static_assert(128 * kCtlRegs + 256 * kEpiRegs <= kThreads * 168, "register split");
constexpr int kEpiWarp0 = 4, kNumEpiWarps = 8;
constexpr int kNumIssuers = 2;  // MMA-issuing threads: lane 0 of warps 1-2
constexpr int kTmemCols = 512, kBufCols = 128;
constexpr int kNumSlots = 2;  // TMEM slots of two chunk buffers (one operand stage) each

// Weight formats: q6_K (two operand planes W_hi, W_lo) and q4_K (one plane
// sc * q, and the min term from the tf32 min stages below).
enum : int { kFmtQ6 = 0, kFmtQ4 = 1 };

// Shared-memory layout per format. Operand stage: Xh, W_hi (or sc * q) and,
// for q6_K, W_lo tiles of 128 rows x 128 bytes; a q4_K min stage holds the
// block-sum pairs of 128 tokens and the dmin * m pairs of 128 weight rows for
// two super-blocks in the Xh and W slots (32 f32 = 128 bytes a row). Scale
// stage (one super-block): da [8 chunks][128 tokens] and d [128 rows].
template <int kFmt>
struct Lay {
  static constexpr int kOpX = 0, kOpWhi = BT * 128, kOpWlo = kOpWhi + BW * 128;
  static constexpr int kOpStage = (kFmt == kFmtQ6 ? kOpWlo + BW * 128 : kOpWlo);  // 48 / 32 KB
  static constexpr int kScDa = 0, kScD = 8 * BT * 4, kScUs = kScD + BW * 4;
  static constexpr int kScStage = kScUs;  // 4.5 KB
  static constexpr int kRingS = SB * kOpStage;  // the scale ring follows the operand ring
  static constexpr int kXStage = kRingS + SS * kScStage;  // fused quantiser staging, 16 KB
  static constexpr int kRingsBytes = kRingS + SS * kScStage;
  static_assert(kOpStage % 1024 == 0, "operand stages must keep 1024-byte alignment");
  static_assert(kScStage % 128 == 0, "scale stages must keep 128-byte alignment");
};
static_assert(SB * KB == 256, "the epilogue frees operand slot pp of each super-block");

enum : uint32_t { kSiteSEmpty = 1, kSiteSFull = 2, kSiteBEmpty = 3, kSiteBFull = 4,
                  kSiteTFull = 6, kSiteDrain = 8 };

// TMEM slot ts goes back from the epilogue to its issuer through hardware
// named barrier kBarSlot0 + ts: the 8 epilogue warps arrive (bar.arrive, no
// wait) and the issuing warp waits (bar.sync), 288 threads per phase. This
// takes the place of an mbarrier phase on the slot's round trip (MMAs,
// commit, epilogue loads, hand-back), which bounds the kernel; measured on
// GB300 the ffn_down GEMM goes from 0.457 to 0.447 ms. bar.sync has no
// time-out, so the k-th wait of an issuer must meet the k-th arrival of the
// epilogue on that slot, also after a bounded wait has been given up: then
// neither side leaves its walk early; the issuer stops issuing, the epilogue
// stops waiting and writing Y, and both still walk every operand stage of the
// CTA's units (one arrival and one wait per stage, as in a normal run), while
// all other waits return at once. Handing back the stages still ahead in one
// burst instead could put two stages' arrivals into one barrier phase and
// leave an issuer's last wait short of arrivals.
constexpr int kBarSlot0 = 1;  // named barriers 1, 2 (0 is __syncthreads)
constexpr int kSlotBarThreads = 32 * (kNumEpiWarps + 1);
__device__ __forceinline__ void slot_bar_sync(int ts) {
  asm volatile("bar.sync %0, %1;" ::"r"(kBarSlot0 + ts), "n"(kSlotBarThreads) : "memory");
}
__device__ __forceinline__ void slot_bar_arrive(int ts) {
  asm volatile("bar.arrive %0, %1;" ::"r"(kBarSlot0 + ts), "n"(kSlotBarThreads) : "memory");
}

struct Bars {
  uint64_t s_full[SS], s_empty[SS];
  uint64_t b_full[SB], b_empty[SB];
  uint64_t tfull[kNumSlots], drain;
  uint32_t tmem_base;
  int abort;
};

// Bytes of shared memory past the rings: the fused quantiser's staging rows
// (128 rows of 128 bytes), then the barriers.
template <bool kFuseX>
constexpr int extra_bytes() { return kFuseX ? BT * 128 : 0; }
template <int kFmt, bool kFuseX = false>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Lay<kFmt>::kRingsBytes + extra_bytes<kFuseX>() + sizeof(Bars);
}
static_assert(smem_bytes<kFmtQ6>() <= 232448 && smem_bytes<kFmtQ4>() <= 232448 &&
                  smem_bytes<kFmtQ6, true>() <= 232448,
              "shared memory budget");
static_assert(Lay<kFmtQ6>::kXStage % 128 == 0, "staging rows keep 16-byte alignment");

// Work units: units 0 .. Tw-1 are whole tiles; when the last round of tiles
// would leave more than half the CTAs idle, each of its tiles is split into
// two units over the two halves of its super-blocks (units Tw + 2i and
// Tw + 2i + 1 for tile Tw + i), which add their sums into a zeroed Y. When
// the tiles fill at most half of the SMs at all (few tokens or rows), every
// tile is instead split into `splits` K parts (unit u: tile u / splits, part
// u % splits), which store their sums to a partial-sum buffer that a second
// kernel adds in a fixed order.
struct Unit {
  int t, sb0, sb1;
  bool split;  // one of the two halves of a tile of the split last round
  int part;    // K part (splits > 1)
};
__device__ __forceinline__ Unit unit_of(int u, int Tw, int nsb, int splits) {
  if (splits > 1) {
    const int t = u / splits, j = u - t * splits;
    return Unit{t, nsb * j / splits, nsb * (j + 1) / splits, false, j};
  }
  if (u < Tw) return Unit{u, 0, nsb, false, 0};
  const int i = u - Tw, half = i & 1;
  return Unit{Tw + (i >> 1), half ? nsb / 2 : 0, half ? nsb : nsb / 2, true, half};
}

// Zeroes the Y blocks of the split tiles: block (i, y) clears rows 32y..32y+31
// of tile Tw + i, four columns per store where Y allows it.
__global__ void __launch_bounds__(256) zero_split_tiles_kernel(float* __restrict__ Y, int ldy,
                                                               int M, int N, int Tw, int y_vec4) {
  const int NT = (N + BT - 1) / BT;
  const int t = Tw + blockIdx.x;
  const int m0 = (t / NT) * BW, n0 = (t % NT) * BT + 32 * blockIdx.y;
  const int mw = min(BW, M - m0), nw = min(32, N - n0);
  if (nw <= 0) return;
  const int mv = y_vec4 ? (mw & ~3) : 0;  // columns cleared four at a time (m0 % 4 == 0)
  for (int i = threadIdx.x; i < nw * (mv / 4); i += blockDim.x) {
    const int r = i / (mv / 4), c = 4 * (i - r * (mv / 4));
    *reinterpret_cast<float4*>(Y + (size_t)(n0 + r) * ldy + m0 + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i = threadIdx.x; i < nw * (mw - mv); i += blockDim.x) {
    const int r = i / (mw - mv), c = mv + (i - r * (mw - mv));
    Y[(size_t)(n0 + r) * ldy + m0 + c] = 0.0f;
  }
}

// Y = the sum of the K parts, added in part order (so the result does not
// depend on which part finished first): part is [splits][N][M].
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part,
                                                            int splits, int N, int M,
                                                            float* __restrict__ Y, int ldy) {
  const long long total = (long long)N * M;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i / M), m = (int)(i - (long long)n * M);
    float v = 0.0f;
    for (int j = 0; j < splits; ++j) v += part[(size_t)j * total + i];
    Y[(size_t)n * ldy + m] = v;
  }
}

// sb[j] (+)= (da, da) * S[j] for 32 columns (16 pairs).
template <bool kFirst>
__device__ __forceinline__ void chunk_fma(float2* sb, const uint32_t (&p)[32], float da) {
  const float2 dav = make_float2(da, da);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 s = make_float2(__uint_as_float(p[2 * j]), __uint_as_float(p[2 * j + 1]));
    sb[j] = kFirst ? __fmul2_rn(dav, s) : __ffma2_rn(dav, s, sb[j]);
  }
}

// acc[j] -= T[j] for 32 columns (16 pairs): the min term of a q4_K min stage.
__device__ __forceinline__ void sub_words(float2* acc, const uint32_t (&t)[32]) {
  const float2 neg = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    acc[j] = __ffma2_rn(neg, make_float2(__uint_as_float(t[2 * j]), __uint_as_float(t[2 * j + 1])),
                        acc[j]);
}

// q4_K min stages of a unit. The min term of super-blocks sb0 .. sb1-1,
//   sum over their chunks c of us[n][c] * mv[m][c]
// (us = da * S, mv = dmin * m), runs on the tensor cores: one min stage per
// pair of super-blocks {2g, 2g+1} that the unit touches, whose tiles hold the
// hi/lo pairs of both (see Lay); per super-block four K = 8 kind::tf32 MMAs
// (hi*hi, hi*lo, lo*hi, lo*lo) into one TMEM buffer, which the epilogue
// subtracts from Y. mv has at most 17 significant bits, so its pair is exact;
// us's pair is within 2^-21 |us|; each product of tf32 values is exact in
// f32. The count is padded to a multiple of 4 with empty stages (no copies,
// no MMAs) so that every unit keeps a multiple of four operand stages.
__device__ __forceinline__ int min_groups(const Unit& w) {
  return ((w.sb1 - 1) >> 1) - (w.sb0 >> 1) + 1;
}
__device__ __forceinline__ int min_stages(const Unit& w) { return (min_groups(w) + 3) & ~3; }

// ---------------------------------------------------- fused quantiser ---
// With kFuseX the epilogue warps also produce the A operand: epilogue thread
// (tok, colh) quantises one 32-element block of each operand stage four
// stages ahead of the one it consumes, token n = n0 + tok, elements k0 ..
// k0 + 31, with the standalone quantiser's arithmetic (q6_quant.cuh), so the
// codes and scales are bit for bit those of q8_quantize_act.
// fx_issue starts the copy of the warp's 32 blocks (tokens 32 q .. 32 q +
// 31, q = tok / 32, elements k0 .. k0 + 31) into the staging rows of their
// threads: row t of the target stage's Xh tile (colh 0) or of the 16 KB
// staging rows after the scale ring (colh 1), 16-byte unit i at unit
// i ^ (t % 8) so that a warp's rows spread over all banks. Eight lanes copy
// one 128-byte row, four rows per instruction, so each instruction touches
// four cache lines (with one row per thread it touched 32, and the L1 tag
// stage took more cycles than the GEMM's whole stage). Rows n >= N are
// zero-filled, which gives the codes and scale of a zero block, as the
// separate path's zero-filled tiles do.
constexpr int kBarFx = 3;  // named barrier of the 256 epilogue threads

__device__ __forceinline__ void fx_issue(uint32_t stg0, int tok, const float* __restrict__ Xf,
                                         int ldx, int N, int n0w, int k0) {
  const int lane = tok & 31, piece = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + (lane >> 3);  // row of the warp's 32
    const int n = n0w + r;
    const bool valid = n < N;
    const char* src =
        reinterpret_cast<const char*>(Xf + (size_t)(valid ? n : 0) * ldx + k0) + 16 * piece;
    const uint32_t dst = stg0 + (uint32_t)(r * 128) + (uint32_t)((piece ^ (r & 7)) << 4);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16u : 0u)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// fx_finish waits for the copy and reads the block; after all 256 epilogue
// threads have read theirs (the codes of row tok overwrite the staging of
// thread (tok, 0)) it writes the block's binary16 codes into the
// 128-byte-swizzled Xh tile (16-byte unit j of row tok at unit j ^ (tok % 8))
// and its scale, and makes the codes visible to the tensor core.
__device__ __forceinline__ void fx_finish(const uint8_t* stg, uint8_t* xh, int tok, int colh,
                                          float* da_out) {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncwarp();  // the row was copied by eight lanes of this warp
  float4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = reinterpret_cast<const float4*>(stg)[i ^ (tok & 7)];
  asm volatile("bar.sync %0, %1;" ::"n"(kBarFx), "n"(32 * kNumEpiWarps) : "memory");
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    a = fmaxf(a, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  const float d = __fdiv_rn(a, 127.0f);
  const float r = recip_or_zero(d);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 h;
    quant8h(v[2 * i], v[2 * i + 1], d, r, h);
    const int j = 4 * colh + i;
    *reinterpret_cast<uint4*>(xh + tok * 128 + ((j ^ (tok & 7)) << 4)) = h;
  }
  *da_out = d;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The exact integers of 32 columns of a chunk accumulator, to the debug
// output at out[(n * M + m) * stride + off] (off = c * mul + add).
template <bool kPartials>
__device__ __forceinline__ void dump_partials(int32_t* __restrict__ out, int M, int N,
                                              int stride, int n, int m_first, int off,
                                              const uint32_t (&p)[32]) {
  if (kPartials) {
    if (n < N) {
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
        const int m = m_first + j;
        if (m < M) out[((size_t)n * M + m) * (size_t)stride + off] = (int32_t)__uint_as_float(p[j]);
      }
    }
    __syncwarp();
  }
}

template <int kFmt, bool kPartials, bool kFuseX>
__global__ void __launch_bounds__(kThreads, 1)
    mmq_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWhi,
                  const __grid_constant__ CUtensorMap tmWlo, const __grid_constant__ CUtensorMap tmDa,
                  const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmUs,
                  const __grid_constant__ CUtensorMap tmMv, int M, int K, int N, int Tw, int U,
                  float* __restrict__ Y, int ldy, int y_vec4, int32_t* __restrict__ partials,
                  int p_stride, int p_mul, int p_add, int write_y,
                  const float* __restrict__ Xf, int ldx, int splits, float* __restrict__ part,
                  unsigned int* __restrict__ status) {
  using L = Lay<kFmt>;
  constexpr bool kQ4 = kFmt == kFmtQ4;
  static_assert(!(kFuseX && kQ4), "the fused quantiser serves the q6_K kernel");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kRingsBytes + extra_bytes<kFuseX>());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = (N + BT - 1) / BT;
  const int nsb = K / 256;  // super-blocks per tile
  volatile int* abort_flag = &bars->abort;

  if (threadIdx.x == 0) {
    // with the fused quantiser the epilogue warps also fill da and Xh, and
    // each arrives once per scale stage and per operand stage
    constexpr int kFillers = 1 + (kFuseX ? kNumEpiWarps : 0);
    for (int s = 0; s < SS; ++s) {
      mbar_init(&bars->s_full[s], kFillers);
      mbar_init(&bars->s_empty[s], kNumEpiWarps);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&bars->b_full[s], kFillers);
      mbar_init(&bars->b_empty[s], 1);
    }
    for (int b = 0; b < kNumSlots; ++b) mbar_init(&bars->tfull[b], 1);
    mbar_init(&bars->drain, kNumIssuers);  // one commit per issuer
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    if (!kFuseX) {
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmDa);
    }
    tma_prefetch_desc(&tmWhi);
    tma_prefetch_desc(&tmWlo);
    tma_prefetch_desc(&tmD);
    if (kQ4) {
      tma_prefetch_desc(&tmUs);
      tma_prefetch_desc(&tmMv);
    }
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
        // (with the fused quantiser, da and the Xh tiles come from the epilogue)
        constexpr uint32_t kTxS = (kFuseX ? 0 : 8 * BT * 4) + BW * 4;
        constexpr uint32_t kTxB = ((kFuseX ? 0 : BT) + (kQ4 ? 1 : 2) * BW) * 128;  // and a min stage
        int gs = 0, gk = 0;  // scale / operand stages issued so far
        bool ok = true;
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
          const Unit w = unit_of(u, Tw, nsb, splits);
          const int m0 = (w.t / NT) * BW, n0 = (w.t % NT) * BT;
          for (int sb = w.sb0; sb < w.sb1 && ok; ++sb) {
            {
              const int slot = gs % SS;
              if (!(ok = mbar_wait_bounded(&bars->s_empty[slot], ((gs / SS) & 1) ^ 1, abort_flag,
                                           status, kSiteSEmpty)))
                break;
              uint8_t* st = smem + L::kRingS + slot * L::kScStage;
              mbar_arrive_expect_tx(&bars->s_full[slot], kTxS);
              if (!kFuseX) tma_load_2d(st + L::kScDa, &tmDa, &bars->s_full[slot], n0, 8 * sb);
              tma_load_2d(st + L::kScD, &tmD, &bars->s_full[slot], m0, sb);
              ++gs;
            }
            for (int h = 0; h < 4; ++h) {
              const int kb = 4 * sb + h, slot = gk % SB;
              if (!(ok = mbar_wait_bounded(&bars->b_empty[slot], ((gk / SB) & 1) ^ 1, abort_flag,
                                           status, kSiteBEmpty)))
                break;
              uint8_t* bt = smem + slot * L::kOpStage;
              mbar_arrive_expect_tx(&bars->b_full[slot], kTxB);
              if (!kFuseX) tma_load_2d(bt + L::kOpX, &tmX, &bars->b_full[slot], kb * KB, n0);
              tma_load_2d(bt + L::kOpWhi, &tmWhi, &bars->b_full[slot], kb * KB, m0);
              if (!kQ4) tma_load_2d(bt + L::kOpWlo, &tmWlo, &bars->b_full[slot], kb * KB, m0);
              ++gk;
            }
          }
          if (kQ4) {
            // the unit's min stages: pair group g's 128-byte rows of us and mv
            const int g0 = w.sb0 >> 1, ng = min_groups(w), ns = min_stages(w);
            for (int i = 0; i < ns && ok; ++i) {
              const int slot = gk % SB;
              if (!(ok = mbar_wait_bounded(&bars->b_empty[slot], ((gk / SB) & 1) ^ 1, abort_flag,
                                           status, kSiteBEmpty)))
                break;
              uint8_t* bt = smem + slot * L::kOpStage;
              if (i < ng) {
                mbar_arrive_expect_tx(&bars->b_full[slot], kTxB);
                tma_load_2d(bt + L::kOpX, &tmUs, &bars->b_full[slot], 32 * (g0 + i), n0);
                tma_load_2d(bt + L::kOpWhi, &tmMv, &bars->b_full[slot], 32 * (g0 + i), m0);
              } else {
                mbar_arrive(&bars->b_full[slot]);  // an empty stage: nothing to copy
              }
              ++gk;
            }
          }
        }
        if (!ok) {
          // Let copies already issued land before the CTA exits.
          volatile int no_abort = 0;
          for (int k = (gs > SS ? gs - SS : 0); k < gs; ++k)
            mbar_wait_bounded(&bars->s_full[k % SS], (k / SS) & 1, &no_abort, status, kSiteSFull);
          for (int k = (gk > SB ? gk - SB : 0); k < gk; ++k)
            mbar_wait_bounded(&bars->b_full[k % SB], (k / SB) & 1, &no_abort, status, kSiteBFull);
        }
      }
    } else {
      // --------------------------------------------------------------- MMA --
      // Operand stage g (two chunks) goes to issuer g % kNumIssuers and into
      // TMEM slot g % 2. tcgen05.mma issue stalls until the tensor pipe has
      // room, so while one issuer waits on a barrier or commits, the other
      // keeps the pipe fed. One commit per stage signals both its chunks
      // (an mbarrier hand-off costs about 200 cycles), and the slot comes
      // back once per stage as well (per-chunk hand-backs on two named
      // barriers per slot measured slower: 0.455 against 0.447 ms).
      if (warp <= kNumIssuers) {
        // The whole warp walks the stages (bar.sync wants the warp
        // converged); lane 0 issues. Issuer `me` owns TMEM slot `me`.
        // Once a wait has been given up (ok == false) the issuer issues
        // nothing more but still walks every stage and takes every hand-back,
        // as the epilogue still walks every stage and hands every one back:
        // the named-barrier phases stay paired one to one (bar.sync has no
        // time-out), and every other wait then returns at once.
        constexpr uint32_t idesc = idesc_f16_f32(BT, BW);
        constexpr uint32_t idesc_min = idesc_tf32_f32(BT, BW);
        const int me = warp - 1;
        bool ok = true;
        int gbase = 0;  // global index of the unit's first operand stage
        int uses = 0;   // operand stages walked (issued into my slot)
        for (int u = blockIdx.x; u < U; u += gridDim.x) {
          const Unit w = unit_of(u, Tw, nsb, splits);
          const int nb = 4 * (w.sb1 - w.sb0);  // the unit's chunk stages
          const int nt = nb + (kQ4 ? min_stages(w) : 0);  // and its min stages
          for (int kb = (me - gbase % kNumIssuers + kNumIssuers) % kNumIssuers; kb < nt;
               kb += kNumIssuers) {
            const int gk = gbase + kb;  // global operand stage; gk % 2 == me
            const int slot = gk % SB;
            if (ok && !mbar_wait_warp(&bars->b_full[slot], (gk / SB) & 1, abort_flag, status,
                                      kSiteBFull))
              ok = false;
            // the epilogue has loaded the previous stage out of my slot
            if (uses++ > 0) slot_bar_sync(me);
            tc_fence_after();
            if (lane == 0 && ok && kQ4 && kb >= nb) {
              // a min stage: pair group g = sb0/2 + (kb - nb); super-block
              // 2g + h has its hi parts at byte 64 h and its lo parts at
              // 64 h + 32 of each row (descriptor start + 4 h, + 4 h + 2)
              const int g = (w.sb0 >> 1) + (kb - nb);
              const uint8_t* bt = smem + slot * L::kOpStage;
              const uint32_t udesc = sw128_desc_lo(smem_u32(bt + L::kOpX));
              const uint32_t vdesc = sw128_desc_lo(smem_u32(bt + L::kOpWhi));
              const uint32_t d_tmem = tmem + (uint32_t)(2 * me * kBufCols);
              uint32_t acc_on = 0;
              if (kb - nb < min_groups(w)) {
                for (int h = 0; h < 2; ++h) {
                  const int sb = 2 * g + h;
                  if (sb < w.sb0 || sb >= w.sb1) continue;
#pragma unroll
                  for (int ab = 0; ab < 4; ++ab) {
                    const uint32_t ua = (uint32_t)(4 * h + 2 * (ab >> 1));
                    const uint32_t vb = (uint32_t)(4 * h + 2 * (ab & 1));
                    umma_tf32(d_tmem, udesc + ua, vdesc + vb, idesc_min, acc_on);
                    acc_on = 1;
                  }
                }
              }
              // the epilogue frees the operand stage when it sees this commit
              umma_commit(&bars->tfull[me]);
            } else if (lane == 0 && ok) {
              // descriptors of the stage's three tiles; a K step of 16
              // elements (32 bytes) adds 2 to the start-address field
              const uint8_t* bt = smem + slot * L::kOpStage;
              const uint32_t xdesc = sw128_desc_lo(smem_u32(bt + L::kOpX));
              const uint32_t hdesc = sw128_desc_lo(smem_u32(bt + L::kOpWhi));
              const uint32_t ldesc = sw128_desc_lo(smem_u32(bt + L::kOpWlo));
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const uint32_t d_tmem = tmem + (uint32_t)((2 * me + q) * kBufCols);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint32_t koff = (uint32_t)((2 * q + h) * 2);  // sub-block within the stage
                  umma_f16(d_tmem, xdesc + koff, hdesc + koff, idesc, (uint32_t)h);
                  if (!kQ4) umma_f16(d_tmem, xdesc + koff, ldesc + koff, idesc, 1u);
                }
              }
              // the epilogue frees the operand stage when it sees this commit
              umma_commit(&bars->tfull[me]);
            }
            __syncwarp();
          }
          gbase += nt;
        }
        // take the epilogue's hand-back of the last stage, so every phase
        // of the slot's barrier closes
        if (uses > 0) slot_bar_sync(me);
        if (lane == 0) {
          // Every MMA of every issuer must be finished before TMEM is released.
          umma_commit(&bars->drain);
          volatile int no_abort = 0;
          mbar_wait_bounded(&bars->drain, 0, &no_abort, status, kSiteDrain);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ warpgroups 1-2: epilogue --
    regs_alloc<kEpiRegs>();
    const int ew = warp - kEpiWarp0;  // 0..7
    const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
    const int colh = ew >> 2;         // weight-row columns 64*colh .. +63
    const int tok = 32 * quarter + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(64 * colh);
    float2 acc[32], sb[32];
    uint32_t pA[32], pB[32];
    int gs = 0;
    bool ok = true;
    // fused quantiser: the thread's staging row for operand ring slot pp, and
    // the da entry of chunk cc of scale ring slot ss
    auto fx_stg = [&](int pp) -> uint8_t* {
      return colh == 0 ? smem + pp * L::kOpStage + L::kOpX + tok * 128
                       : smem + L::kXStage + tok * 128;
    };
    const int wrow = 32 * quarter;  // the warp's first token row
    auto fx_stg0 = [&](int pp) -> uint32_t {
      return smem_u32(fx_stg(pp)) - (uint32_t)(lane * 128);
    };
    auto fx_da = [&](int ss, int cc) -> float* {
      return reinterpret_cast<float*>(smem + L::kRingS + ss * L::kScStage + L::kScDa) + cc * BT +
             tok;
    };
    if (kFuseX && (int)blockIdx.x < U) {
      // the CTA's first four operand stages (its first super-block)
      const Unit w0 = unit_of(blockIdx.x, Tw, nsb, splits);
      const int n0 = (w0.t % NT) * BT;
      for (int pp = 0; pp < 4; ++pp) {
        fx_issue(fx_stg0(pp), tok, Xf, ldx, N, n0 + wrow, (4 * w0.sb0 + pp) * KB + 32 * colh);
        fx_finish(fx_stg(pp), smem + pp * L::kOpStage + L::kOpX, tok, colh, fx_da(0, 2 * pp + colh));
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->b_full[pp]);
          if (pp == 3) mbar_arrive(&bars->s_full[0]);
        }
      }
    }
    // Once a wait has been given up (ok == false) the epilogue stops waiting
    // and writes no Y, but still walks every stage and hands every TMEM slot
    // use back, so that the issuers' bar.sync phases stay paired (and, with
    // the fused quantiser, every thread still takes every quantisation step,
    // so that its barrier stays paired too).
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
      const Unit w = unit_of(u, Tw, nsb, splits);
      const int m0 = (w.t / NT) * BW, n0 = (w.t % NT) * BT;
      const int n = n0 + tok;
      const int mcol = m0 + 64 * colh;
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = make_float2(0.0f, 0.0f);
      for (int s = w.sb0; s < w.sb1; ++s) {
        const int slot = gs % SS;
        if (ok && !mbar_wait_warp(&bars->s_full[slot], (gs / SS) & 1, abort_flag, status,
                                  kSiteSFull))
          ok = false;
        const uint8_t* st = smem + L::kRingS + slot * L::kScStage;
        const float* sda = reinterpret_cast<const float*>(st + L::kScDa) + tok;
        // fused quantiser: this super-block's stages quantise those of the
        // next super-block (of this unit, or the CTA's next unit's first),
        // four operand stages ahead, into the same ring slots
        int fx_sb = s + 1, fx_n0 = n0;
        bool fx_on = kFuseX;
        if (kFuseX && fx_sb >= w.sb1) {
          const int un = u + (int)gridDim.x;
          fx_on = un < U;
          if (fx_on) {
            const Unit wn = unit_of(un, Tw, nsb, splits);
            fx_sb = wn.sb0;
            fx_n0 = (wn.t % NT) * BT;
          }
        }
        const int fx_slot = (gs + 1) % SS;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          // Operand stage 4s + pp: its two chunks sit in TMEM slot pp % 2 (a
          // tile has a multiple of four stages), in the slot's use (pp / 2) % 2.
          const uint32_t ts = (uint32_t)(pp & 1);
          if (ok && !mbar_wait_warp(&bars->tfull[ts], (uint32_t)((pp >> 1) & 1), abort_flag,
                                    status, kSiteTFull))
            ok = false;
          // the stage's Xh tile has been read: stage the block four ahead
          if (fx_on)
            fx_issue(fx_stg0(pp), tok, Xf, ldx, N, fx_n0 + wrow,
                     (4 * fx_sb + pp) * KB + 32 * colh);
          // The stage's MMAs are complete, so its operand ring slot (pp: the
          // super-block starts at a global stage that is a multiple of SB)
          // can be refilled: one arrive per stage, from one thread.
          if (ew == 0 && lane == 0) mbar_arrive(&bars->b_empty[pp]);
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int cc = 2 * pp + q, c = 8 * s + cc;
            const uint32_t col = (2 * ts + (uint32_t)q) * kBufCols;
            tmem_ld32(lane_addr + col, pA);
            tmem_ld32(lane_addr + col + 32u, pB);
            const float da = sda[cc * BT];
            tmem_wait_ld2(pA, pB);
            if (q == 1) {
              // both chunks of the stage are in registers: free the slot
              tc_fence_before();
              __syncwarp();
              slot_bar_arrive((int)ts);
            }
            if (cc == 0) {
              chunk_fma<true>(sb, pA, da);
              chunk_fma<true>(sb + 16, pB, da);
            } else {
              chunk_fma<false>(sb, pA, da);
              chunk_fma<false>(sb + 16, pB, da);
            }
            dump_partials<kPartials>(partials, M, N, p_stride, n, mcol, c * p_mul + p_add, pA);
            dump_partials<kPartials>(partials, M, N, p_stride, n, mcol + 32, c * p_mul + p_add,
                                     pB);
          }
          if (fx_on) {
            // quantise the staged block into ring slot pp's Xh tile and its
            // scale into the next super-block's scale stage
            fx_finish(fx_stg(pp), smem + pp * L::kOpStage + L::kOpX, tok, colh,
                      fx_da(fx_slot, 2 * pp + colh));
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&bars->b_full[pp]);
              if (pp == 3) mbar_arrive(&bars->s_full[fx_slot]);
            }
          }
        }
        // Y += d * Sb for this super-block
        const float4* dv = reinterpret_cast<const float4*>(st + L::kScD) + 16 * colh;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float4 d4 = dv[j];
          acc[2 * j] = __ffma2_rn(make_float2(d4.x, d4.y), sb[2 * j], acc[2 * j]);
          acc[2 * j + 1] = __ffma2_rn(make_float2(d4.z, d4.w), sb[2 * j + 1], acc[2 * j + 1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_empty[slot]);
        ++gs;
      }
      if (kQ4) {
        // q4_K: Y -= the min term, one TMEM buffer per min stage (slot use
        // and ring slot follow the chunk stages: every unit starts at a
        // multiple of four operand stages, and so do its min stages)
        const int ng = min_groups(w), ns = min_stages(w);
        for (int i4 = 0; i4 < ns; i4 += 4) {
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            const uint32_t ts = (uint32_t)(pp & 1);
            if (ok && !mbar_wait_warp(&bars->tfull[ts], (uint32_t)((pp >> 1) & 1), abort_flag,
                                      status, kSiteTFull))
              ok = false;
            if (ew == 0 && lane == 0) mbar_arrive(&bars->b_empty[pp]);
            tc_fence_after();
            const bool real = i4 + pp < ng;  // warp-uniform
            if (real) {
              const uint32_t col = 2 * ts * kBufCols;
              tmem_ld32(lane_addr + col, pA);
              tmem_ld32(lane_addr + col + 32u, pB);
              tmem_wait_ld2(pA, pB);
            }
            tc_fence_before();
            __syncwarp();
            slot_bar_arrive((int)ts);
            if (real) {
              sub_words(acc, pA);
              sub_words(acc + 16, pB);
            }
          }
        }
      }
      if (ok && n < N && write_y) {
        // a K part stores its sums to its slice of the partial-sum buffer
        // [splits][N][M] (row stride M, 16-byte aligned rows when M % 4 == 0)
        const bool to_part = splits > 1;
        float* yr = to_part ? part + ((size_t)w.part * N + n) * (size_t)M + mcol
                            : Y + (size_t)n * ldy + mcol;
        const int vec4 = to_part ? ((M & 3) == 0) : y_vec4;
        const int mleft = M - mcol;
        if (!w.split) {
          if (vec4 && mleft >= 64) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              reinterpret_cast<float4*>(yr)[j] =
                  make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x, acc[2 * j + 1].y);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (2 * j < mleft) yr[2 * j] = acc[j].x;
              if (2 * j + 1 < mleft) yr[2 * j + 1] = acc[j].y;
            }
          }
        } else {
          // one of the two K halves of a split tile: add into the zeroed Y
          // (two addends onto zero: the sum is the same in either order)
          if (y_vec4 && mleft >= 64) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              atomicAdd(reinterpret_cast<float4*>(yr) + j,
                        make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x, acc[2 * j + 1].y));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (2 * j < mleft) atomicAdd(yr + 2 * j, acc[j].x);
              if (2 * j + 1 < mleft) atomicAdd(yr + 2 * j + 1, acc[j].y);
            }
          }
        }
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

int g_num_sms[64] = {0};

int sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  int& n = g_num_sms[dev & 63];
  if (n == 0 && (e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev))) return (int)e;
  *sms = n;
  return 0;
}

template <int F, bool P, bool X = false>
cudaError_t launch_one(const TcMaps& maps, int M, int K, int N, float* Y, int ldy,
                       const TcDebugOut& dbg, unsigned int* status, cudaStream_t s,
                       float* part, const float* Xf = nullptr, int ldx = 0) {
  int sms = 0;
  cudaError_t e = (cudaError_t)sm_count(&sms);
  if (e != cudaSuccess) return e;
  const TcPlan p = mmq_tc_plan(M, K, N, sms, part != nullptr);
  const int y_vec4 = (ldy % 4 == 0) && (reinterpret_cast<uintptr_t>(Y) % 16 == 0);
  if (p.splits == 1 && p.U > p.Tw && dbg.write_y) {
    zero_split_tiles_kernel<<<dim3((unsigned)((p.U - p.Tw) / 2), BT / 32), 256, 0, s>>>(
        Y, ldy, M, N, p.Tw, y_vec4);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  mmq_tc_kernel<F, P, X><<<p.grid, kThreads, smem_bytes<F, X>(), s>>>(
      maps.x, maps.whi, maps.wlo, maps.da, maps.d, maps.us, maps.mv, M, K, N, p.Tw, p.U, Y, ldy,
      y_vec4, dbg.out, dbg.stride, dbg.mul, dbg.add, dbg.write_y, Xf, ldx, p.splits, part,
      status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.splits > 1 && dbg.write_y) {
    const long long total = (long long)N * M;
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, s>>>(part, p.splits, N, M, Y, ldy);
    e = cudaGetLastError();
  }
  return e;
}

template <int F, bool P, bool X = false>
cudaError_t raise_smem() {
  return cudaFuncSetAttribute(mmq_tc_kernel<F, P, X>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<F, X>());
}

}  // namespace

size_t mmq_tc_smem_bytes() { return smem_bytes<kFmtQ6>(); }

// Grid and work units for an M x K x N GEMM on `sms` SMs: one persistent CTA
// per SM walks the units; the last round of tiles is split in two along K
// when that keeps more than half of the SMs busy instead of idle. When the
// tiles fill at most half of the SMs (and a partial-sum buffer is given),
// every tile is split into sms / T K parts instead (at most one per
// super-block, at most 8), so that 17 tokens against 4096 weight rows (32
// tiles) take 128 SMs instead of 32.
TcPlan mmq_tc_plan(int M, int K, int N, int sms, bool allow_splitk) {
  const long long T = (long long)((N + BT - 1) / BT) * ((M + BW - 1) / BW);
  const int nsb = K / 256;
  TcPlan p;
  p.splits = 1;
  if (allow_splitk && 2 * T <= sms && nsb >= 2) {
    long long s = sms / T;
    if (s > nsb) s = nsb;
    if (s > 8) s = 8;
    p.splits = (int)s;
    p.Tw = 0;
    p.U = (int)(T * s);
    p.grid = (unsigned)p.U;
    p.launches = 2;
    return p;
  }
  p.grid = (unsigned)(T < sms ? T : sms);
  const long long rem = T % sms;
  if (T > sms && rem > 0 && 2 * rem <= sms && nsb >= 2) {
    p.Tw = (int)(T - rem);
    p.U = (int)(T + rem);
  } else {
    p.Tw = (int)T;
    p.U = (int)T;
  }
  p.launches = (p.U > p.Tw) ? 2 : 1;
  return p;
}

cudaError_t mmq_tc_plan_here(int M, int K, int N, bool allow_splitk, TcPlan* plan) {
  int sms = 0;
  const cudaError_t e = (cudaError_t)sm_count(&sms);
  if (e != cudaSuccess) return e;
  *plan = mmq_tc_plan(M, K, N, sms, allow_splitk);
  return cudaSuccess;
}

// Raises the dynamic shared-memory limit of every instantiation; once per device.
cudaError_t mmq_tc_prepare() {
  cudaError_t e;
  if ((e = raise_smem<kFmtQ6, false>()) || (e = raise_smem<kFmtQ6, true>()) ||
      (e = raise_smem<kFmtQ4, false>()) || (e = raise_smem<kFmtQ4, true>()))
    return e;
  return raise_smem<kFmtQ6, false, true>();
}

cudaError_t launch_mmq_tc(const TcMaps& maps, int M, int K, int N, float* Y, int ldy,
                          const TcDebugOut& dbg, unsigned int* status, cudaStream_t s,
                          float* part) {
  return dbg.out ? launch_one<kFmtQ6, true>(maps, M, K, N, Y, ldy, dbg, status, s, part)
                 : launch_one<kFmtQ6, false>(maps, M, K, N, Y, ldy, dbg, status, s, part);
}

cudaError_t launch_mmq_tc_q4k(const TcMaps& maps, int M, int K, int N, float* Y, int ldy,
                              const TcDebugOut& dbg, unsigned int* status, cudaStream_t s,
                              float* part) {
  return dbg.out ? launch_one<kFmtQ4, true>(maps, M, K, N, Y, ldy, dbg, status, s, part)
                 : launch_one<kFmtQ4, false>(maps, M, K, N, Y, ldy, dbg, status, s, part);
}

cudaError_t launch_mmq_tc_fused(const TcMaps& maps, int M, int K, const float* X, int ldx, int N,
                                float* Y, int ldy, unsigned int* status, cudaStream_t s,
                                float* part) {
  return launch_one<kFmtQ6, false, true>(maps, M, K, N, Y, ldy, TcDebugOut{}, status, s, part, X,
                                         ldx);
}

}  // namespace q6
