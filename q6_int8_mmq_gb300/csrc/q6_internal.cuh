// Internal declarations and sm_103a device helpers of the q6mmq library.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q6mmq.h"

namespace q6 {

// ---------------------------------------------------------------- status ---
// Codes a kernel records in the per-device status word when it gives up a
// bounded wait. Bits 0..7: code; bits 8..15: the wait site.
enum : uint32_t {
  kStatusTimeout = 1u,
};
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Packed-plane geometry (all offsets 256-byte aligned).
struct PlaneGeom {
  size_t qlh_off, sc_off, d_off, dt_off, total;
  size_t qlh_row;  // 3K/4 bytes
  size_t d_row;    // bytes per row of the binary16 d sub-plane: K/128 rounded up to 16
  int ldm;         // row stride (elements) of the transposed d sub-plane: M rounded up to 4
};
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline PlaneGeom plane_geom(int M, int K) {
  PlaneGeom g;
  const size_t m = (size_t)M, k = (size_t)K;
  g.ldm = (M + 3) / 4 * 4;
  g.qlh_row = k / 128 * 96;
  g.qlh_off = 0;
  g.sc_off = round_up(m * g.qlh_row, 256);
  g.d_row = round_up(k / 256 * 2, 16);
  g.d_off = g.sc_off + round_up(m * (k / 16), 256);
  g.dt_off = g.d_off + round_up(m * g.d_row, 256);
  g.total = g.dt_off + round_up((k / 256) * (size_t)g.ldm * 4, 256);
  return g;
}

// Packed q4_K plane geometry (q4k.cu; all offsets 256-byte aligned).
// Row length (f32 elements) of the q4_K min-term operand planes: per
// super-block 16 values, the hi parts of its 8 chunks then the lo parts,
// padded to an even number of super-blocks (32 values, one 128-byte tile row,
// per pair of super-blocks).
__host__ __device__ constexpr int q4_min_ld(int K) { return 32 * ((K / 256 + 1) / 2); }

struct Q4Geom {
  size_t qs_off, sc_off, mn_off, dt_off, mv_off, ddm_off, total;
  int ldm;  // row stride (elements) of the transposed d sub-plane: M rounded up to 4
};
inline Q4Geom q4_geom(int M, int K) {
  Q4Geom g;
  const size_t m = (size_t)M, k = (size_t)K;
  g.ldm = (M + 3) / 4 * 4;
  g.qs_off = 0;
  g.sc_off = round_up(m * (k / 2), 256);
  g.mn_off = g.sc_off + round_up(m * (k / 32), 256);
  g.dt_off = g.mn_off + round_up(m * (k / 32), 256);
  g.mv_off = g.dt_off + round_up((k / 256) * (size_t)g.ldm * 4, 256);
  g.ddm_off = g.mv_off + round_up(m * (size_t)q4_min_ld(K) * 4, 256);
  g.total = g.ddm_off + round_up(m * (k / 256) * 8, 256);
  return g;
}

// --------------------------------------------------------- kernel launches ---
// Each returns cudaGetLastError() of its launch.
// us (nullable) [K/32][ldda] receives da * (sum of the block's codes), the
// activation block sum the q4_K min term needs.
cudaError_t launch_quantize(const float* X, int N, int K, int ldx, int8_t* Xq, float* da, int ldda,
                            __half* Xh, float* us, cudaStream_t s);
cudaError_t launch_q4k_pack(const uint8_t* raw, int M, int K, uint8_t* plane, cudaStream_t s);
// The binary16 operand plane [M][K] of a packed q4_K plane: sc * q, or q alone
// when unit (the debug partials).
cudaError_t launch_q4k_expand(const uint8_t* plane, int M, int K, bool unit, __half* wq,
                              cudaStream_t s);
cudaError_t launch_pack(const uint8_t* raw, int M, int K, uint8_t* plane, int8_t* wexp,
                        cudaStream_t s);
// Debug outputs of the GEMM kernels (both optional, int32, token-major):
//   partials   [N][M][K/16]: P = sum over a 16-element sub-block of (q - 32) * xq;
//   chunk_sums [N][M][K/32]: S = sc[2c] * P[2c] + sc[2c+1] * P[2c+1].
struct Debug {
  int32_t* partials = nullptr;
  int32_t* chunk_sums = nullptr;
  bool any() const { return partials != nullptr || chunk_sums != nullptr; }
};
cudaError_t launch_mmq_skinny(const uint8_t* plane, int M, int K, const int8_t* Xq, const float* da,
                              int ldda, int N, float* Y, int ldy, Debug dbg,
                              unsigned int* status, cudaStream_t s);
// The same product for 3 <= N <= 16 (correct from N = 2) on the warp-level
// f16 tensor path with TMA-staged weights (mmq_skinny_mma.cu).
cudaError_t launch_mmq_skinny_mma(const uint8_t* plane, int M, int K, const int8_t* Xq,
                                  const float* da, int ldda, int N, float* Y, int ldy,
                                  Debug dbg, unsigned int* status, cudaStream_t s);
cudaError_t mmq_skinny_mma_prepare();
cudaError_t mmq_skinny_prepare();
// A 2D tensor map without swizzle or interleave (uint64 elements, or f32 when
// f32 is set) for the few-token kernels' TMA stages; needs
// mmq_skinny_mma_prepare() to have run (it looks up the encoder).
CUresult skinny_tensor_map(CUtensorMap* map, bool f32, const void* base, uint64_t inner,
                           uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                           uint32_t box_outer);
// Quantise + GEMM for N <= 2 tokens from f32 X [N][ldx] in one launch
// (mmq_skinny.cu); needs mmq_skinny_fused_smem(K, N) <= kFusedSmemMax bytes
// of shared memory.
constexpr int kFusedSmemMax = 227 * 1024;
size_t mmq_skinny_fused_smem(int K, int N);
cudaError_t launch_mmq_skinny_fused(const uint8_t* plane, int M, int K, const float* X, int ldx,
                                    int N, float* Y, int ldy, cudaStream_t s);
cudaError_t launch_mmq_sync(const uint8_t* plane, const int8_t* wexp, int M, int K,
                            const int8_t* Xq, const float* da, int ldda, int N, float* Y, int ldy,
                            Debug dbg, cudaStream_t s);
cudaError_t mmq_sync_prepare();

struct TcMaps {
  CUtensorMap x;    // Xh   [N][K] f16, box {64, 128}, 128B swizzle
  CUtensorMap whi;  // W_hi [M][K] f16, box {64, 128}, 128B swizzle
  CUtensorMap wlo;  // W_lo [M][K] f16, box {64, 128}, 128B swizzle
  CUtensorMap da;   // da   [K/32][ldda] f32, box {128, 8}
  CUtensorMap d;    // d^T  [K/256][ldm] f32, box {128, 1}
  CUtensorMap us;   // q4_K: da * S as hi/lo pairs [N][q4_min_ld] f32, box {32, 128}, 128B swizzle
  CUtensorMap mv;   // q4_K: dmin * m as hi/lo pairs [M][q4_min_ld] f32, box {32, 128}, 128B swizzle
};
// What one tensor-core GEMM launch writes besides (or instead of) Y: the
// exact integer of each (token, weight row, 32-element chunk c) accumulator
// at out[(n * M + m) * stride + c * mul + add], when out is not NULL.
//   chunk sums of the folded planes: stride K/32, mul 1, add 0;
//   P of sub-block parity p (planes from launch_expand_unit): stride K/16,
//   mul 2, add p.
// write_y == 0 leaves Y untouched (a debug pass on unit-scale planes).
struct TcDebugOut {
  int32_t* out = nullptr;
  int stride = 0, mul = 1, add = 0;
  int write_y = 1;
};
// part: a buffer of tc_part_bytes(mmq_tc_plan(.., true)) bytes (16-byte
// aligned) that lets a call with few tiles split K over the idle SMs, or NULL.
cudaError_t launch_mmq_tc(const TcMaps& maps, int M, int K, int N, float* Y, int ldy,
                          const TcDebugOut& dbg, unsigned int* status, cudaStream_t s,
                          float* part = nullptr);
// The same GEMM quantising its A operand itself: f32 X [N][ldx] (16-byte
// aligned rows) is quantised per 32-element block inside the kernel, bit for
// bit as q8_quantize_act does, into the Xh tiles and da; maps.x and maps.da
// are unused.
cudaError_t launch_mmq_tc_fused(const TcMaps& maps, int M, int K, const float* X, int ldx, int N,
                                float* Y, int ldy, unsigned int* status, cudaStream_t s,
                                float* part = nullptr);
// The q4_K form of the same GEMM (one operand plane, sc * q, in maps.whi; the
// min term on the tensor cores from maps.us and maps.mv).
cudaError_t launch_mmq_tc_q4k(const TcMaps& maps, int M, int K, int N, float* Y, int ldy,
                              const TcDebugOut& dbg, unsigned int* status, cudaStream_t s,
                              float* part = nullptr);
// The q4_K GEMM for a few tokens (N <= Q6_Q4K_SKINNY_MAX_N): dp4a on the
// packed plane's nibbles, Xq [N][K], da [K/32][ldda] and the block-sum pairs
// us [N][q4_min_ld(K)]; partials (nullable) [N][M][K/32].
cudaError_t launch_q4k_skinny(const uint8_t* plane, int M, int K, const int8_t* Xq,
                              const float* da, int ldda, const float* us, int N, float* Y,
                              int ldy, int32_t* partials, cudaStream_t s);
// q4_K quantise + GEMM for N <= 2 tokens from f32 X [N][ldx] in one launch
// (q4k_skinny.cu); needs q4k_skinny_fused_smem(K, N) <= kFusedSmemMax bytes.
size_t q4k_skinny_fused_smem(int K, int N);
cudaError_t launch_q4k_skinny_fused(const uint8_t* plane, int M, int K, const float* X, int ldx,
                                    int N, float* Y, int ldy, cudaStream_t s);
cudaError_t q4k_skinny_prepare();
// The same product for a few more tokens (N <= 16) on the warp-level f16
// tensor path with TMA-staged nibbles and activations (q4k_skinny_mma.cu).
cudaError_t launch_q4k_skinny_mma(const uint8_t* plane, int M, int K, const int8_t* Xq,
                                  const float* da, int ldda, const float* us, int N, float* Y,
                                  int ldy, int32_t* partials, unsigned int* status,
                                  cudaStream_t s);
cudaError_t q4k_skinny_mma_prepare();
// Tensor maps of a q4_K GEMM call (api.cu): Xh, the operand plane wq [M][K],
// da [K/32][ldda], the block-sum pairs us [N][q4_min_ld], and the packed q4_K
// plane's dT and min-pair sub-planes.
int encode_tc_maps_q4k(TcMaps* maps, const uint8_t* q4plane, const void* wq, const void* Xh,
                       const float* da, const float* us, int M, int K, int N);
// Tensor maps of one tensor-core GEMM call (api.cu): Xh [N][K], the operand
// planes W_hi at wop and W_lo at wop + M*K, da [K/32][ldda], and the
// transposed d sub-plane of the packed plane. Allocates nothing.
int encode_tc_maps(TcMaps* maps, const uint8_t* plane, const void* wop, const void* Xh,
                   const float* da, int M, int K, int N);
// The two binary16 operand planes W_hi, W_lo [M][K] (W_lo at wh + M*K) with
// the sub-block scale folded in, from the packed plane's qlh and sc
// sub-planes, or from the W_exp plane and the sc sub-plane.
cudaError_t launch_expand_raw(const uint8_t* plane, int M, int K, __half* wh, cudaStream_t s);
// Debug planes: W_hi = 0 and W_lo = v on the sub-blocks of parity `parity`
// (0 elsewhere), so the GEMM's chunk accumulator holds P of that sub-block.
cudaError_t launch_expand_unit(const uint8_t* plane, int M, int K, int parity, __half* wh,
                               cudaStream_t s);
cudaError_t launch_expand_wexp(const int8_t* wexp, const uint8_t* plane, int M, int K, __half* wh,
                               cudaStream_t s);
size_t mmq_tc_smem_bytes();
// Launch plan of the tensor-core GEMM for an M x K x N call on `sms` SMs.
struct TcPlan {
  unsigned grid;  // persistent CTAs
  int Tw, U;      // units 0..Tw-1 are whole tiles; Tw..U-1 are K halves of split tiles
  int splits;     // > 1: every tile is split into this many K parts (few tiles)
  int launches;   // kernels per call: the GEMM, plus one that zeroes Y of split
                  // tiles or one that adds the K parts
};
// allow_splitk: a partial-sum buffer of tc_part_bytes() is available.
TcPlan mmq_tc_plan(int M, int K, int N, int sms, bool allow_splitk);
// Bytes of the K-part partial sums of a plan (0 unless splits > 1).
inline size_t tc_part_bytes(const TcPlan& p, int M, int N) {
  return p.splits > 1 ? (size_t)p.splits * (size_t)N * (size_t)M * 4 : 0;
}
// mmq_tc_plan on the current device.
cudaError_t mmq_tc_plan_here(int M, int K, int N, bool allow_splitk, TcPlan* plan);
cudaError_t mmq_tc_prepare();
cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned int* status, cudaStream_t s);

// Launches kernel<<<grid, block, smem, s>>>(args...) as a programmatic
// dependent launch: its CTAs may start while the previous kernel in the stream
// is still running (once that kernel has run griddep_launch_dependents() or
// exited), so its launch and prologue overlap that kernel's tail. The kernel
// must run griddep_wait(), which returns once the previous kernel has
// completed and its writes are visible, before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------- device helpers ---
#if defined(__CUDACC__)
#ifndef MBAR_POLL
#define MBAR_POLL mbar_try_wait
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch ---------------------------------------------
// Waits until the grid this one depends on has completed and its writes are
// visible (returns at once for a kernel launched without the attribute).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel in the stream, if launched with the attribute, start
// its CTAs before this grid has finished.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, giving up after about
// `limit_ns` (measured with the SM cycle counter at up to 2.1 GHz, so the real
// limit is at least that long) or as soon as another thread of the CTA has
// given up (*abort != 0). On expiry it records (site, timeout) in *status and
// sets *abort. Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, unsigned int* status,
                                                  uint32_t site,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (MBAR_POLL(bar, parity)) return true;
  if (*abort) return false;  // another thread has given up already
  const long long limit_cycles = (long long)(limit_ns * 21ull / 10ull);
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (MBAR_POLL(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*abort) return false;
      if (clock64() - t0 > limit_cycles) {
        atomicOr(status, kStatusTimeout | (site << 8));
        *abort = 1;
        return false;
      }
    }
  }
}

// The same wait executed by every lane of a warp, with a warp-uniform result
// and the warp converged afterwards (needed before .sync.aligned tcgen05 ops).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               unsigned int* status, uint32_t site) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, status, site);
  return __all_sync(0xffffffffu, ok);
}

// TMA -----------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (the tensor core reads its operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// tcgen05 -------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes stacked
// densely (stride-dimension offset 1024 B), atom base 1024-byte aligned.
//   bits 0-13  start address >> 4        bits 16-29 leading offset (unused: 1)
//   bits 32-45 stride offset >> 4 (64)   bits 46-48 fixed 0b001
//   bits 61-63 swizzle: 128-byte (2)
// Only the low word depends on the tile, so the MMA issue builds the 64-bit
// value from a 32-bit low word and this constant high word (32-bit address
// arithmetic per K step: +2 in the start-address field per 32 bytes).
constexpr uint32_t kSw128DescHi = (1024u >> 4) | (1u << (46 - 32)) | (2u << (61 - 32));
__device__ __forceinline__ uint32_t sw128_desc_lo(uint32_t saddr) {
  return ((saddr & 0x3FFFFu) >> 4) | (1u << 16);
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, issued by one thread; the
// operands are given by the low words of their descriptors.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 ad, {%1, %5};\n\t"
      "mov.b64 bd, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kSw128DescHi)
      : "memory");
}

// Instruction descriptor, kind::f16: f16 x f16 -> f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (0u << 7) | (0u << 10)       // A, B format: f16
         | ((uint32_t)(N >> 3) << 17)   // N >> 3
         | ((uint32_t)(M >> 4) << 24);  // M >> 4
}

// Instruction descriptor, kind::tf32: tf32 x tf32 -> f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (2u << 7) | (2u << 10)       // A, B format: tf32
         | ((uint32_t)(N >> 3) << 17)   // N >> 3
         | ((uint32_t)(M >> 4) << 24);  // M >> 4
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::tf32 (K = 8 per instruction, 32
// bytes of a row, as for kind::f16), issued by one thread.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 ad, {%1, %5};\n\t"
      "mov.b64 bd, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], ad, bd, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kSw128DescHi)
      : "memory");
}

// The hi/lo pair of a f32 value for a two-term tf32 product: hi keeps the
// sign, exponent and the top 10 stored mantissa bits (a tf32 value), lo =
// x - hi (exact in f32). A tensor core reading lo as tf32 drops its low 13
// mantissa bits, so hi + tf32(lo) is within 2^-21 |x| of x, and equals x
// when x has at most 17 significant bits.
__host__ __device__ inline void tf32_split(float x, float& hi, float& lo) {
  union { float f; uint32_t u; } v;
  v.f = x;
  v.u &= 0xFFFFE000u;
  hi = v.f;
  lo = x - hi;
}

// Issues one 32x32b.x32 TMEM load: 32 consecutive 32-bit columns of this
// thread's lane. The registers are valid only after a tmem_wait_* call.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(addr)
      : "memory");
}
// tmem_ld32 for a pipelined consumer: `prev` (the buffer loaded before) is an
// in-out operand, so the math on it cannot be scheduled above this load and
// runs while the load is in flight.
__device__ __forceinline__ void tmem_ld32_before(uint32_t addr, uint32_t (&r)[32],
                                                 uint32_t (&prev)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "+r"(prev[0]), "+r"(prev[1]), "+r"(prev[2]), "+r"(prev[3]), "+r"(prev[4]), "+r"(prev[5]), "+r"(prev[6]), "+r"(prev[7]), "+r"(prev[8]), "+r"(prev[9]), "+r"(prev[10]), "+r"(prev[11]), "+r"(prev[12]), "+r"(prev[13]), "+r"(prev[14]), "+r"(prev[15]), "+r"(prev[16]), "+r"(prev[17]), "+r"(prev[18]), "+r"(prev[19]), "+r"(prev[20]), "+r"(prev[21]), "+r"(prev[22]), "+r"(prev[23]), "+r"(prev[24]), "+r"(prev[25]), "+r"(prev[26]), "+r"(prev[27]), "+r"(prev[28]), "+r"(prev[29]), "+r"(prev[30]), "+r"(prev[31])
      : "r"(addr)
      : "memory");
}
// Waits for this thread's outstanding TMEM loads. The two arrays are in-out
// operands so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
               :
               : "memory");
}

// The same wait for a pipelined consumer: `a` is the buffer just loaded and
// `s` the 16 accumulator pairs that the math issued since that load wrote, so
// the math stays between the load and the wait and overlaps the load.
__device__ __forceinline__ void tmem_wait_ld_after(uint32_t (&a)[32], float2* s) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31]),
                 "+f"(s[0].x), "+f"(s[0].y), "+f"(s[1].x), "+f"(s[1].y), "+f"(s[2].x), "+f"(s[2].y), "+f"(s[3].x), "+f"(s[3].y), "+f"(s[4].x), "+f"(s[4].y), "+f"(s[5].x), "+f"(s[5].y), "+f"(s[6].x), "+f"(s[6].y), "+f"(s[7].x), "+f"(s[7].y), "+f"(s[8].x), "+f"(s[8].y), "+f"(s[9].x), "+f"(s[9].y), "+f"(s[10].x), "+f"(s[10].y), "+f"(s[11].x), "+f"(s[11].y), "+f"(s[12].x), "+f"(s[12].y), "+f"(s[13].x), "+f"(s[13].y), "+f"(s[14].x), "+f"(s[14].y), "+f"(s[15].x), "+f"(s[15].y)
               :
               : "memory");
}

// Moves this warpgroup's per-thread register budget (all four warps of the
// warpgroup must execute the same call).
template <uint32_t kRegs>
__device__ __forceinline__ void regs_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void regs_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegs));
}

// Warp-level f16 tensor path (mma.sync) of the few-token kernels ----------
// a - b on f16x2 pairs.
__device__ __forceinline__ uint32_t hsub2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
constexpr uint32_t kH2_1024 = 0x64006400u;  // (1024, 1024) as f16x2
constexpr uint32_t kH2_1152 = 0x64806480u;  // (1152, 1152) as f16x2
// Activations (-127..127) of bytes (kOdd, kOdd + 2) of a word w as binary16
// pairs, given wb = w ^ 0x80808080 (x + 128 as unsigned bytes): the exponent
// byte 0x64 placed above each byte gives 1024 + (x + 128), minus 1152.
template <int kOdd>
__device__ __forceinline__ uint32_t x_pair(uint32_t wb) {
  return hsub2u(__byte_perm(wb, 0x64u, kOdd ? 0x4341u : 0x4240u), kH2_1152);
}
// D = A (16x16 f16, row) * B (16x8 f16, col) + C, f32 accumulation.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

#endif  // __CUDACC__

}  // namespace q6
