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
  size_t qlh_off, dsc_off, sc_off, d_off, total;
  size_t qlh_row;  // 3K/4 bytes
};
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline PlaneGeom plane_geom(int M, int K) {
  PlaneGeom g;
  const size_t m = (size_t)M, k = (size_t)K;
  g.qlh_row = k / 128 * 96;
  g.qlh_off = 0;
  g.dsc_off = round_up(m * g.qlh_row, 256);
  g.sc_off = g.dsc_off + round_up(m * (k / 16) * 4, 256);
  g.d_off = g.sc_off + round_up(m * (k / 16), 256);
  g.total = g.d_off + round_up(m * (k / 256) * 2, 256);
  return g;
}

// --------------------------------------------------------- kernel launches ---
// Each returns cudaGetLastError() of its launch.
cudaError_t launch_quantize(const float* X, int N, int K, int ldx, int8_t* Xq, float* da, int ldda,
                            __half* Xh, cudaStream_t s);
cudaError_t launch_pack(const uint8_t* raw, int M, int K, uint8_t* plane, int8_t* wexp,
                        cudaStream_t s);
cudaError_t launch_mmq_skinny(const uint8_t* plane, int M, int K, const int8_t* Xq, const float* da,
                              int ldda, int N, float* Y, int ldy, int32_t* partials,
                              cudaStream_t s);

struct TcMaps {
  CUtensorMap x;    // Xh   [N][K] f16, box {64, 128}, 128B swizzle
  CUtensorMap w;    // qlh  [M][3K/4] u8, box {96, 128}  or  wexp [M][K] u8, box {128, 128}
  CUtensorMap da;   // da   [K/32][ldda] f32, box {128, 4}
  CUtensorMap dsc;  // dsc  [M][K/16] f32, box {8, 128}
};
cudaError_t launch_mmq_tc(const TcMaps& maps, bool wexp, int M, int K, int N, float* Y, int ldy,
                          int32_t* partials, unsigned int* status, cudaStream_t s);
size_t mmq_tc_smem_bytes();
cudaError_t mmq_tc_prepare();
cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned int* status, cudaStream_t s);

// ---------------------------------------------------------- device helpers ---
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
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

// Waits for phase `parity` of `bar` to complete, giving up after `limit_ns`
// or as soon as another thread of the CTA has given up (*abort != 0). On
// expiry it records (site, timeout) in *status and sets *abort. Returns false
// when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, unsigned int* status,
                                                  uint32_t site,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
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
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
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
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // bits 0-13  start address >> 4
  d |= (uint64_t)1u << 16;                   // bits 16-29 leading offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;         // bits 32-45 stride offset >> 4
  d |= (uint64_t)1u << 46;                   // bits 46-48 fixed 0b001
  d |= (uint64_t)2u << 61;                   // bits 61-63 swizzle: 128-byte
  return d;
}

// Instruction descriptor, kind::f16: f16 x f16 -> f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                      // D format: f32
         | (0u << 7) | (0u << 10)       // A, B format: f16
         | ((uint32_t)(N >> 3) << 17)   // N >> 3
         | ((uint32_t)(M >> 4) << 24);  // M >> 4
}

// Loads 2 x 16 consecutive 32-bit TMEM columns of this thread's lane (one
// 32x32b.x16 load from each address) and waits for both.
__device__ __forceinline__ void tmem_ld2x16(uint32_t a0, uint32_t a1, uint32_t (&r0)[16],
                                            uint32_t (&r1)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]),
        "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]),
        "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r1[0]), "=r"(r1[1]),
        "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]),
        "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]),
        "=r"(r1[14]), "=r"(r1[15])
      : "r"(a0), "r"(a1)
      : "memory");
}

#endif  // __CUDACC__

}  // namespace q6
