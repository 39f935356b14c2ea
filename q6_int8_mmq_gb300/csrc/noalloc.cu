// q6k_mmq_noalloc: the q6_K x int8 GEMM for callers that cannot allocate
// device memory when they call it -- for example code that runs under a
// fixed memory budget or pool that forbids new allocations, or a latency-
// critical path that must never enter the allocator.
//
// It computes what q6k_mmq computes with the weights unpacked per call, but
// its scratch memory lives in one file-scope static device array instead of a
// caller workspace or a library allocation: the first 256 bytes hold the
// status word the tensor-core kernel records a bounded-wait time-out in, the
// rest holds the two binary16 weight operand planes the unpack pass writes
// (so M * K * 4 must fit in kScratchWeightBytes). Nothing on this path calls cudaMalloc,
// cudaFree or any allocating routine.
//
// The array belongs to the module: every GPU that loads this part of the
// library holds it until the process exits. All calls share it and it keeps
// the last call's contents, so calls that overlap on the GPU (different
// streams, or other devices' threads racing on the same device) race on it.
// The status word is cleared on the call's stream at the start of each call;
// q6k_mmq_noalloc_status() waits for the stream, reads it, clears it and
// reports a time-out as Q6_ETIMEOUT, as q6_sync_status() does for q6k_mmq.
//
// Set-up happens in the first call on each device (with that device
// current): the architecture check, the kernels' shared-memory limits and
// the array's device address (cudaGetSymbolAddress; in host code the array's
// name is only a stand-in, so kernels get that address). That first call
// should come before any stream capture. The tensor maps are encoded by the
// library's shared encoder, which allocates nothing.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "q6_internal.cuh"

namespace q6 {
int record_error(int code, const char* fmt, va_list ap);  // defined with q6_last_error()
}

namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kScratchWeightBytes = 64u << 20;  // a 4096 x 4096 layer: two binary16 planes
static __device__ __align__(256) unsigned char g_noalloc_scratch[kStatusBytes + kScratchWeightBytes];

int na_fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  const int rc = q6::record_error(code, fmt, ap);
  va_end(ap);
  return rc;
}

struct NaDev {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
};
std::mutex g_na_mu;
NaDev g_na_dev[64];

// Set-up of the calling thread's current device, once: the architecture
// check, the kernels' shared-memory limits and the array's device address.
int na_setup(NaDev** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return na_fail(Q6_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return na_fail(Q6_ECUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_na_mu);
  NaDev& st = g_na_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)))
      return na_fail(Q6_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if (major != 10 || minor != 3)
      return na_fail(Q6_EARCH, "device %d is compute capability %d.%d; needs 10.3", dev, major,
                     minor);
    if ((e = q6::mmq_tc_prepare()) || (e = q6::mmq_skinny_prepare()) ||
        (e = q6::mmq_sync_prepare()))
      return na_fail(Q6_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    void* addr = nullptr;
    if ((e = cudaGetSymbolAddress(&addr, g_noalloc_scratch)) || !addr)
      return na_fail(Q6_ECUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    st.scratch = static_cast<unsigned char*>(addr);
    st.ready = true;
  }
  *out = &st;
  return Q6_OK;
}

bool na_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int q6k_mmq_noalloc(const void* plane, const int8_t* wexp, int M, int K,
                               const int8_t* Xq, const float* da, const uint16_t* Xh, int N,
                               float* Y, int ldy, int* path_out, q6_stream_t s) {
  if (path_out) *path_out = Q6_PATH_NONE;
  if (M <= 0 || K <= 0 || K % 256 || N < 0)
    return na_fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0");
  if (ldy < M) return na_fail(Q6_EINVAL, "ldy (%d) < M (%d)", ldy, M);
  if (N == 0) return Q6_OK;
  if (!plane || !da || !Y) return na_fail(Q6_EINVAL, "plane, da and Y are required");
  const bool skinny = N <= Q6_SKINNY_MAX_N;
  // as q6k_mmq: a few more tokens with Xq run the few-token kernels on token
  // groups (no scratch needed) instead of unpacking the weights
  const bool groups = !skinny && N <= Q6_SKINNY_GROUPS_MAX_N && Xq;
  if (skinny && !Xq) return na_fail(Q6_EINVAL, "Xq is required when N <= %d", Q6_SKINNY_MAX_N);
  if (!skinny && !groups && !Xh)
    return na_fail(Q6_EINVAL, "Xh is required when N > %d", Q6_SKINNY_MAX_N);
  if (!na_aligned(plane, 256) || !na_aligned(da, 16) || !na_aligned(Y, 4) ||
      (wexp && !na_aligned(wexp, 16)) || (Xq && !na_aligned(Xq, 16)) || (Xh && !na_aligned(Xh, 16)))
    return na_fail(Q6_EALIGN, "plane 256 B; Xq, Xh, da, wexp 16 B; Y 4 B");
  if (!skinny && !groups && (size_t)M * (size_t)K * 4 > kScratchWeightBytes)
    return na_fail(Q6_ESIZE,
                   "M*K*4 = %zu bytes exceeds this entry point's static scratch of %zu bytes "
                   "(M*K <= %zu weights)",
                   (size_t)M * (size_t)K * 4, kScratchWeightBytes, kScratchWeightBytes / 4);
  if ((long long)N * ldy > (1LL << 40) || (long long)M * K > (1LL << 40))
    return na_fail(Q6_ESIZE, "problem too large");
  NaDev* st;
  int rc = na_setup(&st);
  if (rc) return rc;
  const int ldda = (N + 3) / 4 * 4;
  cudaError_t e;
  unsigned int* status = reinterpret_cast<unsigned int*>(st->scratch);
  if ((e = cudaMemsetAsync(status, 0, sizeof(unsigned int), (cudaStream_t)s)))
    return na_fail(Q6_ECUDA, "clearing the status word: %s", cudaGetErrorString(e));
  if (skinny || groups) {
    // token group g: rows n0 .. n0 + ng - 1 of Xq and Y, columns n0 .. of da
    // (n0 a multiple of 32: 16-byte aligned); one group when N <= 16
    for (int n0 = 0; n0 < N; n0 += Q6_SKINNY_GROUP_N) {
      const int ng = N - n0 < Q6_SKINNY_GROUP_N ? N - n0 : Q6_SKINNY_GROUP_N;
      e = q6::launch_mmq_skinny(static_cast<const uint8_t*>(plane), M, K, Xq + (size_t)n0 * K,
                                da + n0, ldda, ng, Y + (size_t)n0 * ldy, ldy, q6::Debug{}, status,
                                (cudaStream_t)s);
      if (e != cudaSuccess)
        return na_fail(Q6_ECUDA, "skinny kernel launch: %s", cudaGetErrorString(e));
    }
    if (path_out) *path_out = Q6_PATH_SKINNY;
    return Q6_OK;
  }
  __half* wh = reinterpret_cast<__half*>(st->scratch + kStatusBytes);
  const uint8_t* pb = static_cast<const uint8_t*>(plane);
  e = wexp ? q6::launch_expand_wexp(wexp, pb, M, K, wh, (cudaStream_t)s)
           : q6::launch_expand_raw(pb, M, K, wh, (cudaStream_t)s);
  if (e != cudaSuccess) return na_fail(Q6_ECUDA, "weight unpack launch: %s", cudaGetErrorString(e));
  q6::TcMaps maps;
  if ((rc = q6::encode_tc_maps(&maps, pb, wh, Xh, da, M, K, N))) return rc;
  e = q6::launch_mmq_tc(maps, M, K, N, Y, ldy, q6::TcDebugOut{}, status, (cudaStream_t)s);
  if (e != cudaSuccess) return na_fail(Q6_ECUDA, "tensor-core kernel launch: %s", cudaGetErrorString(e));
  if (path_out) *path_out = wexp ? Q6_PATH_TC_WEXP : Q6_PATH_TC_RAW;
  return Q6_OK;
}

extern "C" int q6k_mmq_noalloc_status(q6_stream_t s) {
  NaDev* st;
  int rc = na_setup(&st);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)s);
  if (e != cudaSuccess) return na_fail(Q6_ECUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int word = 0;
  if ((e = cudaMemcpy(&word, st->scratch, sizeof(word), cudaMemcpyDeviceToHost)))
    return na_fail(Q6_ECUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (word == 0) return Q6_OK;
  if ((e = cudaMemset(st->scratch, 0, sizeof(word))))
    return na_fail(Q6_ECUDA, "clearing the status word: %s", cudaGetErrorString(e));
  return na_fail(Q6_ETIMEOUT, "a kernel gave up a bounded wait (status 0x%x, wait site %u)", word,
                 (word >> 8) & 0xFFu);
}
