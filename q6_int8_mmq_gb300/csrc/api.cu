// C-ABI entry points of the q6mmq library: argument checks, per-device
// state, TMA descriptor encoding and kernel dispatch by shape.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "q6_internal.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(Q6_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DevState {
  bool init = false;
  int arch_ok = 0;
  unsigned int* status = nullptr;  // 256-byte block; word 0 is the status word
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// The driver's tensor-map encoder, looked up once (allocates nothing).
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// The calling thread's current device, checked to be sm_103 and prepared
// (status block allocated, kernel attributes raised) on first use.
int device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(Q6_ECUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& st = g_dev[dev];
  if (!st.init) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      return fail(Q6_EARCH, "device %d is compute capability %d.%d; this library is built for 10.3",
                  dev, major, minor);
    }
    if ((e = cudaMalloc(&st.status, 256))) return cuda_fail(e, "cudaMalloc(status)");
    if ((e = cudaMemset(st.status, 0, 256))) return cuda_fail(e, "cudaMemset(status)");
    if ((e = q6::mmq_tc_prepare()) || (e = q6::mmq_skinny_prepare()) ||
        (e = q6::mmq_sync_prepare()) || (e = q6::q4k_skinny_mma_prepare()) ||
        (e = q6::q4k_skinny_prepare()))
      return cuda_fail(e, "cudaFuncSetAttribute");
    if (!encoder()) return fail(Q6_ECUDA, "cuTensorMapEncodeTiled entry point not found");
    st.arch_ok = 1;
    st.init = true;
  }
  *out = &st;
  return Q6_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz, const char* what) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  if (!encoder()) return fail(Q6_ECUDA, "cuTensorMapEncodeTiled entry point not found");
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(Q6_ECUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return Q6_OK;
}

int ldda_of(int N) { return (N + 3) / 4 * 4; }

// The address a kernel reads `raw` through: device memory as it is, or host
// memory this device reads directly: page-locked (registered or
// cudaHostAlloc'd; its device pointer), or any host memory when the device
// reads pageable memory (coherent host memory, as on Grace-Blackwell).
int device_readable(const uint8_t* raw, const uint8_t** src) {
  *src = raw;
  cudaPointerAttributes pa;
  cudaError_t e = cudaPointerGetAttributes(&pa, raw);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(raw)");
  if (pa.type == cudaMemoryTypeHost && pa.devicePointer) {
    *src = static_cast<const uint8_t*>(pa.devicePointer);
  } else if (pa.type == cudaMemoryTypeUnregistered) {
    int dev = 0, pageable = 0;
    if ((e = cudaGetDevice(&dev)) ||
        (e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute(pageable memory access)");
    if (!pageable)
      return fail(Q6_EINVAL,
                  "raw is pageable host memory this device cannot read: page-lock it "
                  "(cudaHostRegister) or copy it to the device");
  }
  return Q6_OK;
}

}  // namespace

namespace q6 {
// Tensor maps of one GEMM call: Xh [N][K] and the two weight operand planes
// (W_hi at wop, W_lo at wop + M*K) as 64 x 128 boxes with the 128-byte
// swizzle, da [K/32][ldda] as 128 tokens x 8 chunks, and the transposed d
// sub-plane [K/256][ldm] as 128 rows x 1 super-block. Allocates nothing (the
// no-allocation entry point uses it too).
int encode_tc_maps(TcMaps* maps, const uint8_t* plane, const void* wop, const void* Xh,
                   const float* da, int M, int K, int N) {
  memset(maps, 0, sizeof(*maps));
  const PlaneGeom g = plane_geom(M, K);
  const uint16_t* whi = static_cast<const uint16_t*>(wop);
  const uint16_t* wlo = whi + (size_t)M * (size_t)K;
  int rc;
  // Xh and da are NULL for the fused quantiser, which makes them itself
  if (Xh && (rc = encode_2d(&maps->x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xh, (uint64_t)K,
                            (uint64_t)N, (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B,
                            "Xh")))
    return rc;
  if (da && (rc = encode_2d(&maps->da, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, da, (uint64_t)N,
                            (uint64_t)K / 32, (uint64_t)ldda_of(N) * 4, 128, 8,
                            CU_TENSOR_MAP_SWIZZLE_NONE, "da")))
    return rc;
  if ((rc = encode_2d(&maps->whi, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, whi, (uint64_t)K, (uint64_t)M,
                      (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "W_hi")) ||
      (rc = encode_2d(&maps->wlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wlo, (uint64_t)K, (uint64_t)M,
                      (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "W_lo")) ||
      (rc = encode_2d(&maps->d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, plane + g.dt_off, (uint64_t)M,
                      (uint64_t)K / 256, (uint64_t)g.ldm * 4, 128, 1, CU_TENSOR_MAP_SWIZZLE_NONE,
                      "d")))
    return rc;
  return Q6_OK;
}

int encode_tc_maps_q4k(TcMaps* maps, const uint8_t* q4plane, const void* wq, const void* Xh,
                       const float* da, const float* us, int M, int K, int N) {
  memset(maps, 0, sizeof(*maps));
  const Q4Geom g = q4_geom(M, K);
  int rc;
  if ((rc = encode_2d(&maps->x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xh, (uint64_t)K, (uint64_t)N,
                      (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "Xh")) ||
      (rc = encode_2d(&maps->whi, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wq, (uint64_t)K, (uint64_t)M,
                      (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "Wq")) ||
      (rc = encode_2d(&maps->da, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, da, (uint64_t)N, (uint64_t)K / 32,
                      (uint64_t)ldda_of(N) * 4, 128, 8, CU_TENSOR_MAP_SWIZZLE_NONE, "da")) ||
      (rc = encode_2d(&maps->us, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, us, (uint64_t)q4_min_ld(K),
                      (uint64_t)N, (uint64_t)q4_min_ld(K) * 4, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B,
                      "us")) ||
      (rc = encode_2d(&maps->d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, q4plane + g.dt_off, (uint64_t)M,
                      (uint64_t)K / 256, (uint64_t)g.ldm * 4, 128, 1, CU_TENSOR_MAP_SWIZZLE_NONE,
                      "dT")) ||
      (rc = encode_2d(&maps->mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, q4plane + g.mv_off,
                      (uint64_t)q4_min_ld(K), (uint64_t)M, (uint64_t)q4_min_ld(K) * 4, 32, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B, "mv pairs")))
    return rc;
  return Q6_OK;
}
}  // namespace q6

namespace q6 {
// Records `code` and its text as the calling thread's last error (for the
// entry points defined in other translation units).
int record_error(int code, const char* fmt, va_list ap) {
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  return code;
}
}  // namespace q6

extern "C" {

const char* q6_last_error(void) { return g_err; }

int q6_device_check(void) {
  DevState* st;
  return device_state(&st);
}

int q6_sync_status(q6_stream_t s) {
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  if ((e = cudaMemcpy(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "cudaMemcpy(status)");
  if (word == 0) return Q6_OK;
  if ((e = cudaMemset(st->status, 0, sizeof(word)))) return cuda_fail(e, "cudaMemset(status)");
  return fail(Q6_ETIMEOUT, "a kernel gave up a bounded wait (status 0x%x, wait site %u)", word,
              (word >> 8) & 0xFFu);
}

int q6_selftest_wait_timeout(int limit_ms, q6_stream_t s) {
  if (limit_ms < 1 || limit_ms > 2000) return fail(Q6_EINVAL, "limit_ms must be in 1..2000");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = q6::launch_wait_selftest((unsigned long long)limit_ms * 1000000ull, st->status,
                                           (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return Q6_OK;
}

int q8_act_plane_bytes(int N, int K, size_t* xq_bytes, size_t* da_bytes, size_t* xh_bytes,
                       int* ldda) {
  if (N < 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need N >= 0, K > 0, K %% 256 == 0");
  const size_t n = (size_t)N, k = (size_t)K;
  if (xq_bytes) *xq_bytes = n * k;
  if (da_bytes) *da_bytes = (k / 32) * (size_t)ldda_of(N) * 4;
  if (xh_bytes) *xh_bytes = n * k * 2;
  if (ldda) *ldda = ldda_of(N);
  return Q6_OK;
}

int q8_act_sums_bytes(int N, int K, size_t* us_bytes, int* ldus) {
  if (N < 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need N >= 0, K > 0, K %% 256 == 0");
  if (us_bytes) *us_bytes = (size_t)N * (size_t)q6::q4_min_ld(K) * 4;
  if (ldus) *ldus = q6::q4_min_ld(K);
  return Q6_OK;
}

static int quantize_entry(const float* X, int N, int K, int ldx, int8_t* Xq, float* da,
                          uint16_t* Xh, float* us, q6_stream_t s, const char* name) {
  if (N < 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need N >= 0, K > 0, K %% 256 == 0");
  if (ldx < K) return fail(Q6_EINVAL, "ldx (%d) < K (%d)", ldx, K);
  if (N == 0) return Q6_OK;
  if (!X || !da || (!Xq && !Xh)) return fail(Q6_EINVAL, "X, da and one of Xq, Xh are required");
  if (!aligned(X, 16) || ldx % 4 || (Xq && !aligned(Xq, 16)) || !aligned(da, 16) ||
      (Xh && !aligned(Xh, 16)) || (us && !aligned(us, 16)))
    return fail(Q6_EALIGN, "X, Xq, da, Xh, us must be 16-byte aligned and ldx a multiple of 4");
  if ((long long)N * K > (1LL << 40)) return fail(Q6_ESIZE, "N*K too large");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = q6::launch_quantize(X, N, K, ldx, Xq, da, ldda_of(N),
                                      reinterpret_cast<__half*>(Xh), us, (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return Q6_OK;
}

int q8_quantize_act(const float* X, int N, int K, int ldx, int8_t* Xq, float* da, uint16_t* Xh,
                    q6_stream_t s) {
  return quantize_entry(X, N, K, ldx, Xq, da, Xh, nullptr, s, "q8_quantize_act launch");
}

int q8_quantize_act_sums(const float* X, int N, int K, int ldx, int8_t* Xq, float* da,
                         uint16_t* Xh, float* us, q6_stream_t s) {
  if (N > 0 && !us) return fail(Q6_EINVAL, "us is required");
  return quantize_entry(X, N, K, ldx, Xq, da, Xh, us, s, "q8_quantize_act_sums launch");
}

int q6k_plane_bytes(int M, int K, size_t* plane_bytes, size_t* wexp_bytes) {
  if (M <= 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need M > 0, K > 0, K %% 256 == 0");
  const q6::PlaneGeom g = q6::plane_geom(M, K);
  if (plane_bytes) *plane_bytes = g.total;
  if (wexp_bytes) *wexp_bytes = (size_t)M * (size_t)K;
  return Q6_OK;
}

int q6k_pack_weights(const uint8_t* raw, int M, int K, void* plane, int8_t* wexp, uint16_t* wh,
                     q6_stream_t s) {
  if (M <= 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need M > 0, K > 0, K %% 256 == 0");
  if (!raw || !plane) return fail(Q6_EINVAL, "raw and plane are required");
  if (!aligned(plane, 256) || (wexp && !aligned(wexp, 16)) || (wh && !aligned(wh, 16)))
    return fail(Q6_EALIGN, "plane must be 256-byte aligned, wexp and wh 16-byte aligned");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  const uint8_t* src = nullptr;
  if ((rc = device_readable(raw, &src))) return rc;
  cudaError_t e = q6::launch_pack(src, M, K, static_cast<uint8_t*>(plane), wexp, (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "q6k_pack_weights launch");
  if (wh) {
    e = q6::launch_expand_raw(static_cast<const uint8_t*>(plane), M, K,
                              reinterpret_cast<__half*>(wh), (cudaStream_t)s);
    if (e != cudaSuccess) return cuda_fail(e, "q6k_pack_weights expand launch");
  }
  return Q6_OK;
}

int q6k_unpack_weights(const void* plane, const int8_t* wexp, int M, int K, uint16_t* wh,
                       q6_stream_t s) {
  if (M <= 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need M > 0, K > 0, K %% 256 == 0");
  if (!wh || !plane) return fail(Q6_EINVAL, "plane and wh are required");
  if (!aligned(plane, 256) || (wexp && !aligned(wexp, 16)) || !aligned(wh, 16))
    return fail(Q6_EALIGN, "plane 256 B; wexp, wh 16 B");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  const uint8_t* pb = static_cast<const uint8_t*>(plane);
  cudaError_t e = wexp ? q6::launch_expand_wexp(wexp, pb, M, K, reinterpret_cast<__half*>(wh),
                                                (cudaStream_t)s)
                       : q6::launch_expand_raw(pb, M, K, reinterpret_cast<__half*>(wh),
                                               (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "q6k_unpack_weights launch");
  return Q6_OK;
}

// Bytes of the K-part partial sums a tensor-core call with few tiles uses,
// planned for GB300's 152 SMs (independent of the device, so that it can be
// asked anywhere); a call splits K only when its workspace holds the plan of
// the device it runs on.
static size_t part_bytes_bound(int M, int K, int N) {
  const q6::TcPlan p = q6::mmq_tc_plan(M, K, N, 152, true);
  return q6::tc_part_bytes(p, M, N);
}

int q6k_tc_part_bytes(int M, int K, int N, size_t* bytes) {
  if (M <= 0 || K <= 0 || K % 256 || N < 0 || !bytes)
    return fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0, bytes != NULL");
  *bytes = N > 0 ? part_bytes_bound(M, K, N) : 0;
  return Q6_OK;
}

int q6k_mmq_workspace_bytes(int M, int K, int N, size_t* bytes) {
  if (M <= 0 || K <= 0 || K % 256 || N < 0 || !bytes)
    return fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0, bytes != NULL");
  *bytes = N > Q6_SKINNY_MAX_N
               ? q6::round_up((size_t)M * (size_t)K * 4, 256) + part_bytes_bound(M, K, N)
               : 0;
  return Q6_OK;
}

// The K-part buffer of a tensor-core call inside the caller's workspace:
// after the first `used` bytes (the unpacked planes), when the workspace
// holds the device's plan; NULL otherwise (the call then runs unsplit).
static int part_buffer(int M, int K, int N, void* workspace, size_t workspace_bytes,
                       size_t used, float** part) {
  *part = nullptr;
  if (!workspace) return Q6_OK;
  q6::TcPlan p;
  cudaError_t e = q6::mmq_tc_plan_here(M, K, N, true, &p);
  if (e != cudaSuccess) return cuda_fail(e, "SM count");
  const size_t need = q6::tc_part_bytes(p, M, N), off = q6::round_up(used, 256);
  if (need > 0 && off + need <= workspace_bytes)
    *part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + off);
  return Q6_OK;
}

// The sub-block partials P of the tensor-core path (debug): two more GEMM
// launches on operand planes unpacked into the workspace with unit scale,
// W_hi = 0 and W_lo = v on the sub-blocks of one parity (0 on the others),
// so each chunk accumulator holds P of one of its two sub-blocks; Y is left
// as the main launch wrote it.
static int tc_subblock_partials(const uint8_t* pb, int M, int K, int N, const uint16_t* Xh,
                                const float* da, float* Y, int ldy, __half* ws, int32_t* partials,
                                unsigned int* status, cudaStream_t s) {
  for (int parity = 0; parity < 2; ++parity) {
    cudaError_t e = q6::launch_expand_unit(pb, M, K, parity, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "debug unpack launch");
    q6::TcMaps maps;
    int rc = q6::encode_tc_maps(&maps, pb, ws, Xh, da, M, K, N);
    if (rc) return rc;
    q6::TcDebugOut dbg;
    dbg.out = partials;
    dbg.stride = K / 16;
    dbg.mul = 2;
    dbg.add = parity;
    dbg.write_y = 0;
    if ((e = q6::launch_mmq_tc(maps, M, K, N, Y, ldy, dbg, status, s)) != cudaSuccess)
      return cuda_fail(e, "debug tensor-core kernel launch");
  }
  return Q6_OK;
}

int q6k_mmq_launches(int M, int K, int N, int has_wh, int* launches) {
  if (M <= 0 || K <= 0 || K % 256 || N < 0 || !launches)
    return fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0, launches != NULL");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  if (N == 0) {
    *launches = 0;
  } else if (N <= Q6_SKINNY_MAX_N) {
    *launches = 1;
  } else if (N <= Q6_SKINNY_GROUP_N || (!has_wh && N <= Q6_SKINNY_GROUPS_MAX_N)) {
    *launches = (N + Q6_SKINNY_GROUP_N - 1) / Q6_SKINNY_GROUP_N;  // token groups (given Xq)
  } else {
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    *launches = q6::mmq_tc_plan(M, K, N, sms, true).launches + (has_wh ? 0 : 1);
  }
  return Q6_OK;
}

int q6k_mmq(const void* plane, const int8_t* wexp, const uint16_t* wh, int M, int K,
            const int8_t* Xq, const float* da, const uint16_t* Xh, int N, float* Y, int ldy,
            void* workspace, size_t workspace_bytes, int32_t* partials, int32_t* chunk_sums,
            int* path_out, q6_stream_t s) {
  if (path_out) *path_out = Q6_PATH_NONE;
  if (M <= 0 || K <= 0 || K % 256 || N < 0)
    return fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0");
  if (ldy < M) return fail(Q6_EINVAL, "ldy (%d) < M (%d)", ldy, M);
  if (N == 0) return Q6_OK;
  if (!plane || !da || !Y) return fail(Q6_EINVAL, "plane, da and Y are required");
  const bool skinny = N <= Q6_SKINNY_MAX_N;
  // a few more tokens given Xq: the few-token kernels on token groups, up to
  // one group's width whatever the weight source (faster than the tensor
  // cores there), and up to Q6_SKINNY_GROUPS_MAX_N without resident planes
  // (instead of unpacking the weights for the tensor cores)
  const bool groups = !skinny && Xq &&
                      (N <= Q6_SKINNY_GROUP_N || (N <= Q6_SKINNY_GROUPS_MAX_N && !wh));
  if (skinny && !Xq) return fail(Q6_EINVAL, "Xq is required when N <= %d", Q6_SKINNY_MAX_N);
  if (!skinny && !groups && !Xh)
    return fail(Q6_EINVAL, "Xh is required when N > %d", Q6_SKINNY_MAX_N);
  if (!aligned(plane, 256) || !aligned(da, 16) || !aligned(Y, 4) ||
      (wexp && !aligned(wexp, 16)) || (wh && !aligned(wh, 16)) || (Xq && !aligned(Xq, 16)) ||
      (Xh && !aligned(Xh, 16)) || (partials && !aligned(partials, 4)) ||
      (chunk_sums && !aligned(chunk_sums, 4)) || (workspace && !aligned(workspace, 256)))
    return fail(Q6_EALIGN,
                "plane, workspace 256 B; Xq, Xh, da, wexp, wh 16 B; Y, partials, chunk_sums 4 B");
  if ((long long)N * ldy > (1LL << 40) || (long long)M * K > (1LL << 40))
    return fail(Q6_ESIZE, "problem too large");
  if (!skinny && !groups && (!wh || partials)) {
    const size_t need = (size_t)M * (size_t)K * 4;
    if (!workspace || workspace_bytes < need)
      return fail(Q6_ESIZE, "workspace of %zu bytes needed to unpack the weights (got %zu)", need,
                  workspace ? workspace_bytes : (size_t)0);
  }
  q6::Debug dbg;
  dbg.partials = partials;
  dbg.chunk_sums = chunk_sums;
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e;
  if (skinny) {
    e = q6::launch_mmq_skinny(static_cast<const uint8_t*>(plane), M, K, Xq, da, ldda_of(N), N, Y,
                              ldy, dbg, st->status, (cudaStream_t)s);
    if (e != cudaSuccess) return cuda_fail(e, "skinny kernel launch");
    if (path_out) *path_out = Q6_PATH_SKINNY;
    return Q6_OK;
  }
  if (groups) {
    // token group g: rows n0 .. n0 + ng - 1 of Xq, Y and the debug outputs,
    // columns n0 .. of da (n0 a multiple of 32: 16-byte aligned)
    for (int n0 = 0; n0 < N; n0 += Q6_SKINNY_GROUP_N) {
      const int ng = N - n0 < Q6_SKINNY_GROUP_N ? N - n0 : Q6_SKINNY_GROUP_N;
      q6::Debug dg;
      dg.partials = partials ? partials + (size_t)n0 * M * (K / 16) : nullptr;
      dg.chunk_sums = chunk_sums ? chunk_sums + (size_t)n0 * M * (K / 32) : nullptr;
      e = q6::launch_mmq_skinny(static_cast<const uint8_t*>(plane), M, K, Xq + (size_t)n0 * K,
                                da + n0, ldda_of(N), ng, Y + (size_t)n0 * ldy, ldy, dg,
                                st->status, (cudaStream_t)s);
      if (e != cudaSuccess) return cuda_fail(e, "skinny kernel launch (token group)");
    }
    if (path_out) *path_out = Q6_PATH_SKINNY;
    return Q6_OK;
  }
  int path = Q6_PATH_TC_WH;
  const uint8_t* pb = static_cast<const uint8_t*>(plane);
  const void* wop = wh;
  if (!wh) {
    __half* ws = static_cast<__half*>(workspace);
    if (wexp) {
      e = q6::launch_expand_wexp(wexp, pb, M, K, ws, (cudaStream_t)s);
      path = Q6_PATH_TC_WEXP;
    } else {
      e = q6::launch_expand_raw(pb, M, K, ws, (cudaStream_t)s);
      path = Q6_PATH_TC_RAW;
    }
    if (e != cudaSuccess) return cuda_fail(e, "weight unpack launch");
    wop = ws;
  }
  q6::TcMaps maps;
  if ((rc = encode_tc_maps(&maps, pb, wop, Xh, da, M, K, N))) return rc;
  q6::TcDebugOut tdbg;
  tdbg.out = chunk_sums;
  tdbg.stride = K / 32;
  float* part = nullptr;
  if ((rc = part_buffer(M, K, N, workspace, workspace_bytes,
                        (!wh || partials) ? (size_t)M * (size_t)K * 4 : 0, &part)))
    return rc;
  e = q6::launch_mmq_tc(maps, M, K, N, Y, ldy, tdbg, st->status, (cudaStream_t)s, part);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
  if (partials &&
      (rc = tc_subblock_partials(pb, M, K, N, Xh, da, Y, ldy, static_cast<__half*>(workspace),
                                 partials, st->status, (cudaStream_t)s)))
    return rc;
  if (path_out) *path_out = path;
  return Q6_OK;
}

int q6k_mmq_f32(const void* plane, int M, int K, const float* X, int ldx, int N, float* Y,
                int ldy, int* path_out, q6_stream_t s) {
  if (path_out) *path_out = Q6_PATH_NONE;
  if (M <= 0 || K <= 0 || K % 256 || N < 0 || N > Q6_FUSED_MAX_N)
    return fail(Q6_EINVAL, "need M > 0, 0 <= N <= %d, K > 0, K %% 256 == 0", Q6_FUSED_MAX_N);
  if (ldx < K) return fail(Q6_EINVAL, "ldx (%d) < K (%d)", ldx, K);
  if (ldy < M) return fail(Q6_EINVAL, "ldy (%d) < M (%d)", ldy, M);
  if (N == 0) return Q6_OK;
  if (!plane || !X || !Y) return fail(Q6_EINVAL, "plane, X and Y are required");
  if (!aligned(plane, 256) || !aligned(X, 16) || ldx % 4 || !aligned(Y, 4))
    return fail(Q6_EALIGN, "plane 256 B, X 16 B with ldx %% 4 == 0, Y 4 B");
  if (q6::mmq_skinny_fused_smem(K, N) > (size_t)q6::kFusedSmemMax)
    return fail(Q6_ESIZE, "K = %d is too large for %d token(s) in one launch", K, N);
  if ((long long)N * ldy > (1LL << 40) || (long long)M * K > (1LL << 40))
    return fail(Q6_ESIZE, "problem too large");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = q6::launch_mmq_skinny_fused(static_cast<const uint8_t*>(plane), M, K, X, ldx, N,
                                              Y, ldy, (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "fused one/two-token kernel launch");
  if (path_out) *path_out = Q6_PATH_SKINNY_FUSED;
  return Q6_OK;
}

int q6k_mmq_f32_tc(const void* plane, const uint16_t* wh, int M, int K, const float* X, int ldx,
                   int N, float* Y, int ldy, void* workspace, size_t workspace_bytes,
                   int* path_out, q6_stream_t s) {
  if (path_out) *path_out = Q6_PATH_NONE;
  if (M <= 0 || K <= 0 || K % 256 || N < 0)
    return fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0");
  if (ldx < K) return fail(Q6_EINVAL, "ldx (%d) < K (%d)", ldx, K);
  if (ldy < M) return fail(Q6_EINVAL, "ldy (%d) < M (%d)", ldy, M);
  if (N == 0) return Q6_OK;
  if (!plane || !X || !Y) return fail(Q6_EINVAL, "plane, X and Y are required");
  if (!aligned(plane, 256) || !aligned(X, 16) || ldx % 4 || !aligned(Y, 4) ||
      (wh && !aligned(wh, 16)) || (workspace && !aligned(workspace, 256)))
    return fail(Q6_EALIGN, "plane, workspace 256 B; X 16 B with ldx %% 4 == 0; wh 16 B; Y 4 B");
  if ((long long)N * ldy > (1LL << 40) || (long long)M * K > (1LL << 40) ||
      (long long)N * ldx > (1LL << 40))
    return fail(Q6_ESIZE, "problem too large");
  if (!wh) {
    const size_t need = (size_t)M * (size_t)K * 4;
    if (!workspace || workspace_bytes < need)
      return fail(Q6_ESIZE, "workspace of %zu bytes needed to unpack the weights (got %zu)", need,
                  workspace ? workspace_bytes : (size_t)0);
  }
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e;
  const uint8_t* pb = static_cast<const uint8_t*>(plane);
  const void* wop = wh;
  int path = Q6_PATH_TC_FUSED_WH;
  if (!wh) {
    __half* ws = static_cast<__half*>(workspace);
    if ((e = q6::launch_expand_raw(pb, M, K, ws, (cudaStream_t)s)) != cudaSuccess)
      return cuda_fail(e, "weight unpack launch");
    wop = ws;
    path = Q6_PATH_TC_FUSED_RAW;
  }
  q6::TcMaps maps;
  if ((rc = encode_tc_maps(&maps, pb, wop, nullptr, nullptr, M, K, N))) return rc;
  float* part = nullptr;
  if ((rc = part_buffer(M, K, N, workspace, workspace_bytes, wh ? 0 : (size_t)M * (size_t)K * 4,
                        &part)))
    return rc;
  e = q6::launch_mmq_tc_fused(maps, M, K, X, ldx, N, Y, ldy, st->status, (cudaStream_t)s, part);
  if (e != cudaSuccess) return cuda_fail(e, "fused-quantiser tensor-core kernel launch");
  if (path_out) *path_out = path;
  return Q6_OK;
}

int q6k_mmq_mma_sync(const void* plane, const int8_t* wexp, int M, int K, const int8_t* Xq,
                     const float* da, int N, float* Y, int ldy, int32_t* partials,
                     int32_t* chunk_sums, int* path_out, q6_stream_t s) {
  if (path_out) *path_out = Q6_PATH_NONE;
  if (M <= 0 || K <= 0 || K % 256 || N < 0)
    return fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0");
  if (ldy < M) return fail(Q6_EINVAL, "ldy (%d) < M (%d)", ldy, M);
  if (N == 0) return Q6_OK;
  if (!plane || !wexp || !Xq || !da || !Y)
    return fail(Q6_EINVAL, "plane, wexp, Xq, da and Y are required");
  if (!aligned(plane, 256) || !aligned(wexp, 16) || !aligned(Xq, 16) || !aligned(da, 16) ||
      !aligned(Y, 4) || (partials && !aligned(partials, 4)) ||
      (chunk_sums && !aligned(chunk_sums, 4)))
    return fail(Q6_EALIGN, "plane 256 B; wexp, Xq, da 16 B; Y, partials, chunk_sums 4 B");
  if ((long long)N * ldy > (1LL << 40) || (long long)M * K > (1LL << 40))
    return fail(Q6_ESIZE, "problem too large");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  q6::Debug dbg;
  dbg.partials = partials;
  dbg.chunk_sums = chunk_sums;
  cudaError_t e = q6::launch_mmq_sync(static_cast<const uint8_t*>(plane), wexp, M, K, Xq, da,
                                      ldda_of(N), N, Y, ldy, dbg, (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "mma.sync kernel launch");
  if (path_out) *path_out = Q6_PATH_SYNC_WEXP;
  return Q6_OK;
}

/* ------------------------------------------------------------------ q4_K */

int q4k_plane_bytes(int M, int K, size_t* plane_bytes, size_t* wq_bytes) {
  if (M <= 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need M > 0, K > 0, K %% 256 == 0");
  if (plane_bytes) *plane_bytes = q6::q4_geom(M, K).total;
  if (wq_bytes) *wq_bytes = (size_t)M * (size_t)K * 2;
  return Q6_OK;
}

int q4k_pack_weights(const uint8_t* raw, int M, int K, void* plane, uint16_t* wq, q6_stream_t s) {
  if (M <= 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need M > 0, K > 0, K %% 256 == 0");
  if (!raw || !plane) return fail(Q6_EINVAL, "raw and plane are required");
  if (!aligned(plane, 256) || (wq && !aligned(wq, 16)))
    return fail(Q6_EALIGN, "plane must be 256-byte aligned, wq 16-byte aligned");
  if ((long long)M * K > (1LL << 40)) return fail(Q6_ESIZE, "M*K too large");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  const uint8_t* src = nullptr;
  if ((rc = device_readable(raw, &src))) return rc;
  cudaError_t e = q6::launch_q4k_pack(src, M, K, static_cast<uint8_t*>(plane), (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "q4k_pack_weights launch");
  if (wq) {
    e = q6::launch_q4k_expand(static_cast<const uint8_t*>(plane), M, K, false,
                              reinterpret_cast<__half*>(wq), (cudaStream_t)s);
    if (e != cudaSuccess) return cuda_fail(e, "q4k_pack_weights expand launch");
  }
  return Q6_OK;
}

int q4k_unpack_weights(const void* plane, int M, int K, uint16_t* wq, q6_stream_t s) {
  if (M <= 0 || K <= 0 || K % 256) return fail(Q6_EINVAL, "need M > 0, K > 0, K %% 256 == 0");
  if (!plane || !wq) return fail(Q6_EINVAL, "plane and wq are required");
  if (!aligned(plane, 256) || !aligned(wq, 16)) return fail(Q6_EALIGN, "plane 256 B, wq 16 B");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = q6::launch_q4k_expand(static_cast<const uint8_t*>(plane), M, K, false,
                                        reinterpret_cast<__half*>(wq), (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "q4k_unpack_weights launch");
  return Q6_OK;
}

int q4k_mmq_f32(const void* plane, int M, int K, const float* X, int ldx, int N, float* Y,
                int ldy, int* path_out, q6_stream_t s) {
  if (path_out) *path_out = Q6_PATH_NONE;
  if (M <= 0 || K <= 0 || K % 256 || N < 0 || N > Q6_FUSED_MAX_N)
    return fail(Q6_EINVAL, "need M > 0, 0 <= N <= %d, K > 0, K %% 256 == 0", Q6_FUSED_MAX_N);
  if (ldx < K) return fail(Q6_EINVAL, "ldx (%d) < K (%d)", ldx, K);
  if (ldy < M) return fail(Q6_EINVAL, "ldy (%d) < M (%d)", ldy, M);
  if (N == 0) return Q6_OK;
  if (!plane || !X || !Y) return fail(Q6_EINVAL, "plane, X and Y are required");
  if (!aligned(plane, 256) || !aligned(X, 16) || ldx % 4 || !aligned(Y, 4))
    return fail(Q6_EALIGN, "plane 256 B, X 16 B with ldx %% 4 == 0, Y 4 B");
  if (q6::q4k_skinny_fused_smem(K, N) > (size_t)q6::kFusedSmemMax)
    return fail(Q6_ESIZE, "K = %d is too large for %d token(s) in one launch", K, N);
  if ((long long)N * ldy > (1LL << 40) || (long long)M * K > (1LL << 40))
    return fail(Q6_ESIZE, "problem too large");
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = q6::launch_q4k_skinny_fused(static_cast<const uint8_t*>(plane), M, K, X, ldx,
                                              N, Y, ldy, (cudaStream_t)s);
  if (e != cudaSuccess) return cuda_fail(e, "q4_K fused one/two-token kernel launch");
  if (path_out) *path_out = Q6_PATH_Q4K_SKINNY_FUSED;
  return Q6_OK;
}

int q4k_mmq(const void* plane, const uint16_t* wq, int M, int K, const int8_t* Xq,
            const uint16_t* Xh, const float* da, const float* us, int N, float* Y, int ldy,
            void* workspace, size_t workspace_bytes, int32_t* partials, int* path_out,
            q6_stream_t s) {
  if (path_out) *path_out = Q6_PATH_NONE;
  if (M <= 0 || K <= 0 || K % 256 || N < 0)
    return fail(Q6_EINVAL, "need M > 0, N >= 0, K > 0, K %% 256 == 0");
  if (ldy < M) return fail(Q6_EINVAL, "ldy (%d) < M (%d)", ldy, M);
  if (N == 0) return Q6_OK;
  const bool skinny = N <= Q6_Q4K_SKINNY_MAX_N;
  // a few more tokens given Xq: the few-token f16 kernel on token groups, up
  // to one group's width whatever the weight source (faster than the tensor
  // cores there), and up to Q6_Q4K_GROUPS_MAX_N without a resident operand
  // plane (instead of unpacking the weights for the tensor cores)
  const bool groups = !skinny && Xq &&
                      (N <= Q6_Q4K_GROUP_N || (N <= Q6_Q4K_GROUPS_MAX_N && !wq));
  if (!plane || !da || !us || !Y) return fail(Q6_EINVAL, "plane, da, us and Y are required");
  if (skinny && !Xq) return fail(Q6_EINVAL, "Xq is required when N <= %d", Q6_Q4K_SKINNY_MAX_N);
  if (!skinny && !groups && !Xh)
    return fail(Q6_EINVAL, "Xh is required when N > %d", Q6_Q4K_SKINNY_MAX_N);
  if (!aligned(plane, 256) || (Xq && !aligned(Xq, 16)) || (Xh && !aligned(Xh, 16)) ||
      !aligned(da, 16) || !aligned(us, 16) || !aligned(Y, 4) || (wq && !aligned(wq, 16)) ||
      (partials && !aligned(partials, 4)) || (workspace && !aligned(workspace, 256)))
    return fail(Q6_EALIGN, "plane, workspace 256 B; Xq, Xh, da, us, wq 16 B; Y, partials 4 B");
  if ((long long)N * ldy > (1LL << 40) || (long long)M * K > (1LL << 40))
    return fail(Q6_ESIZE, "problem too large");
  if (skinny || groups) {
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    const uint8_t* pb = static_cast<const uint8_t*>(plane);
    const int ldus = q6::q4_min_ld(K);
    // token group g: rows n0 .. n0 + ng - 1 of Xq, us, Y and partials,
    // columns n0 .. of da (n0 a multiple of 32: 16-byte aligned)
    for (int n0 = 0; n0 < N; n0 += Q6_Q4K_GROUP_N) {
      const int ng = N - n0 < Q6_Q4K_GROUP_N ? N - n0 : Q6_Q4K_GROUP_N;
      int32_t* pg = partials ? partials + (size_t)n0 * M * (K / 32) : nullptr;
      const int8_t* xg = Xq + (size_t)n0 * K;
      const float* ug = us + (size_t)n0 * ldus;
      float* yg = Y + (size_t)n0 * ldy;
      cudaError_t e =
          ng <= Q6_Q4K_DP4A_MAX_N
              ? q6::launch_q4k_skinny(pb, M, K, xg, da + n0, ldda_of(N), ug, ng, yg, ldy, pg,
                                      (cudaStream_t)s)
              : q6::launch_q4k_skinny_mma(pb, M, K, xg, da + n0, ldda_of(N), ug, ng, yg, ldy, pg,
                                          st->status, (cudaStream_t)s);
      if (e != cudaSuccess) return cuda_fail(e, "q4_K few-token kernel launch");
    }
    if (path_out) *path_out = Q6_PATH_Q4K_SKINNY;
    return Q6_OK;
  }
  if (!wq || partials) {
    const size_t need = (size_t)M * (size_t)K * 2;
    if (!workspace || workspace_bytes < need)
      return fail(Q6_ESIZE, "workspace of %zu bytes needed to unpack the weights (got %zu)", need,
                  workspace ? workspace_bytes : (size_t)0);
  }
  DevState* st;
  int rc = device_state(&st);
  if (rc) return rc;
  const uint8_t* pb = static_cast<const uint8_t*>(plane);
  __half* ws = static_cast<__half*>(workspace);
  cudaError_t e;
  const void* wop = wq;
  int path = Q6_PATH_Q4K_TC_WQ;
  if (!wq) {
    if ((e = q6::launch_q4k_expand(pb, M, K, false, ws, (cudaStream_t)s)) != cudaSuccess)
      return cuda_fail(e, "q4_K weight unpack launch");
    wop = ws;
    path = Q6_PATH_Q4K_TC_RAW;
  }
  q6::TcMaps maps;
  if ((rc = q6::encode_tc_maps_q4k(&maps, pb, wop, Xh, da, us, M, K, N))) return rc;
  float* part = nullptr;
  if ((rc = part_buffer(M, K, N, workspace, workspace_bytes,
                        (!wq || partials) ? (size_t)M * (size_t)K * 2 : 0, &part)))
    return rc;
  e = q6::launch_mmq_tc_q4k(maps, M, K, N, Y, ldy, q6::TcDebugOut{}, st->status, (cudaStream_t)s,
                            part);
  if (e != cudaSuccess) return cuda_fail(e, "q4_K tensor-core kernel launch");
  if (partials) {
    // the per-sub-block P = sum q * xq: one more launch on the plane of the
    // raw nibbles (unit scale), writing the chunk accumulators and not Y
    if ((e = q6::launch_q4k_expand(pb, M, K, true, ws, (cudaStream_t)s)) != cudaSuccess)
      return cuda_fail(e, "q4_K debug unpack launch");
    if ((rc = q6::encode_tc_maps_q4k(&maps, pb, ws, Xh, da, us, M, K, N))) return rc;
    q6::TcDebugOut dbg;
    dbg.out = partials;
    dbg.stride = K / 32;
    dbg.write_y = 0;
    if ((e = q6::launch_mmq_tc_q4k(maps, M, K, N, Y, ldy, dbg, st->status, (cudaStream_t)s)))
      return cuda_fail(e, "q4_K debug kernel launch");
  }
  if (path_out) *path_out = path;
  return Q6_OK;
}

}  // extern "C"
