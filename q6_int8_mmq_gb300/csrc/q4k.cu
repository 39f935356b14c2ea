// The q4_K weight format: load-time packing and the unpack to the tensor-core
// GEMM's binary16 operand plane.
//
// Block ("r18: Load-time B pre-expansion -- staging becomes a bulk copy",
// Sec. 1 and 3.2): 144 bytes per 256 weights; d (f16) at byte 0, dmin (f16) at
// byte 2, eight 6-bit scales and eight 6-bit mins packed in the 12 bytes at
// byte 4, and 128 bytes of nibbles at byte 16, where the 32 bytes of nibble
// pair p (0..3) hold sub-block 2p in their low nibbles and sub-block 2p + 1 in
// their high nibbles, element-ordered. The weight is d * sc[j] * q - dmin *
// m[j] for sub-block j (32 elements), q the raw nibble 0..15; the GEMM's
// rescale has the two terms of "r38 -- q6_K BT-style raw-byte mma kernel",
// Sec. 2.2. The pages call the helper that unpacks the 12 scale bytes but do
// not print it; it is read as the GGUF q4_K layout (sub-blocks 0..3: the low
// 6 bits of bytes j and j + 4; sub-blocks 4..7: the nibbles of byte j + 4 as
// the low 4 bits, the top two bits of bytes j - 4 and j as bits 4-5).
//
// Packed plane (all sub-planes 256-byte aligned, gaps zero):
//   qs  : uint8 [M][K/2], each block's 128 nibble bytes as they are;
//   sc  : uint8 [M][K/32], the decoded 6-bit scales;
//   mn  : uint8 [M][K/32], the decoded 6-bit mins;
//   dT  : f32 [K/256][ldm], d as f32 (exact), transposed, rows M..ldm-1 zero;
//   mvp : f32 [M][q4_min_ld(K)], dmin * m (at most 11 + 6 = 17 significant
//         bits) as the exact tf32 pair hi + lo: per super-block b, the hi
//         parts of its 8 chunks at 16 b .. 16 b + 7 and the lo parts at
//         16 b + 8 .. 16 b + 15; an odd super-block count leaves 16 zeros at
//         the end of each row. The GEMM's min term runs on the tensor cores
//         from these pairs (kind::tf32);
//   ddm : float2 [M][K/256], (d, dmin) of each super-block as f32 (exact),
//         row-major, for the few-token kernel.
// Operand plane (the unpack): binary16 [M][K], sc[j] * q (at most 63 * 15 =
// 945, exact), or with unit scale q alone (the debug partials).
#include "q6_internal.cuh"

namespace q6 {
namespace {

// The scale (kMin = false) or min of sub-block j from the 12 packed bytes.
__device__ __forceinline__ int q4_unpack6(const uint8_t* s, int j, bool min) {
  if (j < 4) return s[j + (min ? 4 : 0)] & 63;
  const int low = min ? (s[j + 4] >> 4) : (s[j + 4] & 15);
  const int top = s[min ? j : j - 4] >> 6;
  return low | (top << 4);
}

// One warp per super-block.
__global__ void __launch_bounds__(256) q4k_pack_kernel(const uint8_t* __restrict__ raw, int M, int K,
                                                       uint8_t* __restrict__ plane, Q4Geom g) {
  const int nsb = K / 256;
  const long long nblk = (long long)M * nsb;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < nblk;
       i += warps) {
    const int m = (int)(i / nsb), b = (int)(i - (long long)m * nsb);
    const uint8_t* src = raw + (size_t)i * 144;
    uint8_t* qs = plane + g.qs_off + (size_t)m * (K / 2) + (size_t)b * 128;
    for (int t = lane; t < 128; t += 32) qs[t] = src[16 + t];
    if (lane < 8) {
      const int sc = q4_unpack6(src + 4, lane, false), mn = q4_unpack6(src + 4, lane, true);
      const size_t c = (size_t)b * 8 + lane;
      plane[g.sc_off + (size_t)m * (K / 32) + c] = (uint8_t)sc;
      plane[g.mn_off + (size_t)m * (K / 32) + c] = (uint8_t)mn;
      const float dmin = __half2float(__ushort_as_half((unsigned short)(src[2] | (src[3] << 8))));
      float hi, lo;
      tf32_split(dmin * (float)mn, hi, lo);
      float* mv = reinterpret_cast<float*>(plane + g.mv_off) + (size_t)m * q4_min_ld(K) + 16 * b;
      mv[lane] = hi;
      mv[8 + lane] = lo;
      if ((nsb & 1) && b == nsb - 1) {  // the odd super-block count's padding
        mv[16 + lane] = 0.0f;
        mv[24 + lane] = 0.0f;
      }
    } else if (lane == 8) {
      reinterpret_cast<float*>(plane + g.dt_off)[(size_t)b * g.ldm + m] =
          __half2float(__ushort_as_half((unsigned short)(src[0] | (src[1] << 8))));
    } else if (lane == 9) {
      reinterpret_cast<float2*>(plane + g.ddm_off)[i] =
          make_float2(__half2float(__ushort_as_half((unsigned short)(src[0] | (src[1] << 8)))),
                      __half2float(__ushort_as_half((unsigned short)(src[2] | (src[3] << 8)))));
    }
  }
  // rows M .. ldm-1 of the transposed d sub-plane, and the gaps between sub-planes
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthr = (long long)gridDim.x * blockDim.x;
  const int pad = g.ldm - M;
  for (long long j = tid; j < (long long)pad * nsb; j += nthr) {
    const long long r = j / pad;
    const int col = M + (int)(j - r * pad);
    reinterpret_cast<float*>(plane + g.dt_off)[(size_t)r * g.ldm + col] = 0.0f;
  }
  if (blockIdx.x == 0) {
    const size_t ends[6] = {(size_t)M * (K / 2), g.sc_off + (size_t)M * (K / 32),
                            g.mn_off + (size_t)M * (K / 32), g.dt_off + (size_t)nsb * g.ldm * 4,
                            g.mv_off + (size_t)M * q4_min_ld(K) * 4,
                            g.ddm_off + (size_t)nblk * 8};
    const size_t starts[6] = {g.sc_off, g.mn_off, g.dt_off, g.mv_off, g.ddm_off, g.total};
    for (int r = 0; r < 6; ++r)
      for (size_t j = ends[r] + threadIdx.x; j < starts[r]; j += blockDim.x) plane[j] = 0;
  }
}

// Eight consecutive elements of one sub-block per thread: their nibbles from
// 8 bytes of the block's nibble run, each as binary16 (1024 + q) - 1024 = q,
// times the sub-block scale (exact: sc * q <= 945).
template <bool kUnit>
__global__ void __launch_bounds__(256) q4k_expand_kernel(const uint8_t* __restrict__ qs,
                                                         const uint8_t* __restrict__ scp,
                                                         long long n8, int K,
                                                         __half* __restrict__ wq) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6400));  // 1024
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const long long e0 = 8 * i;                   // first element (row-major [M][K])
    const long long m = e0 / K;
    const int k = (int)(e0 - m * K);
    const int b = k >> 8, c = (k >> 5) & 7, t = k & 31;
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(qs + (size_t)m * (K / 2) + (size_t)b * 128 +
                                                         32 * (c >> 1) + t));
    const uint32_t sh = (c & 1) ? 4u : 0u;
    const uint32_t lo = (w.x >> sh) & 0x0F0F0F0Fu, hi = (w.y >> sh) & 0x0F0F0F0Fu;
    const int sc = kUnit ? 1 : (int)__ldg(scp + (size_t)m * (K / 32) + (k >> 5));
    const __half2 f = __half2half2(__int2half_rn(sc));
    uint32_t o[4];
    const uint32_t words[2] = {lo, hi};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t a = __byte_perm(words[h], 0x64646464u, 0x4140);
      uint32_t bb = __byte_perm(words[h], 0x64646464u, 0x4342);
      const __half2 ha = __hmul2(__hsub2(*reinterpret_cast<__half2*>(&a), bias), f);
      const __half2 hb = __hmul2(__hsub2(*reinterpret_cast<__half2*>(&bb), bias), f);
      o[2 * h] = *reinterpret_cast<const uint32_t*>(&ha);
      o[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&hb);
    }
    *reinterpret_cast<uint4*>(wq + e0) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

unsigned grid_of(long long items) {
  long long blocks = (items + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  return (unsigned)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_q4k_pack(const uint8_t* raw, int M, int K, uint8_t* plane, cudaStream_t s) {
  const Q4Geom g = q4_geom(M, K);
  const long long nblk = (long long)M * (K / 256);
  long long blocks = (nblk + 7) / 8;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  q4k_pack_kernel<<<(unsigned)blocks, 256, 0, s>>>(raw, M, K, plane, g);
  return cudaGetLastError();
}

cudaError_t launch_q4k_expand(const uint8_t* plane, int M, int K, bool unit, __half* wq,
                              cudaStream_t s) {
  const Q4Geom g = q4_geom(M, K);
  const long long n8 = (long long)M * K / 8;
  if (unit)
    q4k_expand_kernel<true><<<grid_of(n8), 256, 0, s>>>(plane + g.qs_off, plane + g.sc_off, n8, K, wq);
  else
    q4k_expand_kernel<false><<<grid_of(n8), 256, 0, s>>>(plane + g.qs_off, plane + g.sc_off, n8, K,
                                                        wq);
  return cudaGetLastError();
}

}  // namespace q6
