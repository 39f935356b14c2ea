// Weight unpack pass: q6_K codes and sub-block scales -> the two binary16
// operand planes W_hi, W_lo [M][K] that the tensor-core GEMM stages with TMA.
//
// Element map ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 3.2; the
// 16-element group form of "r41 -- q6_K B-expand widened to uint4 group
// loads", Sec. 3.2): within a 128-element half block, 16-element group g
// takes its low 4 bits from the 16 ql bytes at 16*(g mod 4) (low nibble for
// g < 4, high nibble otherwise) and its high 2 bits from field (g/2) mod 4 of
// the 16 qh bytes at 16*(g mod 2); the value is v = code - 32, in [-32, 31].
// The W_exp source ("r53 -- q6_K bundle: W_exp pre-expansion plane",
// Sec. 2.3) already holds v as int8. Each 16-element group is one sub-block.
//
// The sub-block scale sc (int8) is folded into the operand, split so both
// parts stay exact in binary16: sc = 16*sh + sl with sh = floor(sc/16) in
// [-8, 7] and sl in [0, 15]; W_hi = 16*sh*v (|.| <= 4096, a multiple of 16
// with at most 9 significant bits) and W_lo = sl*v (|.| <= 480). So
// W_hi + W_lo = sc * v exactly, and two MMAs over the same activation
// operand give the integer sum of sc * v * xq of a sub-block.
//
// Both kernels are bandwidth-bound (0.81 or 1.06 bytes read and 4 written per
// weight).
#include "q6_internal.cuh"

namespace q6 {
namespace {

// Four 6-bit codes -> two binary16 pairs holding code - 32 exactly: bytes
// 0x64cc are the f16 value 1024 + cc, and subtracting 1056 leaves cc - 32.
__device__ __forceinline__ void codes_to_f16(uint32_t code, uint32_t& lo, uint32_t& hi) {
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6420));  // 1056
  uint32_t a = __byte_perm(code, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(code, 0x64646464u, 0x4342);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// Four int8 values -> two binary16 pairs: flipping bit 7 gives v + 128 as an
// unsigned byte, 0x64xx is 1024 + that, and subtracting 1152 leaves v.
__device__ __forceinline__ void i8_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// o[8] (sixteen binary16 v) -> W_hi and W_lo runs of one sub-block.
__device__ __forceinline__ void store_folded(const uint32_t (&o)[8], int sc, __half* hi, __half* lo) {
  const int sh = sc >> 4, sl = sc & 15;  // arithmetic shift: floor(sc / 16)
  const __half2 fh = __half2half2(__int2half_rn(16 * sh));
  const __half2 fl = __half2half2(__int2half_rn(sl));
  uint32_t h[8], l[8];
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const __half2 v = *reinterpret_cast<const __half2*>(&o[w]);
    const __half2 a = __hmul2(v, fh), b = __hmul2(v, fl);
    h[w] = *reinterpret_cast<const uint32_t*>(&a);
    l[w] = *reinterpret_cast<const uint32_t*>(&b);
  }
  uint4* dh = reinterpret_cast<uint4*>(hi);
  uint4* dl = reinterpret_cast<uint4*>(lo);
  dh[0] = make_uint4(h[0], h[1], h[2], h[3]);
  dh[1] = make_uint4(h[4], h[5], h[6], h[7]);
  dl[0] = make_uint4(l[0], l[1], l[2], l[3]);
  dl[1] = make_uint4(l[4], l[5], l[6], l[7]);
}

// One thread per 32-element chunk (two sub-blocks of one half block): its
// two 16-byte ql runs and the half block's 32 qh bytes are loaded together
// before any conversion.
__global__ void __launch_bounds__(256) expand_raw_kernel(const uint8_t* __restrict__ qlh,
                                                         const int8_t* __restrict__ sc, int M, int K,
                                                         size_t qlh_row, __half* __restrict__ wh) {
  const int chunks = K / 32;
  const long long items = (long long)M * chunks;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const size_t plane = (size_t)M * K;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < items; i += stride) {
    const int m = (int)(i / chunks), c = (int)(i - (long long)m * chunks);
    const int hb = c >> 2, g0 = 2 * (c & 3);  // half block, first group (even) within it
    const uint8_t* src = qlh + (size_t)m * qlh_row + (size_t)hb * 96;
    const uint4 La = __ldg(reinterpret_cast<const uint4*>(src + 16 * (g0 & 3)));
    const uint4 Lb = __ldg(reinterpret_cast<const uint4*>(src + 16 * ((g0 + 1) & 3)));
    const uint4 H0 = __ldg(reinterpret_cast<const uint4*>(src + 64));
    const uint4 H1 = __ldg(reinterpret_cast<const uint4*>(src + 80));
    const uint16_t s2 = __ldg(reinterpret_cast<const uint16_t*>(sc + 2 * i));
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int g = g0 + u;
      const uint4 L = u ? Lb : La;
      const uint4 H = (g & 1) ? H1 : H0;
      const int nsh = 4 * (g >> 2), fsh = 2 * ((g >> 1) & 3);
      const uint32_t Lw[4] = {L.x, L.y, L.z, L.w}, Hw[4] = {H.x, H.y, H.z, H.w};
      uint32_t o[8];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t code = ((Lw[w] >> nsh) & 0x0F0F0F0Fu) | (((Hw[w] >> fsh) & 0x03030303u) << 4);
        codes_to_f16(code, o[2 * w], o[2 * w + 1]);
      }
      const int scv = (int)(int8_t)(u ? (s2 >> 8) : (s2 & 0xFF));
      const size_t off = (size_t)m * K + (size_t)(2 * c + u) * 16;
      store_folded(o, scv, wh + off, wh + plane + off);
    }
  }
}

__global__ void __launch_bounds__(256) expand_wexp_kernel(const int8_t* __restrict__ wexp,
                                                          const int8_t* __restrict__ sc, long long n16,
                                                          __half* __restrict__ wh) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const size_t plane = (size_t)n16 * 16;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(wexp) + i);
    const int s = __ldg(sc + i);
    uint32_t o[8];
    i8_to_f16(v.x, o[0], o[1]);
    i8_to_f16(v.y, o[2], o[3]);
    i8_to_f16(v.z, o[4], o[5]);
    i8_to_f16(v.w, o[6], o[7]);
    store_folded(o, s, wh + 16 * (size_t)i, wh + plane + 16 * (size_t)i);
  }
}

unsigned grid_for(long long items) {
  long long blocks = (items + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  return (unsigned)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_expand_raw(const uint8_t* plane, int M, int K, __half* wh, cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  expand_raw_kernel<<<grid_for((long long)M * (K / 32)), 256, 0, s>>>(
      plane + g.qlh_off, reinterpret_cast<const int8_t*>(plane + g.sc_off), M, K, g.qlh_row, wh);
  return cudaGetLastError();
}

cudaError_t launch_expand_wexp(const int8_t* wexp, const uint8_t* plane, int M, int K, __half* wh,
                               cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  const long long n16 = (long long)M * K / 16;
  expand_wexp_kernel<<<grid_for(n16), 256, 0, s>>>(
      wexp, reinterpret_cast<const int8_t*>(plane + g.sc_off), n16, wh);
  return cudaGetLastError();
}

}  // namespace q6
