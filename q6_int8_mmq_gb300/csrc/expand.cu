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
// weight); each warp's stores cover whole 512-byte runs.
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

// o[4] (eight binary16 v of one sub-block) -> 16 bytes of W_hi and of W_lo.
__device__ __forceinline__ void store_folded8(const uint32_t (&o)[4], int sc, __half* hi, __half* lo) {
  const int sh = sc >> 4, sl = sc & 15;  // arithmetic shift: floor(sc / 16)
  const __half2 fh = __half2half2(__int2half_rn(16 * sh));
  const __half2 fl = __half2half2(__int2half_rn(sl));
  uint32_t h[4], l[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const __half2 v = *reinterpret_cast<const __half2*>(&o[w]);
    const __half2 a = __hmul2(v, fh), b = __hmul2(v, fl);
    h[w] = *reinterpret_cast<const uint32_t*>(&a);
    l[w] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

// One warp per super-block, lane l owning its elements 8l .. 8l + 7 (half p =
// l % 2 of sub-block s = l / 2), so that each 16-byte store of the warp lands
// in one contiguous 512-byte run of W_hi or W_lo. A lane reads the 8 ql bytes
// and the 8 qh bytes of its elements (sub-block s of half h = s / 8 is group
// j = s % 8 of the element map) and the sub-block's scale.
// kUnit (debug planes): the scale is replaced by 1 on the sub-blocks of
// parity `parity` and by 0 on the others, so W_hi = 0 and W_lo is v or 0.
template <bool kUnit>
__global__ void __launch_bounds__(256) expand_raw_kernel(const uint8_t* __restrict__ qlh,
                                                         const int8_t* __restrict__ sc, int M, int K,
                                                         size_t qlh_row, int parity,
                                                         __half* __restrict__ wh) {
  const int nsb = K / 256;
  const long long blocks = (long long)M * nsb;  // super-blocks
  const long long wstride = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  const int s = lane >> 1, p = lane & 1, h = s >> 3, j = s & 7;
  const int nsh = 4 * (j >> 2), fsh = 2 * (j >> 1);
  const size_t plane = (size_t)M * K;
  for (long long b = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < blocks;
       b += wstride) {
    const int m = (int)(b / nsb), sb = (int)(b - (long long)m * nsb);
    const uint8_t* src = qlh + (size_t)m * qlh_row + (size_t)sb * 192 + 96 * h;
    const uint2 L = __ldg(reinterpret_cast<const uint2*>(src + 16 * (j & 3) + 8 * p));
    const uint2 H = __ldg(reinterpret_cast<const uint2*>(src + 64 + 16 * (j & 1) + 8 * p));
    const int scv = kUnit ? (int)((s & 1) == parity) : __ldg(sc + (size_t)m * (K / 16) + 16 * sb + s);
    uint32_t o[4];
    codes_to_f16(((L.x >> nsh) & 0x0F0F0F0Fu) | (((H.x >> fsh) & 0x03030303u) << 4), o[0], o[1]);
    codes_to_f16(((L.y >> nsh) & 0x0F0F0F0Fu) | (((H.y >> fsh) & 0x03030303u) << 4), o[2], o[3]);
    const size_t off = (size_t)m * K + (size_t)sb * 256 + 8 * lane;
    store_folded8(o, scv, wh + off, wh + plane + off);
  }
}

// The same from the W_exp plane: one thread per eight elements.
__global__ void __launch_bounds__(256) expand_wexp_kernel(const int8_t* __restrict__ wexp,
                                                          const int8_t* __restrict__ sc, long long n8,
                                                          __half* __restrict__ wh) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const size_t plane = (size_t)n8 * 8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(wexp) + i);
    const int s = __ldg(sc + (i >> 1));
    uint32_t o[4];
    i8_to_f16(v.x, o[0], o[1]);
    i8_to_f16(v.y, o[2], o[3]);
    store_folded8(o, s, wh + 8 * (size_t)i, wh + plane + 8 * (size_t)i);
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
  expand_raw_kernel<false><<<grid_for((long long)M * (K / 256) * 32), 256, 0, s>>>(
      plane + g.qlh_off, reinterpret_cast<const int8_t*>(plane + g.sc_off), M, K, g.qlh_row, 0, wh);
  return cudaGetLastError();
}

cudaError_t launch_expand_unit(const uint8_t* plane, int M, int K, int parity, __half* wh,
                               cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  expand_raw_kernel<true><<<grid_for((long long)M * (K / 256) * 32), 256, 0, s>>>(
      plane + g.qlh_off, nullptr, M, K, g.qlh_row, parity, wh);
  return cudaGetLastError();
}

cudaError_t launch_expand_wexp(const int8_t* wexp, const uint8_t* plane, int M, int K, __half* wh,
                               cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  const long long n8 = (long long)M * K / 8;
  expand_wexp_kernel<<<grid_for(n8), 256, 0, s>>>(
      wexp, reinterpret_cast<const int8_t*>(plane + g.sc_off), n8, wh);
  return cudaGetLastError();
}

}  // namespace q6
