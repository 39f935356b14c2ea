// Load-time weight packing: raw GGUF q6_K super-blocks -> the packed plane
// (qlh / sc / d / d^T sub-planes) and, optionally, the W_exp plane.
//
// Element map ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 3.2): a
// super-block is two 128-element halves; inside half h, element r takes its
// low 4 bits from ql[64h + r%64] (low nibble if r < 64, else high) and its
// high 2 bits from field floor(r/32) of qh[32h + r%32]; the value is code - 32.
// The qlh sub-plane keeps each half's 64 ql bytes and 32 qh bytes together so
// one 96-byte TMA row carries everything the unpack of that half needs.
// The super-block scale d is kept twice: as the raw binary16 bits [M][K/256]
// (rows padded to 16 bytes, padding zero) and as f32 transposed to [K/256][ldm] (weight rows contiguous, rows M..ldm-1
// zero) so the GEMM can stage the d of 128 rows with one TMA copy. W_exp =
// centered int8, row stride K ("r53 -- q6_K bundle: W_exp pre-expansion
// plane", Sec. 2.3).
//
// One warp per super-block: lanes copy the 192 ql/qh bytes, the scales and,
// for W_exp, expand eight elements each.
#include "q6_internal.cuh"

namespace q6 {
namespace {

__global__ void __launch_bounds__(256) q6k_pack_kernel(const uint8_t* __restrict__ raw, int M, int K,
                                                       uint8_t* __restrict__ plane, PlaneGeom g,
                                                       int8_t* __restrict__ wexp) {
  const int nsb = K / 256;
  const long long nblk = (long long)M * nsb;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long i = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < nblk;
       i += warps) {
    const int m = (int)(i / nsb), b = (int)(i - (long long)m * nsb);
    const uint8_t* src = raw + (size_t)i * 210;
    // qlh: half h -> 96 bytes at (2b + h) * 96 of row m.
    uint8_t* qlh = plane + g.qlh_off + (size_t)m * g.qlh_row + (size_t)b * 192;
    for (int t = lane; t < 192; t += 32) {
      const int h = t / 96, o = t - 96 * h;
      qlh[t] = (o < 64) ? src[64 * h + o] : src[128 + 32 * h + (o - 64)];
    }
    const uint16_t dbits = (uint16_t)(src[208] | (src[209] << 8));
    if (lane < 16) {
      const size_t si = (size_t)m * (K / 16) + (size_t)b * 16 + lane;
      reinterpret_cast<int8_t*>(plane + g.sc_off)[si] = (int8_t)src[192 + lane];
    } else if (lane == 16) {
      reinterpret_cast<uint16_t*>(plane + g.d_off + (size_t)m * g.d_row)[b] = dbits;
    } else if (lane == 17) {
      reinterpret_cast<float*>(plane + g.dt_off)[(size_t)b * g.ldm + m] =
          __half2float(__ushort_as_half(dbits));
    }
    if (wexp != nullptr) {
      // lane -> ql byte pair group: half h = lane / 16, bytes j0 = 4*(lane % 16) .. +3,
      // giving elements 128h + j and 128h + j + 64 for the four j.
      const int h = lane >> 4, j0 = 4 * (lane & 15);
      uint32_t lo_word = 0, hi_word = 0;
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        const uint32_t l = src[64 * h + j];
        const uint32_t qh = src[128 + 32 * h + (j & 31)];
        const int f = 2 * (j >> 5);                 // field of element j; j + 64 uses f + 4
        const uint32_t c0 = (l & 15u) | (((qh >> f) & 3u) << 4);
        const uint32_t c1 = (l >> 4) | (((qh >> (f + 4)) & 3u) << 4);
        lo_word |= ((c0 - 32u) & 0xFFu) << (8 * u);
        hi_word |= ((c1 - 32u) & 0xFFu) << (8 * u);
      }
      int8_t* dst = wexp + (size_t)m * K + (size_t)b * 256 + 128 * h;
      reinterpret_cast<uint32_t*>(dst + j0)[0] = lo_word;
      reinterpret_cast<uint32_t*>(dst + 64 + j0)[0] = hi_word;
    }
  }
  // padding of the binary16 d rows
  const int dpad = (int)(g.d_row / 2) - nsb;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)M * dpad;
       i += (long long)gridDim.x * blockDim.x)
    reinterpret_cast<uint16_t*>(plane + g.d_off + (size_t)(i / dpad) * g.d_row)[nsb + (int)(i % dpad)] =
        0;
  // the gaps that round each sub-plane up to 256 bytes (so that equal
  // weights give byte-equal planes)
  {
    const size_t ends[4] = {(size_t)M * g.qlh_row, g.sc_off + (size_t)M * (K / 16),
                            g.d_off + (size_t)M * g.d_row,
                            g.dt_off + (size_t)nsb * (size_t)g.ldm * 4};
    const size_t starts[4] = {g.sc_off, g.d_off, g.dt_off, g.total};
    if (blockIdx.x == 0)
      for (int r = 0; r < 4; ++r)
        for (size_t i = ends[r] + threadIdx.x; i < starts[r]; i += blockDim.x) plane[i] = 0;
  }
  // rows M .. ldm-1 of the transposed d sub-plane
  const int pad = g.ldm - M;
  const long long npad = (long long)pad * nsb;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long i = tid; i < npad; i += (long long)gridDim.x * blockDim.x)
    reinterpret_cast<float*>(plane + g.dt_off)[(size_t)(i / pad) * g.ldm + M + (size_t)(i % pad)] =
        0.0f;
}

}  // namespace

cudaError_t launch_pack(const uint8_t* raw, int M, int K, uint8_t* plane, int8_t* wexp,
                        cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  const long long nblk = (long long)M * (K / 256);
  long long blocks = (nblk + 7) / 8;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  q6k_pack_kernel<<<(unsigned)blocks, 256, 0, s>>>(raw, M, K, plane, g, wexp);
  return cudaGetLastError();
}

}  // namespace q6
