// q6_K x int8 GEMM for few tokens (N <= 16): a weight-streaming kernel on the
// CUDA cores, bound by HBM (0.82 byte per weight).
//
// Math ("r38 -- q6_K BT-style raw-byte mma kernel", Sec. 2.1-2.2): for each
// 16-element sub-block s the exact integer P = sum (q - 32) * xq is formed
// with dp4a, then Y += (f32(d) * sc[s]) * da[chunk] * P. The element map is
// the one of Sec. 3.2 (see pack.cu).
//
// Work split: one warp per weight row; per iteration a warp covers four
// super-blocks, eight lanes per super-block. Lane (half, s4) of a super-block
// reads the 16 ql bytes at 16*s4 of its half and the 16 qh bytes at
// 16*(s4&1): the low nibbles give sub-block 8*half + s4, the high nibbles
// (same bytes) sub-block 8*half + s4 + 4; their 2-bit fields sit at bits
// 2*(s4>>1) and 2*(s4>>1) + 4 of the qh bytes.
#include "q6_internal.cuh"

namespace q6 {
namespace {

constexpr int kWarps = 8;

// Bytes (code - 32) mod 256 of four 6-bit codes: code + 96 never carries out
// of its byte, and adding 128 more is a flip of bit 7.
__device__ __forceinline__ uint32_t center4(uint32_t code) {
  return (code + 0x60606060u) ^ 0x80808080u;
}

template <bool kPartials>
__global__ void __launch_bounds__(kWarps * 32) mmq_skinny_kernel(
    const uint8_t* __restrict__ plane, PlaneGeom g, int M, int K, const int8_t* __restrict__ Xq,
    const float* __restrict__ da, int ldda, int N, float* __restrict__ Y, int ldy,
    int32_t* __restrict__ partials) {
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (m >= M) return;
  const int nsb = K / 256;
  const int sbi = lane >> 3;        // super-block within the iteration
  const int half = (lane >> 2) & 1;
  const int s4 = lane & 3;
  const int fsh = 2 * (s4 >> 1);    // field of the low-nibble sub-block

  const uint8_t* qlh_row = plane + g.qlh_off + (size_t)m * g.qlh_row;
  const int8_t* sc_row = reinterpret_cast<const int8_t*>(plane + g.sc_off) + (size_t)m * (K / 16);
  const uint16_t* d_row = reinterpret_cast<const uint16_t*>(plane + g.d_off) + (size_t)m * nsb;

  float acc[Q6_SKINNY_MAX_N];
#pragma unroll
  for (int n = 0; n < Q6_SKINNY_MAX_N; ++n) acc[n] = 0.0f;

  for (int sb0 = 0; sb0 < nsb; sb0 += 4) {
    const int sb = sb0 + sbi;
    if (sb < nsb) {
      const uint8_t* hb = qlh_row + (size_t)(2 * sb + half) * 96;
      const uint4 L = *reinterpret_cast<const uint4*>(hb + 16 * s4);
      const uint4 H = *reinterpret_cast<const uint4*>(hb + 64 + 16 * (s4 & 1));
      const uint32_t Lw[4] = {L.x, L.y, L.z, L.w};
      const uint32_t Hw[4] = {H.x, H.y, H.z, H.w};
      uint32_t va[4], vb[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t ca = (Lw[w] & 0x0F0F0F0Fu) | (((Hw[w] >> fsh) & 0x03030303u) << 4);
        const uint32_t cb = ((Lw[w] >> 4) & 0x0F0F0F0Fu) | (((Hw[w] >> (fsh + 4)) & 0x03030303u) << 4);
        va[w] = center4(ca);
        vb[w] = center4(cb);
      }
      const int sa = 8 * half + s4;  // sub-block (0..15) of the low nibbles; sb_b = sa + 4
      const float d = __half2float(__ushort_as_half(d_row[sb]));
      const int sc_a = sc_row[16 * sb + sa], sc_b = sc_row[16 * sb + sa + 4];
      const float dsc_a = d * (float)sc_a;
      const float dsc_b = d * (float)sc_b;
      const int ka = 256 * sb + 16 * sa;  // first element of sub-block a
      const int ca_blk = ka >> 5, cb_blk = (ka + 64) >> 5;
#pragma unroll
      for (int n = 0; n < Q6_SKINNY_MAX_N; ++n) {
        if (n < N) {
          const int8_t* xr = Xq + (size_t)n * K;
          const uint4 xa = *reinterpret_cast<const uint4*>(xr + ka);
          const uint4 xb = *reinterpret_cast<const uint4*>(xr + ka + 64);
          int pa = __dp4a((int)va[0], (int)xa.x, 0);
          pa = __dp4a((int)va[1], (int)xa.y, pa);
          pa = __dp4a((int)va[2], (int)xa.z, pa);
          pa = __dp4a((int)va[3], (int)xa.w, pa);
          int pb = __dp4a((int)vb[0], (int)xb.x, 0);
          pb = __dp4a((int)vb[1], (int)xb.y, pb);
          pb = __dp4a((int)vb[2], (int)xb.z, pb);
          pb = __dp4a((int)vb[3], (int)xb.w, pb);
          const float daa = da[(size_t)ca_blk * ldda + n];
          const float dab = da[(size_t)cb_blk * ldda + n];
          acc[n] = fmaf(dsc_a * daa, (float)pa, acc[n]);
          acc[n] = fmaf(dsc_b * dab, (float)pb, acc[n]);
          if (kPartials) {
            // chunk partials sc*P summed over the chunk's two sub-blocks; the
            // other sub-block of each chunk is in lane ^ 1 (active together)
            const unsigned act = __activemask();
            const int ta = sc_a * pa, tb = sc_b * pb;
            const int sa2 = ta + __shfl_xor_sync(act, ta, 1);
            const int sb2 = tb + __shfl_xor_sync(act, tb, 1);
            if ((s4 & 1) == 0) {
              int32_t* pr = partials + ((size_t)n * M + m) * (size_t)(K / 32) + (size_t)sb * 8;
              pr[sa >> 1] = sa2;
              pr[(sa + 4) >> 1] = sb2;
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int n = 0; n < Q6_SKINNY_MAX_N; ++n) {
    if (n < N) {
      float v = acc[n];
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) Y[(size_t)n * ldy + m] = v;
    }
  }
}

}  // namespace

cudaError_t launch_mmq_skinny(const uint8_t* plane, int M, int K, const int8_t* Xq, const float* da,
                              int ldda, int N, float* Y, int ldy, int32_t* partials,
                              cudaStream_t s) {
  const PlaneGeom g = plane_geom(M, K);
  const unsigned blocks = (unsigned)((M + kWarps - 1) / kWarps);
  if (partials)
    mmq_skinny_kernel<true><<<blocks, kWarps * 32, 0, s>>>(plane, g, M, K, Xq, da, ldda, N, Y, ldy,
                                                           partials);
  else
    mmq_skinny_kernel<false><<<blocks, kWarps * 32, 0, s>>>(plane, g, M, K, Xq, da, ldda, N, Y,
                                                            ldy, nullptr);
  return cudaGetLastError();
}

}  // namespace q6
