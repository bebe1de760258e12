// Shared pieces of the CUDA-core W4A4 product: the block dot product of a
// weight row against activation rows held in shared memory as FP16 E2M1 values,
// and the expansion of activation rows into that layout.
#pragma once

#include "common.cuh"

namespace gdn {

// A "piece" is 32 elements (two 16-blocks): 16 code bytes + 2 scale bytes.
// Lane l handles pieces l, l+32, ... of a row, so a warp's 128-bit shared loads
// are contiguous. Activations live in shared memory as FP16 E2M1 values:
//   xh[((m * 2 + blk) * 2 + half) * npiece + p] : uint4 = 4 half2 (8 values)
//   xs[(m * 2 + blk) * npiece + p]              : float E4M3 block scale

// NP = number of pieces per row when known at compile time (a multiple of
// 32: every lane then takes NP/32 pieces, fully unrolled, with constant shared
// offsets), 0 = npiece at run time. The arithmetic is the same either way.
template <int MB, int NP = 0>
GDN_DEV void dot_row(const uint8_t *codes, const uint8_t *scales, int npiece, int M, const uint4 *xh,
                     const float *xs, int lane, float (&acc)[MB]) {
  static_assert(NP % 32 == 0, "NP multiple of 32");
  const int np = NP ? NP : npiece;
  const int iters = NP ? NP / 32 : (npiece - lane + 31) / 32;
#pragma unroll
  for (int it = 0; it < (NP ? NP / 32 : iters); ++it) {
    const int p = lane + 32 * it;
    const uint4 wc = *reinterpret_cast<const uint4 *>(codes + (size_t)p * 16);
    const uint32_t ws = *reinterpret_cast<const uint16_t *>(scales + (size_t)p * 2);
    float swv[2];
    {  // both blocks' weight scales with one conversion (exact)
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(ws)));
      swv[0] = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
      swv[1] = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
    }
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint32_t w0 = blk == 0 ? wc.x : wc.z;
      const uint32_t w1 = blk == 0 ? wc.y : wc.w;
      __half2 wv[8];
      e2m1x8_to_h2x4(w0, *reinterpret_cast<__half2(*)[4]>(&wv[0]));
      e2m1x8_to_h2x4(w1, *reinterpret_cast<__half2(*)[4]>(&wv[4]));
      const float sw = swv[blk];
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (m < M) {
          const uint4 x0 = xh[((m * 2 + blk) * 2 + 0) * np + p];
          const uint4 x1 = xh[((m * 2 + blk) * 2 + 1) * np + p];
          const __half2 *xa = reinterpret_cast<const __half2 *>(&x0);
          const __half2 *xb = reinterpret_cast<const __half2 *>(&x1);
          __half2 s2 = __float2half2_rn(0.0f);
#pragma unroll
          for (int i = 0; i < 4; ++i) s2 = __hfma2(wv[i], xa[i], s2);
#pragma unroll
          for (int i = 0; i < 4; ++i) s2 = __hfma2(wv[4 + i], xb[i], s2);
          const float blocksum = __low2float(s2) + __high2float(s2);
          acc[m] = fmaf(blocksum, xs[(m * 2 + blk) * np + p] * sw, acc[m]);
        }
      }
    }
  }
}

// Expand one 16-block (codes lo/hi, E4M3 scale byte s) of activation row m,
// block j, into the shared layout above.
GDN_DEV void store_act_block(uint4 *xh, float *xs, int npiece, int m, int j, uint32_t lo, uint32_t hi, uint32_t s) {
  const int p = j >> 1, blk = j & 1;
  __half2 h[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = e2m1x2_to_h2(lo >> (8 * i));
    h[4 + i] = e2m1x2_to_h2(hi >> (8 * i));
  }
  const uint4 *hv = reinterpret_cast<const uint4 *>(h);
  xh[((m * 2 + blk) * 2 + 0) * npiece + p] = hv[0];
  xh[((m * 2 + blk) * 2 + 1) * npiece + p] = hv[1];
  xs[(m * 2 + blk) * npiece + p] = e4m3_to_f32(s);
}

// Shared-memory bytes of MB activation rows of length K in that layout.
__host__ __device__ constexpr size_t act_smem_bytes(int MB, int K) {
  return (size_t)MB * (K >> 5) * (4 * 16 + 2 * 4);
}

}  // namespace gdn
