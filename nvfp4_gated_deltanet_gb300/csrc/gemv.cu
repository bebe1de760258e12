// Block-scaled W4A4 product for a few activation rows (decode buckets), on the
// CUDA cores: the weights are streamed from HBM once with 128-bit loads and
// every activation row is applied to each weight block while it is in
// registers.
//
// Exactness inside a 16-block: E2M1 values are converted to FP16 (exact), each
// half of an FP16x2 accumulator sums 8 products (|sum| <= 8*36 = 288 on a 1/4
// grid, exact in FP16), so the block's integer-valued dot product is exact;
// times the two E4M3 scales it is still exact in FP32. Only the sum over
// blocks rounds (FP32, fixed order: lane-local chunks, then a fixed warp tree).
#include "common.cuh"

namespace gdn {

namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 2;

// Shared-memory layout of the activations, chosen so a warp's 128-bit loads
// (lane l reads 64-element chunk c = l + 32 j) are contiguous:
//   xh[((m * 4 + blk) * 2 + half) * nchunk + c] : uint4 = 4 half2 (8 values)
//   xs[(m * 4 + blk) * nchunk + c]              : float E4M3 block scale
struct XSmem {
  uint4 *xh;
  float *xs;
};

template <int MB>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(GemvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int K = a.K;
  const int nchunk = K >> 6;
  XSmem sm{reinterpret_cast<uint4 *>(smem),
           reinterpret_cast<float *>(smem + (size_t)MB * 4 * 2 * nchunk * sizeof(uint4))};

  // ---- prologue: the activation rows as FP16 E2M1 values + FP32 block scales
  {
    const int nblk = K >> 4;
    const float inv6ts = inv6ts_of(a.ts_a);
    for (int t = threadIdx.x; t < MB * nblk; t += blockDim.x) {
      const int m = t / nblk, j = t % nblk;
      uint32_t lo = 0, hi = 0, s = 0;
      bool live = m < a.M;
      if (live && a.row_slot) {
        const int slot = a.row_slot[m];
        live = slot >= 0 && slot < a.num_slots;
      }
      if (live) {
        if (a.a_bf16) {
          const uint4 *p = reinterpret_cast<const uint4 *>(a.a_bf16 + (size_t)m * K + j * 16);
          float v[16];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            uint4 q = p[i];
            uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              v[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
              v[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            }
          }
          if (!quant_block16(v, a.ts_a, inv6ts, lo, hi, s) && blockIdx.x == 0)
            flag_status(a.status, GDN_E_NONFINITE);
        } else {
          uint2 c = *reinterpret_cast<const uint2 *>(a.a_codes + (size_t)m * (K >> 1) + j * 8);
          lo = c.x;
          hi = c.y;
          s = a.a_scales[(size_t)m * nblk + j];
        }
      }
      const int c = j >> 2, blk = j & 3;
      __half2 h[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        h[i] = e2m1x2_to_h2(lo >> (8 * i));
        h[4 + i] = e2m1x2_to_h2(hi >> (8 * i));
      }
      const uint4 *hv = reinterpret_cast<const uint4 *>(h);
      sm.xh[((m * 4 + blk) * 2 + 0) * nchunk + c] = hv[0];
      sm.xh[((m * 4 + blk) * 2 + 1) * nchunk + c] = hv[1];
      sm.xs[(m * 4 + blk) * nchunk + c] = e4m3_to_f32(s);
    }
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int tw = gridDim.x * kWarps;
  const size_t ldw = (size_t)(K >> 1), lds = (size_t)(K >> 4);

  for (int n0 = gw * kRowsPerWarp; n0 < a.N; n0 += tw * kRowsPerWarp) {
    float acc[kRowsPerWarp][MB];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[r][m] = 0.0f;

    for (int c = lane; c < nchunk; c += 32) {
      uint4 wc[kRowsPerWarp][2];
      uint32_t ws[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int n = min(n0 + r, a.N - 1);
        const uint4 *pc = reinterpret_cast<const uint4 *>(a.w_codes + n * ldw + (size_t)c * 32);
        wc[r][0] = __ldcs(pc);
        wc[r][1] = __ldcs(pc + 1);
        ws[r] = __ldcs(reinterpret_cast<const unsigned int *>(a.w_scales + n * lds + (size_t)c * 4));
      }
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          const uint32_t w0 = (blk < 2) ? (blk == 0 ? wc[r][0].x : wc[r][0].z) : (blk == 2 ? wc[r][1].x : wc[r][1].z);
          const uint32_t w1 = (blk < 2) ? (blk == 0 ? wc[r][0].y : wc[r][0].w) : (blk == 2 ? wc[r][1].y : wc[r][1].w);
          __half2 wv[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            wv[i] = e2m1x2_to_h2(w0 >> (8 * i));
            wv[4 + i] = e2m1x2_to_h2(w1 >> (8 * i));
          }
          const float sw = e4m3_to_f32(ws[r] >> (8 * blk));
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            if (m < a.M) {
              const uint4 x0 = sm.xh[((m * 4 + blk) * 2 + 0) * nchunk + c];
              const uint4 x1 = sm.xh[((m * 4 + blk) * 2 + 1) * nchunk + c];
              const __half2 *xa = reinterpret_cast<const __half2 *>(&x0);
              const __half2 *xb = reinterpret_cast<const __half2 *>(&x1);
              __half2 s2 = __float2half2_rn(0.0f);
#pragma unroll
              for (int i = 0; i < 4; ++i) s2 = __hfma2(wv[i], xa[i], s2);
#pragma unroll
              for (int i = 0; i < 4; ++i) s2 = __hfma2(wv[4 + i], xb[i], s2);
              const float blocksum = __low2float(s2) + __high2float(s2);
              acc[r][m] = fmaf(blocksum, sm.xs[(m * 4 + blk) * nchunk + c] * sw, acc[r][m]);
            }
          }
        }
      }
    }

    // ---- warp reduction of the kRowsPerWarp * MB partial sums, then store
    constexpr int NV = kRowsPerWarp * MB;
    float v[NV];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < MB; ++m) v[r * MB + m] = acc[r][m];
    const float tot = warp_transpose_reduce<NV>(v, lane);
    const int idx = reduce_index<NV>(lane);
    const int r = idx / MB, m = idx % MB;
    const int n = n0 + r;
    if (lane == reduce_owner<NV>(idx) && m < a.M && n < a.N) {
      const float tsw = n < a.n_split ? a.ts_w0 : a.ts_w1;
      const float y = tot * (a.ts_a * tsw);
      if (a.c_is_bf16)
        static_cast<uint16_t *>(a.c)[(size_t)m * a.ldc + n] = f32_to_bf16_bits(y);
      else
        static_cast<float *>(a.c)[(size_t)m * a.ldc + n] = y;
    }
  }
}

template <int MB>
cudaError_t launch_mb(const GemvArgs &a, const LaunchCtx &lc) {
  const size_t smem = (size_t)MB * (a.K >> 6) * (4 * 2 * sizeof(uint4) + 4 * sizeof(float));
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  int ctas = (a.N + kWarps * kRowsPerWarp - 1) / (kWarps * kRowsPerWarp);
  const int cap = lc.num_sms * 4;
  if (ctas > cap) ctas = cap;
  gemv_kernel<MB><<<ctas, kWarps * 32, smem, lc.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs &a, const LaunchCtx &lc) {
  if (a.M <= 0 || a.N <= 0) return cudaSuccess;
  if (a.M == 1) return launch_mb<1>(a, lc);
  if (a.M == 2) return launch_mb<2>(a, lc);
  if (a.M <= 4) return launch_mb<4>(a, lc);
  if (a.M <= 8) return launch_mb<8>(a, lc);
  if (a.M <= 16) return launch_mb<16>(a, lc);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
