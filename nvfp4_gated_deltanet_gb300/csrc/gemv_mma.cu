// One activation row against an NVFP4 weight matrix with warp-level MMA
// (mma.sync m16n8k16, FP16 inputs, FP32 accumulation) doing the 16-element
// block dot products: one MMA covers 16 weight rows x one 16-block, so a
// block costs a warp 4 conversions, one MMA and 2 FMAs instead of a 16-lane
// FP16x2 chain per row. The decode step's one-row projections were
// instruction-bound on the CUDA-core chain (ncu: ~58 warp instructions per
// 16-element block-row); this keeps them bound by the weight stream.
//
// Exactness: weights E2M1 -> FP16 exact; activations enter as x_hat =
// e2m1(code) * e4m3(scale) in FP16, exact (|x_hat| <= 6*448, >= 2^-10); the 16
// products of a block are multiples of one quantum (scale/4) below 2^24 of
// them, so the MMA's FP32 block sum is exact. Each block sum is then scaled by
// the weight block scale in one FMA into an FP32 accumulator, blocks in order;
// the four K quarters are added in order. Deterministic, independent of grid.
//
// Weights come repacked at create time (launch_mma_tiles): for every group of
// 16 rows and every 64 K (4 blocks), the 512 code bytes are stored in lane
// order -- lane (g = l/4, t = l%4) gets, for each of the 4 blocks, bytes 2t and
// 2t+1 of rows g and g+8 -- followed, after the group's codes, by its scales
// [64 K step][16 rows][4 blocks]. MMA k position 2t,2t+1 holds block elements
// 4t,4t+1 and 2t+8,2t+9 holds 4t+2,4t+3; x_hat is read in the same order.
#include "common.cuh"

namespace gdn {

namespace {

constexpr int kMmaWarps = 8;  // 2 row groups x 4 K quarters per CTA

GDN_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// Four E4M3 bytes -> four floats (exact).
GDN_DEV void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
  uint32_t lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
  f[0] = __half2float(__ushort_as_half(uint16_t(lo & 0xFFFFu)));
  f[1] = __half2float(__ushort_as_half(uint16_t(lo >> 16)));
  f[2] = __half2float(__ushort_as_half(uint16_t(hi & 0xFFFFu)));
  f[3] = __half2float(__ushort_as_half(uint16_t(hi >> 16)));
}

__global__ void __launch_bounds__(kMmaWarps * 32) gemv_mma_kernel(GemvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (a.early_trigger) pdl_launch_dependents();
  const int K = a.K, nkb4 = K >> 6, qkb4 = nkb4 >> 2;  // 64-K steps: all, per quarter
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rgl = warp >> 2, q = warp & 3;                // row group in CTA, K quarter
  const int rg = blockIdx.x * 2 + rgl;
  const int ngroups = (a.N + 15) >> 4;
  const size_t group_bytes = (size_t)nkb4 * 576;
  const uint32_t cbytes = (uint32_t)qkb4 * 512, sbytes = (uint32_t)qkb4 * 64;
  // smem: [barriers 8 x 8][per warp: codes cbytes | scales sbytes][x_hat K halves][partials 2 x 4 x 16 floats]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
  unsigned char *mine = smem + 64 + (size_t)warp * (cbytes + sbytes);
  __half *xh = reinterpret_cast<__half *>(smem + 64 + (size_t)kMmaWarps * (cbytes + sbytes));
  float *part = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(xh) + (size_t)K * 2);
  const bool have = rg < ngroups;

  if (lane == 0 && have) {  // this warp's quarter of its row group: codes, then scales
    mbar_init(bars + warp, 1);
    fence_barrier_init();
    const unsigned char *g = a.w_mma + (size_t)rg * group_bytes;
    mbar_arrive_expect_tx(bars + warp, cbytes + sbytes);
    bulk_g2s(mine, g + (size_t)q * cbytes, cbytes, bars + warp);
    bulk_g2s(mine + cbytes, g + (size_t)nkb4 * 512 + (size_t)q * sbytes, sbytes, bars + warp);
  }
  __syncwarp();

  pdl_wait();  // the activation row comes from the preceding kernel

  // ---- prologue: x_hat = e2m1(code) * e4m3(scale) in FP16, block by block
  {
    const int nblk = K >> 4;
    const float inv6ts = inv6ts_of(a.ts_a);
    bool live = a.M > 0;
    if (live && a.row_slot) {
      const int slot = a.row_slot[0];
      live = slot >= 0 && slot < a.num_slots;
    }
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
      uint32_t lo = 0, hi = 0, s = 0;
      if (live) {
        if (a.a_bf16) {
          const uint4 *p = reinterpret_cast<const uint4 *>(a.a_bf16 + (size_t)j * 16);
          float v[16];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint4 w4 = p[i];
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              v[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
              v[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            }
          }
          if (!quant_block16(v, a.ts_a, inv6ts, lo, hi, s) && blockIdx.x == 0)
            flag_status(a.status, GDN_E_NONFINITE);
        } else {
          const uint2 c = *reinterpret_cast<const uint2 *>(a.a_codes + (size_t)j * 8);
          lo = c.x;
          hi = c.y;
          s = a.a_scales[j];
        }
      }
      __half2 h[8];
      e2m1x8_to_h2x4(lo, *reinterpret_cast<__half2(*)[4]>(&h[0]));
      e2m1x8_to_h2x4(hi, *reinterpret_cast<__half2(*)[4]>(&h[4]));
      const __half2 sc = __float2half2_rn(e4m3_to_f32(s));  // exact: an E4M3 value
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = __hmul2(h[i], sc);  // exact: see above
      uint4 *dst = reinterpret_cast<uint4 *>(xh + (size_t)j * 16);
      dst[0] = *reinterpret_cast<const uint4 *>(&h[0]);
      dst[1] = *reinterpret_cast<const uint4 *>(&h[4]);
    }
  }
  __syncthreads();
  if (!a.early_trigger) pdl_launch_dependents();

  // ---- the quarter's block dot products
  const int g = lane >> 2, t = lane & 3;
  float acc0 = 0.0f, acc1 = 0.0f;  // rows g and g+8 (column 0 lives in lanes t == 0)
  bool ok = true;
  if (have) {
    if (!mbar_wait(bars + warp, 0)) {
      ok = false;
    } else {
      const uint4 *codes = reinterpret_cast<const uint4 *>(mine);
      const uint32_t *scl = reinterpret_cast<const uint32_t *>(mine + cbytes);
      for (int s = 0; s < qkb4; ++s) {
        const uint4 c4 = codes[s * 32 + lane];
        float swg[4], swg8[4];
        e4m3x4_to_f32(scl[s * 16 + g], swg);
        e4m3x4_to_f32(scl[s * 16 + g + 8], swg8);
        const int kb0 = (q * qkb4 + s) * 4;  // first block of this 64-K step
        const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __half2 hv[4];  // bytes: (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
          e2m1x8_to_h2x4(cw[j], hv);
          const uint32_t af[4] = {*reinterpret_cast<uint32_t *>(&hv[0]), *reinterpret_cast<uint32_t *>(&hv[2]),
                                  *reinterpret_cast<uint32_t *>(&hv[1]), *reinterpret_cast<uint32_t *>(&hv[3])};
          uint32_t b0 = 0, b1 = 0;
          if (g == 0) {  // column 0 = the activation row; columns 1..7 are zero
            const uint2 xv = *reinterpret_cast<const uint2 *>(xh + (size_t)(kb0 + j) * 16 + 4 * t);
            b0 = xv.x;
            b1 = xv.y;
          }
          float d[4];
          mma16816(d, af, b0, b1);
          acc0 = fmaf(d[0], swg[j], acc0);
          acc1 = fmaf(d[2], swg8[j], acc1);
        }
      }
    }
  }
  if (t == 0) {
    part[(rgl * 4 + q) * 16 + g] = acc0;
    part[(rgl * 4 + q) * 16 + g + 8] = acc1;
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // 2 groups x 16 rows: quarters added in order
    const int gl = threadIdx.x >> 4, r = threadIdx.x & 15;
    const int n = (blockIdx.x * 2 + gl) * 16 + r;
    if (n < a.N) {
      const float sum = ((part[(gl * 4 + 0) * 16 + r] + part[(gl * 4 + 1) * 16 + r]) + part[(gl * 4 + 2) * 16 + r]) +
                        part[(gl * 4 + 3) * 16 + r];
      const float y = sum * (a.ts_a * (n < a.n_split ? a.ts_w0 : a.ts_w1));
      if (a.c_is_bf16)
        static_cast<uint16_t *>(a.c)[n] = f32_to_bf16_bits(y);
      else
        static_cast<float *>(a.c)[n] = y;
    }
  }
  if (!ok && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
}

__global__ void mma_tiles_kernel(const uint8_t *codes, const uint8_t *scales, int rows, int K, uint8_t *dst) {
  const int nkb4 = K / 64;
  const size_t group_bytes = (size_t)nkb4 * 576;
  const size_t total = (size_t)((rows + 15) / 16) * group_bytes;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t rg = i / group_bytes;
    const size_t off = i % group_bytes;
    uint8_t v = 0;
    if (off < (size_t)nkb4 * 512) {  // codes: [kb4][lane][block j][4 bytes]
      const int kb4 = (int)(off / 512), within = (int)(off % 512);
      const int lane = within / 16, j = (within % 16) / 4, e = within % 4;
      const int g = lane / 4, t = lane % 4;
      const int r = (e < 2 ? g : g + 8), byte = 2 * t + (e & 1);
      const size_t row = rg * 16 + r;
      const int blk = kb4 * 4 + j;
      if (row < (size_t)rows) v = codes[row * (K / 2) + (size_t)blk * 8 + byte];
    } else {  // scales: [kb4][row][block j]
      const size_t so = off - (size_t)nkb4 * 512;
      const int kb4 = (int)(so / 64), r = (int)(so % 64) / 4, j = (int)(so % 4);
      const size_t row = rg * 16 + r;
      if (row < (size_t)rows) v = scales[row * (K / 16) + (size_t)kb4 * 4 + j];
    }
    dst[i] = v;
  }
}

}  // namespace

size_t mma_tiles_bytes(int rows, int K) { return (size_t)((rows + 15) / 16) * (K / 64) * 576; }

cudaError_t launch_mma_tiles(const uint8_t *codes, const uint8_t *scales, int rows, int K, uint8_t *dst,
                             cudaStream_t stream) {
  if (K % 256) return cudaErrorInvalidValue;
  mma_tiles_kernel<<<304, 256, 0, stream>>>(codes, scales, rows, K, dst);
  return cudaGetLastError();
}

bool gemv_mma_ok(const GemvArgs &a) { return a.w_mma && a.M == 1 && a.K % 256 == 0 && a.K <= 8192; }

cudaError_t launch_gemv_mma(const GemvArgs &a, const LaunchCtx &lc) {
  const int ngroups = (a.N + 15) / 16;
  const size_t per_warp = (size_t)(a.K / 256) * 576;
  const size_t smem = 64 + kMmaWarps * per_warp + (size_t)a.K * 2 + 2 * 4 * 16 * 4;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((ngroups + 1) / 2, 1, 1);
  cfg.blockDim = dim3(kMmaWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_mma_kernel, a);
}

}  // namespace gdn
