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

constexpr int kMmaWarps = 8;  // GPC row groups x KS K slices per CTA

// GPC 16-row groups per CTA, each split over KS warps by K slice (GPC * KS =
// 8). BULK: the activation rows come into shared memory with one bulk copy
// instead of per-thread loads (fewer requests on the L2 lines every CTA reads).
template <int GPC, int KS, bool BULK>
__global__ void __launch_bounds__(kMmaWarps * 32) gemv_mma_kernel(GemvArgs a) {
  static_assert(GPC * KS == kMmaWarps, "eight warps");
  extern __shared__ __align__(128) unsigned char smem[];
  if (a.early_trigger) pdl_launch_dependents();
  const int K = a.K, nkb4 = K >> 6, qkb4 = nkb4 / KS;   // 64-K steps: all, per K slice
  const int M = a.M;                                    // activation rows = MMA columns, 1..8
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rgl = warp / KS, q = warp % KS;             // row group in CTA, K slice
  const int rg = blockIdx.x * GPC + rgl;
  const int ngroups = (a.N + 15) >> 4;
  const size_t group_bytes = (size_t)nkb4 * 576;
  const uint32_t cbytes = (uint32_t)qkb4 * 512, sbytes = (uint32_t)qkb4 * 64;
  // smem: [barriers 8 x 8 + 1][per warp: codes cbytes | scales sbytes][x_hat M x K halves]
  //       [partials GPC x KS x 16 x M floats][staged activation rows (BULK)]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
  unsigned char *mine = smem + 128 + (size_t)warp * (cbytes + sbytes);
  __half *xh = reinterpret_cast<__half *>(smem + 128 + (size_t)kMmaWarps * (cbytes + sbytes));
  float *part = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(xh) + (size_t)M * K * 2);
  unsigned char *stage = reinterpret_cast<unsigned char *>(part) + (size_t)GPC * KS * 16 * M * 4;
  const bool have = rg < ngroups;

  if (lane == 0 && have) {  // this warp's K slice of its row group: codes, then scales
    mbar_init(bars + warp, 1);
    if (BULK && warp == 0) mbar_init(bars + 8, 1);
    fence_barrier_init();
    const unsigned char *g = a.w_mma + (size_t)rg * group_bytes;
    mbar_arrive_expect_tx(bars + warp, cbytes + sbytes);
    bulk_g2s(mine, g + (size_t)q * cbytes, cbytes, bars + warp);
    bulk_g2s(mine + cbytes, g + (size_t)nkb4 * 512 + (size_t)q * sbytes, sbytes, bars + warp);
  } else if (BULK && threadIdx.x == 0) {
    mbar_init(bars + 8, 1);
    fence_barrier_init();
  }
  __syncwarp();

  pdl_wait();  // the activation rows come from the preceding kernel

  // ---- prologue: x_hat = e2m1(code) * e4m3(scale) in FP16, block by block
  {
    const int nblk = K >> 4;
    const float inv6ts = inv6ts_of(a.ts_a);
    const uint16_t *xb = a.a_bf16;
    const uint8_t *xc = a.a_codes, *xs = a.a_scales;
    bool staged = false;
    if (BULK) {
      __syncthreads();  // barrier 8 initialised
      const uint32_t nb = a.a_bf16 ? (uint32_t)M * K * 2 : (uint32_t)M * (K / 2 + K / 16);
      if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bars + 8, nb);
        if (a.a_bf16) {
          bulk_g2s(stage, a.a_bf16, (uint32_t)M * K * 2, bars + 8);
        } else {
          bulk_g2s(stage, a.a_codes, (uint32_t)M * K / 2, bars + 8);
          bulk_g2s(stage + (size_t)M * K / 2, a.a_scales, (uint32_t)M * K / 16, bars + 8);
        }
      }
      staged = mbar_wait(bars + 8, 0);
      if (staged) {
        if (a.a_bf16) {
          xb = reinterpret_cast<const uint16_t *>(stage);
        } else {
          xc = stage;
          xs = stage + (size_t)M * K / 2;
        }
      }
    }
    for (int jm = threadIdx.x; jm < M * nblk; jm += blockDim.x) {
      const int m = jm / nblk, j = jm - m * nblk;
      bool live = true;
      if (a.row_slot) {
        const int slot = a.row_slot[m];
        live = slot >= 0 && slot < a.num_slots;
      }
      uint32_t lo = 0, hi = 0, s = 0;
      if (live) {
        if (xb) {
          float v[16];
          load_bf16x16(xb + (size_t)m * K + (size_t)j * 16, v);
          if (!quant_block16(v, a.ts_a, inv6ts, lo, hi, s) && blockIdx.x == 0)
            flag_status(a.status, GDN_E_NONFINITE);
        } else {
          const uint2 c = *reinterpret_cast<const uint2 *>(xc + (size_t)m * (K >> 1) + (size_t)j * 8);
          lo = c.x;
          hi = c.y;
          s = xs[(size_t)m * nblk + j];
        }
      }
      store_xhat_block(xh + (size_t)m * K + (size_t)j * 16, lo, hi, s);
    }
  }
  __syncthreads();
  if (!a.early_trigger) pdl_launch_dependents();

  // ---- the slice's block dot products: rows g, g+8 of the group x columns 2t, 2t+1
  const int g = lane >> 2, t = lane & 3;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  bool ok = true;
  if (have) {
    if (!mbar_wait(bars + warp, 0)) {
      ok = false;
    } else {
      const uint4 *codes = reinterpret_cast<const uint4 *>(mine);
      const uint32_t *scl = reinterpret_cast<const uint32_t *>(mine + cbytes);
      const __half *xrow = xh + (size_t)(g < M ? g : 0) * K + 4 * t;  // column g = activation row g
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
          if (g < M) {  // columns M..7 are zero
            const uint2 xv = *reinterpret_cast<const uint2 *>(xrow + (size_t)(kb0 + j) * 16);
            b0 = xv.x;
            b1 = xv.y;
          }
          float d[4];
          mma16816(d, af, b0, b1);
          acc[0] = fmaf(d[0], swg[j], acc[0]);
          acc[1] = fmaf(d[1], swg[j], acc[1]);
          acc[2] = fmaf(d[2], swg8[j], acc[2]);
          acc[3] = fmaf(d[3], swg8[j], acc[3]);
        }
      }
    }
  }
  {
    float *pq = part + (size_t)(rgl * KS + q) * 16 * M;  // [16 rows][M columns]
    const int c0 = 2 * t, c1 = 2 * t + 1;
    if (c0 < M) {
      pq[g * M + c0] = acc[0];
      pq[(g + 8) * M + c0] = acc[2];
    }
    if (c1 < M) {
      pq[g * M + c1] = acc[1];
      pq[(g + 8) * M + c1] = acc[3];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < GPC * 16 * M; i += blockDim.x) {  // K slices added in order
    const int m = i % M, rr = i / M, gl = rr >> 4, r = rr & 15;
    const int n = (blockIdx.x * GPC + gl) * 16 + r;
    if (n < a.N) {
      const float *p0 = part + (size_t)(gl * KS) * 16 * M + r * M + m;
      const size_t qs = (size_t)16 * M;
      float sum = p0[0];
#pragma unroll
      for (int k = 1; k < KS; ++k) sum += p0[k * qs];
      const float y = sum * (a.ts_a * (n < a.n_split ? a.ts_w0 : a.ts_w1));
      if (a.c_is_bf16)
        static_cast<uint16_t *>(a.c)[(size_t)m * a.ldc + n] = f32_to_bf16_bits(y);
      else
        static_cast<float *>(a.c)[(size_t)m * a.ldc + n] = y;
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

bool gemv_mma_ok(const GemvArgs &a) { return a.w_mma && a.M >= 1 && a.M <= 8 && a.K % 256 == 0 && a.K <= 8192; }

namespace {
template <int GPC, int KS, bool BULK>
cudaError_t launch_gemv_mma_t(const GemvArgs &a, const LaunchCtx &lc) {
  const int ngroups = (a.N + 15) / 16;
  const size_t per_warp = (size_t)(a.K / 64 / KS) * 576;
  const size_t stage = BULK ? (a.a_bf16 ? (size_t)a.M * a.K * 2 : (size_t)a.M * (a.K / 2 + a.K / 16)) : 0;
  const size_t smem = 128 + kMmaWarps * per_warp + (size_t)a.M * a.K * 2 + (size_t)GPC * KS * 16 * 4 * a.M + stage;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<GPC, KS, BULK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         200 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((ngroups + GPC - 1) / GPC, 1, 1);
  cfg.blockDim = dim3(kMmaWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<GPC, KS, BULK>, a);
}

template <bool BULK>
cudaError_t launch_gemv_mma_b(const GemvArgs &a, const LaunchCtx &lc) {
  switch (a.mma_tile) {
    case 2:
      if (a.K % 512 == 0) return launch_gemv_mma_t<1, 8, BULK>(a, lc);
      return launch_gemv_mma_t<2, 4, BULK>(a, lc);
    case 3: return launch_gemv_mma_t<4, 2, BULK>(a, lc);
    default: return launch_gemv_mma_t<2, 4, BULK>(a, lc);
  }
}
}  // namespace

cudaError_t launch_gemv_mma(const GemvArgs &a, const LaunchCtx &lc) {
  return a.mma_bulk ? launch_gemv_mma_b<true>(a, lc) : launch_gemv_mma_b<false>(a, lc);
}

}  // namespace gdn
