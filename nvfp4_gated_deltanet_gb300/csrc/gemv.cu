// Block-scaled W4A4 product for a few activation rows (decode buckets) on the
// CUDA cores. The weights are read from HBM exactly once: every warp owns a
// contiguous range of weight rows and streams them, two rows per stage, into
// its own shared-memory ring with bulk asynchronous copies (cp.async.bulk,
// completion on an mbarrier). The copies of the first stages are issued before
// anything else -- before the activation prologue and before waiting on the
// preceding kernel (programmatic dependent launch), since weights never depend
// on it -- so the whole matrix is in flight from the first microsecond.
//
// Exactness inside a 16-block: E2M1 values are converted to FP16 (exact), each
// half of an FP16x2 accumulator sums 8 products (|sum| <= 8*36 = 288 on a 1/4
// grid, exact in FP16), so the block's integer-valued dot product is exact;
// times the two E4M3 scales it is still exact in FP32. Only the sum over
// blocks rounds (FP32, fixed order: lane-local pieces, then a fixed warp tree),
// so results do not depend on how rows are spread over warps or on M.
#include "common.cuh"
#include "gemv_core.cuh"

namespace gdn {

namespace {

constexpr int kWarps = 8;
constexpr int kMaxStages = 4;
constexpr int kBarBytes = kWarps * kMaxStages * 8;  // mbarriers, 256 bytes

// TMA = stream weights through the shared ring (K % 256 == 0, so every copy
// is 16-byte aligned and sized); otherwise lanes read them from global memory.
template <int MB, bool TMA, int NP>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(GemvArgs a, int rows_per_warp, int stages) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (a.early_trigger) pdl_launch_dependents();
  const int K = a.K, npiece = K >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t cbytes = (size_t)K >> 1, sbytes = (size_t)K >> 4;  // per weight row
  const int stage_bytes = 2 * (int)(cbytes + sbytes);

  // smem: [barriers kWarps*stages][ring kWarps*stages*stage_bytes][xh][xs]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
  unsigned char *ring = smem + kBarBytes;
  const size_t ring_bytes = TMA ? (size_t)kWarps * stages * stage_bytes : 0;
  uint4 *xh = reinterpret_cast<uint4 *>(ring + ring_bytes);
  float *xs = reinterpret_cast<float *>(ring + ring_bytes + (size_t)MB * 4 * npiece * sizeof(uint4));

  const int gw = blockIdx.x * kWarps + warp;
  const int r_begin = min(gw * rows_per_warp, a.N);
  const int r_end = min(r_begin + rows_per_warp, a.N);
  const int npairs = (r_end - r_begin + 1) >> 1;
  uint64_t *mybar = bars + warp * stages;
  unsigned char *myring = ring + (size_t)warp * stages * stage_bytes;

  auto issue = [&](int pair) {
    const int n0 = r_begin + 2 * pair;
    const int nr = min(2, r_end - n0);
    const int st = pair % stages;
    unsigned char *dst = myring + (size_t)st * stage_bytes;
    const uint32_t cb = (uint32_t)(nr * cbytes), sb = (uint32_t)(nr * sbytes);
    mbar_arrive_expect_tx(mybar + st, cb + sb);
    bulk_g2s(dst, a.w_codes + (size_t)n0 * cbytes, cb, mybar + st);
    bulk_g2s(dst + 2 * cbytes, a.w_scales + (size_t)n0 * sbytes, sb, mybar + st);
  };
  if (TMA && lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(mybar + s, 1);
    fence_barrier_init();
    for (int s = 0; s < min(stages, npairs); ++s) issue(s);
  }
  __syncwarp();

  // the activations come from the preceding kernel
  pdl_wait();

  // ---- prologue: activation rows as FP16 E2M1 values + FP32 block scales
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
  }
  __syncthreads();
  if (!a.early_trigger) pdl_launch_dependents();

  constexpr int NV = 2 * MB;
  bool ok = true;
  for (int pair = 0; pair < npairs; ++pair) {
    const int n0 = r_begin + 2 * pair;
    const int nr = min(2, r_end - n0);
    const int st = pair % stages;
    const unsigned char *codes0, *scales0;
    if (TMA) {
      if (!mbar_wait(mybar + st, (uint32_t)((pair / stages) & 1))) {
        // give up on this warp's rows; let its copies still in flight land
        // (each wait bounded) before the CTA's shared memory goes away
        ok = false;
        for (int q = pair + 1; q < min(pair + stages, npairs); ++q)
          (void)mbar_wait(mybar + q % stages, (uint32_t)((q / stages) & 1));
        break;
      }
      codes0 = myring + (size_t)st * stage_bytes;
      scales0 = codes0 + 2 * cbytes;
    } else {
      codes0 = a.w_codes + (size_t)n0 * cbytes;
      scales0 = a.w_scales + (size_t)n0 * sbytes;
    }
    float v[NV];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float acc[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) acc[m] = 0.0f;
      if (r < nr) dot_row<MB, NP>(codes0 + r * cbytes, scales0 + r * sbytes, npiece, a.M, xh, xs, lane, acc);
#pragma unroll
      for (int m = 0; m < MB; ++m) v[r * MB + m] = acc[m];
    }
    if (TMA) {
      __syncwarp();  // every lane is done with this stage before it is refilled
      if (lane == 0 && pair + stages < npairs) issue(pair + stages);
    }
    const float tot = warp_transpose_reduce<NV>(v, lane);
    const int idx = reduce_index<NV>(lane);
    const int r = idx / MB, m = idx % MB;
    const int n = n0 + r;
    if (lane == reduce_owner<NV>(idx) && m < a.M && r < nr) {
      const float tsw = n < a.n_split ? a.ts_w0 : a.ts_w1;
      const float y = tot * (a.ts_a * tsw);
      if (a.c_is_bf16)
        static_cast<uint16_t *>(a.c)[(size_t)m * a.ldc + n] = f32_to_bf16_bits(y);
      else
        static_cast<float *>(a.c)[(size_t)m * a.ldc + n] = y;
    }
  }
  if (TMA && !ok) {
    if (lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
  }
}

template <int MB, bool TMA, int NP>
cudaError_t launch_cfg(const GemvArgs &a, const LaunchCtx &lc) {
  const int npiece = a.K >> 5;
  const size_t act = (size_t)MB * npiece * (4 * sizeof(uint4) + 2 * sizeof(float));
  const size_t stage_bytes = 2 * ((size_t)a.K / 2 + a.K / 16);
  const size_t budget = 200 * 1024;
  // rows per warp: spread the rows over every warp that fits (2 CTAs per SM
  // when shared memory allows), in whole row pairs; the ring has at most as
  // many stages as a warp has row pairs
  int stages = TMA ? kMaxStages : 1, rpw = 2;
  size_t smem = 0;
  for (int pass = 0; pass < 2; ++pass) {
    if (TMA)
      while (stages > 1 && kBarBytes + act + kWarps * stages * stage_bytes > budget) --stages;
    smem = kBarBytes + (TMA ? kWarps * stages * stage_bytes : 0) + act;
    const int ctas_per_sm = smem * 2 <= 220 * 1024 ? 2 : 1;
    const int warps_total = lc.num_sms * ctas_per_sm * kWarps;
    rpw = (a.N + warps_total - 1) / warps_total;
    rpw = (rpw + 1) & ~1;
    if (rpw < 2) rpw = 2;
    if (TMA && stages > rpw / 2) stages = rpw / 2;
  }
  smem = kBarBytes + (TMA ? kWarps * stages * stage_bytes : 0) + act;
  if (smem > budget) return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<MB, TMA, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int ctas = (a.N + kWarps * rpw - 1) / (kWarps * rpw);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<MB, TMA, NP>, a, rpw, stages);
}

template <int MB>
cudaError_t launch_mb(const GemvArgs &a, const LaunchCtx &lc) {
  // the layer's two reduction lengths get fully unrolled dot products
  if (a.K == 2048) return launch_cfg<MB, true, 64>(a, lc);
  if (a.K == 4096) return launch_cfg<MB, true, 128>(a, lc);
  if (a.K % 256 == 0) return launch_cfg<MB, true, 0>(a, lc);
  return launch_cfg<MB, false, 0>(a, lc);
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs &a, const LaunchCtx &lc) {
  if (a.M <= 0 || a.N <= 0) return cudaSuccess;
  if (gemv_mma_ok(a)) return launch_gemv_mma(a, lc);
  if (a.M == 1) return launch_mb<1>(a, lc);
  if (a.M == 2) return launch_mb<2>(a, lc);
  if (a.M <= 4) return launch_mb<4>(a, lc);
  if (a.M <= 8) return launch_mb<8>(a, lc);
  if (a.M <= 16) return launch_mb<16>(a, lc);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
