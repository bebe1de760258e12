// Token mixing of a large decode batch in three kernels, so the state stream
// gets a kernel of its own:
//   batch_prep_kernel   conv + SiLU of a whole row, q/k L2 norms, beta and the
//                       log-decay per value head; the row's conv state is
//                       shifted in place
//   batch_delta_kernel  the gated delta rule: per (row, value head, d_v slice)
//                       the state rows in registers, nothing else -- the part
//                       that moves 4 MB per row
//   batch_gnorm_kernel  z-gated RMSNorm + NVFP4 quantisation of y
// Every operation and its order is the fused mixing kernel's (mix.cu), so the
// results are bit-identical to it; only the split differs. Rows whose slot id
// is -1, out of range or repeated are padding: zero y, no state touched.
#include "common.cuh"

namespace gdn {

namespace {

// The row's slot, and whether the row is live; a repeated slot refuses both
// rows (every warp checks, B/32 loads per lane).
GDN_DEV bool row_live(const MixArgs &a, int b, int lane, int &slot, bool &bad) {
  slot = a.slot_ids[b];
  bool live = slot >= 0 && slot < a.num_slots;
  bad = slot < -1 || slot >= a.num_slots;
  if (live) {
    bool dup = false;
    for (int j = lane; j < a.B; j += 32) dup |= (j != b && a.slot_ids[j] == slot);
    if (__any_sync(0xffffffffu, dup)) { bad = true; live = false; }
  }
  return live;
}

// One CTA per row (1024 threads, channel c handled by thread c % 1024): the
// conv over every channel into shared memory, one warp per q/k head for its
// L2 norm (lane-local sums then the butterfly, as in the fused kernel), the
// gates by the first Hv threads. Shared memory: C floats of conv output.
constexpr int kPrepThreads = 1024;

template <int D>
__global__ void __launch_bounds__(kPrepThreads) batch_prep_kernel(MixArgs a, BatchWs w) {
  constexpr int EPL = D / 32;
  extern __shared__ float s_y[];   // [C] conv outputs, then 2*Hk norm factors
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Kc = a.Kc, C = a.C, nqk = 2 * a.Hk;
  float *s_r = s_y + C;
  int slot;
  bool bad;
  const bool live = row_live(a, b, lane, slot, bad);
  uint16_t *cst = a.conv_state + (size_t)(live ? slot : 0) * (Kc - 1) * C;
  pdl_wait();  // the projections come from the preceding kernel
  pdl_launch_dependents();
  if (bad && tid == 0) flag_status(a.status, GDN_E_RANGE);
  if (!live) return;
  const uint16_t *xin = a.qkvz + (size_t)b * a.ld_qkvz;
  for (int c = tid; c < C; c += kPrepThreads) {
    uint16_t tap[3] = {0, 0, 0};
#pragma unroll
    for (int j = 0; j < 3; ++j)
      if (j < Kc - 1) tap[j] = cst[(size_t)j * C + c];
    const uint16_t xn = xin[c];
    float pre = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < Kc) {
        const uint16_t bits = j < Kc - 1 ? tap[j < 3 ? j : 2] : xn;
        pre = fmaf(bf16_bits_to_f32(a.conv_w[(size_t)c * Kc + j]), bf16_bits_to_f32(bits), pre);
      }
    }
    s_y[c] = siluf_(pre);
    // the channel's conv state: taps shift by one, newest raw input last
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (j < Kc - 2) cst[(size_t)j * C + c] = tap[j + 1];
    cst[(size_t)(Kc - 2) * C + c] = xn;
  }
  if (tid < a.Hv) {  // gates
    const uint16_t *bain = a.ba + (size_t)b * a.ld_ba;
    const float b_raw = bf16_bits_to_f32(bain[tid]);
    const float a_raw = bf16_bits_to_f32(bain[a.Hv + tid]);
    w.beta[(size_t)b * a.Hv + tid] = sigmoidf_(b_raw);
    w.gl[(size_t)b * a.Hv + tid] = -expf(a.A_log[tid]) * softplusf_(a_raw + a.dt_bias[tid]);
  }
  __syncthreads();
  for (int hq = warp; hq < nqk; hq += kPrepThreads / 32) {  // q heads, then k heads
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) ss = fmaf(s_y[hq * D + lane * EPL + e], s_y[hq * D + lane * EPL + e], ss);
    ss = warp_sum(ss);
    if (lane == 0)
      s_r[hq] = hq < a.Hk ? (1.0f / sqrtf(ss + a.l2_eps)) * (1.0f / sqrtf((float)D)) : 1.0f / sqrtf(ss + a.l2_eps);
  }
  __syncthreads();
  const int nqkc = nqk * D;
  for (int c = tid; c < C; c += kPrepThreads) {
    const float y = s_y[c];
    if (c < a.Hk * D)
      w.qn[(size_t)b * a.Hk * D + c] = y * s_r[c / D];
    else if (c < nqkc)
      w.kn[(size_t)b * a.Hk * D + (c - a.Hk * D)] = y * s_r[c / D];
    else
      w.v[(size_t)b * a.Hv * D + (c - nqkc)] = y;
  }
}

template <int NS>
__host__ __device__ constexpr int bd_rows_per_warp() { return NS == 1 ? 16 : 8; }

template <int D, int NS, bool SB>
__global__ void __launch_bounds__((D / NS / bd_rows_per_warp<NS>()) * 32, NS == 1 ? 2 : 0)
    batch_delta_kernel(MixArgs a, BatchWs w) {
  constexpr int R = D / NS;
  constexpr int kRPW = bd_rows_per_warp<NS>();
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.x / NS, row0 = (blockIdx.x % NS) * R;
  const int b = blockIdx.y;
  const int kh = h / (a.Hv / a.Hk);
  int slot;
  bool bad;
  const bool live = row_live(a, b, lane, slot, bad);
  const int lr0 = warp * kRPW;
  constexpr size_t kEs = SB ? 2 : 4;
  char *sp = static_cast<char *>(a.ssm_state) +
             ((((size_t)(live ? slot : 0) * a.Hv + h) * D + row0 + lr0) * D + lane * EPL) * kEs;
  float st[kRPW][EPL];
  if (live) {
#pragma unroll
    for (int j = 0; j < kRPW; ++j) {
      const char *p = sp + (size_t)j * D * kEs;
      if (SB) {
        uint16_t bb[EPL];
        if (EPL == 4) {
          const uint2 t = *reinterpret_cast<const uint2 *>(p);
          bb[0] = t.x & 0xFFFFu; bb[1 % EPL] = t.x >> 16; bb[2 % EPL] = t.y & 0xFFFFu; bb[3 % EPL] = t.y >> 16;
        } else if (EPL == 2) {
          const uint32_t t = *reinterpret_cast<const uint32_t *>(p);
          bb[0] = t & 0xFFFFu; bb[1 % EPL] = t >> 16;
        } else {
          bb[0] = *reinterpret_cast<const uint16_t *>(p);
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[j][e] = bf16_bits_to_f32(bb[e]);
      } else if (EPL == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        st[j][0] = t.x; st[j][1 % EPL] = t.y; st[j][2 % EPL] = t.z; st[j][3 % EPL] = t.w;
      } else if (EPL == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        st[j][0] = t.x; st[j][1 % EPL] = t.y;
      } else {
        st[j][0] = *reinterpret_cast<const float *>(p);
      }
    }
  }
  pdl_wait();  // q, k, v, beta, g come from the preceding kernel
  pdl_launch_dependents();
  if (!live) return;
  float kr[EPL], qr[EPL];
  float kq = 0.0f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    kr[e] = w.kn[((size_t)b * a.Hk + kh) * D + lane * EPL + e];
    qr[e] = w.qn[((size_t)b * a.Hk + kh) * D + lane * EPL + e];
    kq = fmaf(kr[e], qr[e], kq);
  }
  kq = warp_sum(kq);
  const float beta = w.beta[(size_t)b * a.Hv + h];
  const float alpha = expf(w.gl[(size_t)b * a.Hv + h]);
  const float *vrow = w.v + ((size_t)b * a.Hv + h) * D + row0 + lr0;
  float vals[2 * kRPW];
#pragma unroll
  for (int j = 0; j < kRPW; ++j) {
    float dk = 0.0f, dq = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      dk = fmaf(st[j][e], kr[e], dk);
      dq = fmaf(st[j][e], qr[e], dq);
    }
    vals[j] = dk;
    vals[kRPW + j] = dq;
  }
  const float tot = warp_transpose_reduce<2 * kRPW>(vals, lane);
  float *orow = w.o + ((size_t)b * a.Hv + h) * D + row0 + lr0;
#pragma unroll
  for (int j = 0; j < kRPW; ++j) {
    const float Sk = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * kRPW>(j));
    const float Sq = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * kRPW>(kRPW + j));
    const float u = beta * (vrow[j] - alpha * Sk);
    const float o = fmaf(u, kq, alpha * Sq);
#pragma unroll
    for (int e = 0; e < EPL; ++e) st[j][e] = fmaf(u, kr[e], alpha * st[j][e]);
    if (lane == 0) orow[j] = o;
  }
#pragma unroll
  for (int j = 0; j < kRPW; ++j) {
    char *p = sp + (size_t)j * D * kEs;
    if (SB) {
      uint32_t bb[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) bb[e] = f32_to_bf16_bits(st[j][e]);
      if (EPL == 4)
        *reinterpret_cast<uint2 *>(p) = make_uint2(bb[0] | (bb[1 % EPL] << 16), bb[2 % EPL] | (bb[3 % EPL] << 16));
      else if (EPL == 2)
        *reinterpret_cast<uint32_t *>(p) = bb[0] | (bb[1 % EPL] << 16);
      else
        *reinterpret_cast<uint16_t *>(p) = (uint16_t)bb[0];
    } else if (EPL == 4) {
      *reinterpret_cast<float4 *>(p) = make_float4(st[j][0], st[j][1 % EPL], st[j][2 % EPL], st[j][3 % EPL]);
    } else if (EPL == 2) {
      *reinterpret_cast<float2 *>(p) = make_float2(st[j][0], st[j][1 % EPL]);
    } else {
      *reinterpret_cast<float *>(p) = st[j][0];
    }
  }
}

template <int D>
__global__ void __launch_bounds__(D) batch_gnorm_kernel(MixArgs a, BatchWs w) {
  __shared__ float s_o[D], s_y[D], s_gsum[D / 16];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const int vd = a.Hv * D;
  int slot;
  bool bad;
  const bool live = row_live(a, b, lane, slot, bad);
  const float nw = a.norm_w[tid];
  pdl_wait();  // o comes from the preceding kernel
  pdl_launch_dependents();
  if (!live) {  // padding: zero y blocks of this head
    if ((tid & 1) == 0) a.y_codes[((size_t)b * vd + h * D + tid) >> 1] = 0;
    if ((tid & 15) == 0) {
      const int blk = (h * D + tid) >> 4;
      a.y_scales[a.y_sf_tiled ? sf_tiled_offset(b, blk, vd >> 4) : ((size_t)b * vd >> 4) + blk] = 0;
    }
    return;
  }
  const float zv = bf16_bits_to_f32(a.qkvz[(size_t)b * a.ld_qkvz + 2 * a.Hk * D + vd + h * D + tid]);
  const float o = w.o[((size_t)b * a.Hv + h) * D + tid];
  s_o[tid] = o;
  __syncthreads();
  if (tid < D / 16) {  // 16-row group sums, rows in order
    float p = 0.0f;
    for (int i = 0; i < 16; ++i) p = fmaf(s_o[tid * 16 + i], s_o[tid * 16 + i], p);
    s_gsum[tid] = p;
  }
  __syncthreads();
  float sumsq = 0.0f;
  for (int gi = 0; gi < D / 16; ++gi) sumsq += s_gsum[gi];
  const float rstd = 1.0f / sqrtf(sumsq / (float)D + a.rms_eps);
  s_y[tid] = s_o[tid] * rstd * nw * siluf_(zv);
  __syncthreads();
  if (tid < D / 16) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = s_y[tid * 16 + i];
    uint32_t lo, hi, s;
    if (!quant_block16(v, a.ts_out, inv6ts_of(a.ts_out), lo, hi, s)) flag_status(a.status, GDN_E_NONFINITE);
    const size_t e0 = (size_t)b * vd + h * D + tid * 16;
    *reinterpret_cast<uint2 *>(a.y_codes + (e0 >> 1)) = make_uint2(lo, hi);
    const int blk = (h * D + tid * 16) >> 4;
    a.y_scales[a.y_sf_tiled ? sf_tiled_offset(b, blk, vd >> 4) : (e0 >> 4)] = uint8_t(s);
  }
}

cudaError_t launch_attr(const void *fn, dim3 grid, int threads, const LaunchCtx &lc, void **args,
                        size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

template <int D>
cudaError_t launch_batch_d(const MixArgs &a, const BatchWs &w, const LaunchCtx &lc) {
  MixArgs ac = a;
  BatchWs wc = w;
  void *args[] = {&ac, &wc};
  const size_t prep_smem = ((size_t)a.C + 2 * a.Hk) * sizeof(float);
  static bool configured = false;
  if (!configured) {
    cudaError_t e0 = cudaFuncSetAttribute(batch_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e0 != cudaSuccess) return e0;
    configured = true;
  }
  if (prep_smem > 200 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = launch_attr(reinterpret_cast<const void *>(batch_prep_kernel<D>), dim3(a.B, 1), kPrepThreads, lc,
                              args, prep_smem);
  if (e != cudaSuccess) return e;
  const int ns = a.slices > 0 ? a.slices : 1;
  const void *dk = nullptr;
  int threads = 0;
  if (ns >= 2 && D >= 64) {
    dk = a.state_bf16 ? reinterpret_cast<const void *>(batch_delta_kernel<D, 2, true>)
                      : reinterpret_cast<const void *>(batch_delta_kernel<D, 2, false>);
    threads = (D / 2 / bd_rows_per_warp<2>()) * 32;
  } else {
    dk = a.state_bf16 ? reinterpret_cast<const void *>(batch_delta_kernel<D, 1, true>)
                      : reinterpret_cast<const void *>(batch_delta_kernel<D, 1, false>);
    threads = (D / bd_rows_per_warp<1>()) * 32;
  }
  const int nsl = (ns >= 2 && D >= 64) ? 2 : 1;
  e = launch_attr(dk, dim3(a.Hv * nsl, a.B), threads, lc, args);
  if (e != cudaSuccess) return e;
  return launch_attr(reinterpret_cast<const void *>(batch_gnorm_kernel<D>), dim3(a.Hv, a.B), D, lc, args);
}

}  // namespace

cudaError_t launch_batch_mix(const MixArgs &a, const BatchWs &w, const LaunchCtx &lc) {
  if (a.B <= 0) return cudaSuccess;
  if (!a.y_codes || !a.y_scales || a.io_mul || a.ssm_src || a.conv_src) return cudaErrorInvalidValue;
  switch (a.D) {
    case 128: return launch_batch_d<128>(a, w, lc);
    case 64: return launch_batch_d<64>(a, w, lc);
    case 32: return launch_batch_d<32>(a, w, lc);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
