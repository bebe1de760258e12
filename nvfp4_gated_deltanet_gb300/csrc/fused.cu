// One decode layer-step for one or two rows as a single persistent kernel.
//
// At one or two rows the step is latency-bound: three dependent kernels each
// wait for the previous grid to finish and then fetch what it wrote. Here one
// cooperative launch (one CTA per SM, all resident) does the whole step:
//
//   prologue  every CTA bulk-copies (cp.async.bulk) its share of BOTH weight
//             matrices and the recurrent state of its (row, value head) unit
//             into shared memory -- the step's whole HBM traffic is requested
//             in the first microsecond -- and quantises x into shared memory.
//   phase A   in-projection rows of this CTA (the CUDA-core block-exact
//             product of gemv_core.cuh) -> q|k|v|z|b|a in global scratch
//   barrier   grid barrier (bounded spin)
//   phase B   conv + SiLU, q/k L2 norm, gates, gated delta rule on the state
//             rows already in shared memory, gated RMSNorm, NVFP4 quantise of y
//   barrier
//   phase C   q/k conv state written back (its readers are done), y expanded
//             into shared memory, out-projection rows of this CTA -> out
//
// The arithmetic of every stage is that of the three-kernel path in the same
// order (the same dot products, reductions and roundings), so the two paths
// give the same results.
#include "common.cuh"
#include "gemv_core.cuh"

namespace gdn {

namespace {

constexpr int kThreadsF = 512;   // 16 warps
constexpr int kDF = 128;         // head size of this kernel

// Grid barrier over all CTAs of a cooperative launch: arrival counter + a
// generation word, both in global memory (bar[0], bar[1]; the host zeroes them
// before every launch), reusable within the launch (the last arriver resets
// the counter before releasing). The wait is bounded by `budget` SM cycles;
// a CTA that gives up records GDN_E_TIMEOUT at once and returns false.
GDN_DEV bool grid_barrier(unsigned int *bar, unsigned int nblocks, long long budget, int32_t *status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile unsigned int *vgen = bar + 1;
    const unsigned int gen = *vgen;
    __threadfence();
    const unsigned int arrived = atomicAdd(bar, 1u) + 1u;
    if (arrived == nblocks) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const long long t0 = clock64();
      while (*vgen == gen) {
        if (clock64() - t0 > budget) {
          ok = 0;
          flag_status(status, GDN_E_TIMEOUT);
          break;
        }
        __nanosleep(20);
      }
      __threadfence();
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

template <int MB>
struct FusedSmem {
  // byte offsets inside dynamic shared memory (all multiples of 128)
  size_t bars, win, wout, state, act, mix, total;
  __host__ __device__ FusedSmem(int rows_in, int rows_out, int H, int Vd) {
    bars = 0;
    win = 128;
    const size_t win_bytes = (size_t)rows_in * (H / 2 + H / 16);
    wout = (win + win_bytes + 127) / 128 * 128;
    const size_t wout_bytes = (size_t)rows_out * (Vd / 2 + Vd / 16);
    state = (wout + wout_bytes + 127) / 128 * 128;
    act = state + (size_t)kDF * kDF * 4;
    const size_t ax = act_smem_bytes(MB, H), ay = act_smem_bytes(MB, Vd);
    mix = (act + (ax > ay ? ax : ay) + 127) / 128 * 128;
    total = mix + 5 * kDF * 4 + 3 * 2 * kDF * 2 + 64;
  }
};

template <int MB>
__global__ void __launch_bounds__(kThreadsF, 1) decode_fused_kernel(FusedArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int D = kDF;
  constexpr int EPL = D / 32;
  constexpr int kRPW = 8;
  const FusedSmem<MB> L(a.rows_in, a.rows_out, a.H, a.Vd);
  uint64_t *mb_in = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint64_t *mb_out = mb_in + 1, *mb_st = mb_in + 2;
  unsigned char *win = smem + L.win, *wout = smem + L.wout;
  float *stS = reinterpret_cast<float *>(smem + L.state);
  uint4 *ah = reinterpret_cast<uint4 *>(smem + L.act);
  float *sq = reinterpret_cast<float *>(smem + L.mix), *sk = sq + D, *sv = sk + D, *so = sv + D, *sy = so + D;
  uint16_t *qknew = reinterpret_cast<uint16_t *>(sy + D);  // [3][2D]
  float *gsum = reinterpret_cast<float *>(qknew + 3 * 2 * D);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H, Vd = a.Vd, G = a.Hv / a.Hk;
  const int cbin = H / 2, sbin = H / 16, cbout = Vd / 2, sbout = Vd / 16;
  const int ri0 = min((int)blockIdx.x * a.rows_in, a.Nin), ri1 = min(ri0 + a.rows_in, a.Nin);
  const int ro0 = min((int)blockIdx.x * a.rows_out, H), ro1 = min(ro0 + a.rows_out, H);
  // this CTA's mixing unit (row b, value head h), if any
  const int unit = blockIdx.x;
  const bool has_unit = unit < a.B * a.Hv;
  const int ub = has_unit ? unit / a.Hv : 0, uh = has_unit ? unit % a.Hv : 0;
  int uslot = has_unit ? a.slot_ids[ub] : -1;
  bool ulive = uslot >= 0 && uslot < a.num_slots;
  bool ubad = has_unit && (uslot < -1 || uslot >= a.num_slots);
  if (ulive)
    for (int j = 0; j < a.B; ++j)
      if (j != ub && a.slot_ids[j] == uslot) { ulive = false; ubad = true; }

  // ---------------------------------------------------------------- prologue
  if (tid == 0) {
    mbar_init(mb_in, 1);
    mbar_init(mb_out, 1);
    mbar_init(mb_st, 1);
    fence_barrier_init();
    const uint32_t cbi = (uint32_t)((ri1 - ri0) * cbin), sbi = (uint32_t)((ri1 - ri0) * sbin);
    mbar_arrive_expect_tx(mb_in, cbi + sbi);
    if (cbi) {
      bulk_g2s(win, a.w_in_codes + (size_t)ri0 * cbin, cbi, mb_in);
      bulk_g2s(win + (size_t)a.rows_in * cbin, a.w_in_scales + (size_t)ri0 * sbin, sbi, mb_in);
    }
    const uint32_t cbo = (uint32_t)((ro1 - ro0) * cbout), sbo = (uint32_t)((ro1 - ro0) * sbout);
    mbar_arrive_expect_tx(mb_out, cbo + sbo);
    if (cbo) {
      bulk_g2s(wout, a.w_out_codes + (size_t)ro0 * cbout, cbo, mb_out);
      bulk_g2s(wout + (size_t)a.rows_out * cbout, a.w_out_scales + (size_t)ro0 * sbout, sbo, mb_out);
    }
    if (ulive) {
      mbar_arrive_expect_tx(mb_st, D * D * 4);
      bulk_g2s(stS, a.ssm_state + ((size_t)uslot * a.Hv + uh) * D * D, D * D * 4, mb_st);
    }
  }
  if (ubad && tid == 0) flag_status(a.status, GDN_E_RANGE);
  // x -> NVFP4 -> FP16 E2M1 values in shared memory (every CTA, MB rows)
  {
    const int nblk = H >> 4, npiece = H >> 5;
    const float inv6ts = inv6ts_of(a.ts_in);
    float *xs = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(ah) + (size_t)MB * 4 * npiece * 16);
    for (int t = tid; t < MB * nblk; t += kThreadsF) {
      const int m = t / nblk, j = t % nblk;
      uint32_t lo = 0, hi = 0, s = 0;
      bool live = m < a.B;
      if (live) {
        const int sl = a.slot_ids[m];
        live = sl >= 0 && sl < a.num_slots;
      }
      if (live) {
        const uint4 *p = reinterpret_cast<const uint4 *>(a.x + (size_t)m * H + j * 16);
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
        if (!quant_block16(v, a.ts_in, inv6ts, lo, hi, s) && blockIdx.x == 0) flag_status(a.status, GDN_E_NONFINITE);
      }
      store_act_block(ah, xs, npiece, m, j, lo, hi, s);
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- phase A
  bool ok = true;
  {
    const int npiece = H >> 5;
    const float *xs = reinterpret_cast<const float *>(reinterpret_cast<const unsigned char *>(ah) +
                                                      (size_t)MB * 4 * npiece * 16);
    if (!mbar_wait(mb_in, 0)) ok = false;
    constexpr int NV = 2 * MB;
    const unsigned char *wsc = win + (size_t)a.rows_in * cbin;
    for (int n0 = ri0 + 2 * warp; ok && n0 < ri1; n0 += 2 * (kThreadsF / 32)) {
      const int nr = min(2, ri1 - n0);
      float v[NV];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float acc[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.0f;
        if (r < nr)
          dot_row<MB>(win + (size_t)(n0 + r - ri0) * cbin, wsc + (size_t)(n0 + r - ri0) * sbin, npiece, a.B, ah, xs,
                      lane, acc);
#pragma unroll
        for (int m = 0; m < MB; ++m) v[r * MB + m] = acc[m];
      }
      const float tot = warp_transpose_reduce<NV>(v, lane);
      const int idx = reduce_index<NV>(lane);
      const int r = idx / MB, m = idx % MB, n = n0 + r;
      if (lane == reduce_owner<NV>(idx) && m < a.B && r < nr) {
        const float tsw = n < a.Nqkvz ? a.ts_qkvz : a.ts_ba;
        a.proj[(size_t)m * a.Nin + n] = f32_to_bf16_bits(tot * (a.ts_in * tsw));
      }
    }
  }
  if (!grid_barrier(a.bar, gridDim.x, a.wait_cycles, a.status)) ok = false;

  // ---------------------------------------------------------------- phase B
  const int kh = uh / G;
  const int C = a.C, Kc = a.Kc;
  uint16_t *cst = a.conv_state + (size_t)(ulive ? uslot : 0) * (Kc - 1) * C;
  if (has_unit && !ulive) {  // padding row: zero y for this head, no state touched
    for (int i = tid; i < D; i += kThreadsF) {
      if ((i & 1) == 0) a.y_codes[((size_t)ub * Vd + uh * D + i) >> 1] = 0;
      if ((i & 15) == 0) a.y_scales[((size_t)ub * Vd + uh * D + i) >> 4] = 0;
    }
  }
  if (ulive) {
    const uint16_t *xin = a.proj + (size_t)ub * a.Nin;
    // conv + SiLU: q, k of key head kh and v of head uh (one channel per thread)
    if (tid < 3 * D) {
      int ch;
      if (tid < D) ch = kh * D + tid;
      else if (tid < 2 * D) ch = a.Hk * D + kh * D + (tid - D);
      else ch = 2 * a.Hk * D + uh * D + (tid - 2 * D);
      uint16_t tap[3];
#pragma unroll
      for (int j = 0; j < 3; ++j) tap[j] = j < Kc - 1 ? cst[(size_t)j * C + ch] : uint16_t(0);
      const uint16_t xn = xin[ch];
      float pre = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < Kc) {
          const uint16_t bits = j < Kc - 1 ? tap[j < 3 ? j : 2] : xn;
          pre = fmaf(bf16_bits_to_f32(a.conv_w[(size_t)ch * Kc + j]), bf16_bits_to_f32(bits), pre);
        }
      }
      const float outv = siluf_(pre);
      if (tid < D) sq[tid] = outv;
      else if (tid < 2 * D) sk[tid - D] = outv;
      else sv[tid - 2 * D] = outv;
      if (tid < 2 * D) {
        for (int j = 0; j < Kc - 2; ++j) qknew[j * 2 * D + tid] = tap[j + 1 < 3 ? j + 1 : 2];
        qknew[(Kc - 2) * 2 * D + tid] = xn;
      } else {  // v channels belong to this unit alone
        for (int j = 0; j < Kc - 2; ++j) cst[(size_t)j * C + ch] = tap[j + 1 < 3 ? j + 1 : 2];
        cst[(size_t)(Kc - 2) * C + ch] = xn;
      }
    }
    __syncthreads();
    float kr[EPL], qr[EPL];
    float ssk = 0.0f, ssq = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kr[e] = sk[lane * EPL + e];
      qr[e] = sq[lane * EPL + e];
      ssk = fmaf(kr[e], kr[e], ssk);
      ssq = fmaf(qr[e], qr[e], ssq);
    }
    ssk = warp_sum(ssk);
    ssq = warp_sum(ssq);
    const float rk = 1.0f / sqrtf(ssk + a.l2_eps);
    const float rq = (1.0f / sqrtf(ssq + a.l2_eps)) * (1.0f / sqrtf((float)D));
    float kq = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kr[e] *= rk;
      qr[e] *= rq;
      kq = fmaf(kr[e], qr[e], kq);
    }
    kq = warp_sum(kq);
    const uint16_t *bain = xin + a.Nqkvz;
    const float beta = sigmoidf_(bf16_bits_to_f32(bain[uh]));
    const float g = -expf(a.A_log[uh]) * softplusf_(bf16_bits_to_f32(bain[a.Hv + uh]) + a.dt_bias[uh]);
    const float alpha = expf(g);
    if (!mbar_wait(mb_st, 0)) ok = false;
    {
      const int lr0 = warp * kRPW;
      float *Sg = a.ssm_state + (((size_t)uslot * a.Hv + uh) * D + lr0) * D + lane * EPL;
      float st[kRPW][EPL];
#pragma unroll
      for (int j = 0; j < kRPW; ++j) {
        const float4 t4 = *reinterpret_cast<const float4 *>(stS + (size_t)(lr0 + j) * D + lane * EPL);
        st[j][0] = t4.x; st[j][1] = t4.y; st[j][2] = t4.z; st[j][3] = t4.w;
      }
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
#pragma unroll
      for (int j = 0; j < kRPW; ++j) {
        const float Sk = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * kRPW>(j));
        const float Sq = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * kRPW>(kRPW + j));
        const float u = beta * (sv[lr0 + j] - alpha * Sk);
        const float o = fmaf(u, kq, alpha * Sq);
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[j][e] = fmaf(u, kr[e], alpha * st[j][e]);
        if (lane == 0) so[lr0 + j] = o;
      }
#pragma unroll
      for (int j = 0; j < kRPW; ++j)
        *reinterpret_cast<float4 *>(Sg + (size_t)j * D) = make_float4(st[j][0], st[j][1], st[j][2], st[j][3]);
    }
    __syncthreads();
    if (tid < D / 16) {
      float p = 0.0f;
      for (int i = 0; i < 16; ++i) p = fmaf(so[tid * 16 + i], so[tid * 16 + i], p);
      gsum[tid] = p;
    }
    __syncthreads();
    float sumsq = 0.0f;
    for (int gi = 0; gi < D / 16; ++gi) sumsq += gsum[gi];
    const float rstd = 1.0f / sqrtf(sumsq / (float)D + a.rms_eps);
    if (tid < D) {
      const float zv = bf16_bits_to_f32(xin[2 * a.Hk * D + Vd + uh * D + tid]);
      sy[tid] = so[tid] * rstd * a.norm_w[tid] * siluf_(zv);
    }
    __syncthreads();
    if (tid < D / 16) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = sy[tid * 16 + i];
      uint32_t lo, hi, s;
      if (!quant_block16(v, a.ts_out, inv6ts_of(a.ts_out), lo, hi, s)) flag_status(a.status, GDN_E_NONFINITE);
      const size_t e0 = (size_t)ub * Vd + uh * D + tid * 16;
      *reinterpret_cast<uint2 *>(a.y_codes + (e0 >> 1)) = make_uint2(lo, hi);
      a.y_scales[e0 >> 4] = uint8_t(s);
    }
  }
  if (!grid_barrier(a.bar, gridDim.x, a.wait_cycles, a.status)) ok = false;

  // ---------------------------------------------------------------- phase C
  if (ulive && uh % G == 0) {  // every reader of this key head's q/k conv state is done
    for (int t = tid; t < 2 * D; t += kThreadsF) {
      const int q = t < D ? kh * D + t : a.Hk * D + kh * D + (t - D);
      for (int j = 0; j < Kc - 1; ++j) cst[(size_t)j * C + q] = qknew[j * 2 * D + t];
    }
  }
  {
    const int nblk = Vd >> 4, npiece = Vd >> 5;
    float *ys = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(ah) + (size_t)MB * 4 * npiece * 16);
    for (int t = tid; t < MB * nblk; t += kThreadsF) {
      const int m = t / nblk, j = t % nblk;
      uint32_t lo = 0, hi = 0, s = 0;
      if (m < a.B) {
        const uint2 c = *reinterpret_cast<const uint2 *>(a.y_codes + (size_t)m * cbout + j * 8);
        lo = c.x;
        hi = c.y;
        s = a.y_scales[(size_t)m * nblk + j];
      }
      store_act_block(ah, ys, npiece, m, j, lo, hi, s);
    }
    __syncthreads();
    if (!mbar_wait(mb_out, 0)) ok = false;
    constexpr int NV = 2 * MB;
    const unsigned char *wsc = wout + (size_t)a.rows_out * cbout;
    for (int n0 = ro0 + 2 * warp; ok && n0 < ro1; n0 += 2 * (kThreadsF / 32)) {
      const int nr = min(2, ro1 - n0);
      float v[NV];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float acc[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.0f;
        if (r < nr)
          dot_row<MB>(wout + (size_t)(n0 + r - ro0) * cbout, wsc + (size_t)(n0 + r - ro0) * sbout, npiece, a.B, ah,
                      ys, lane, acc);
#pragma unroll
        for (int m = 0; m < MB; ++m) v[r * MB + m] = acc[m];
      }
      const float tot = warp_transpose_reduce<NV>(v, lane);
      const int idx = reduce_index<NV>(lane);
      const int r = idx / MB, m = idx % MB, n = n0 + r;
      if (lane == reduce_owner<NV>(idx) && m < a.B && r < nr)
        a.out[(size_t)m * H + n] = f32_to_bf16_bits(tot * (a.ts_out * a.ts_wout));
    }
  }
  if (!ok && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
  // copies that never got waited on (a timeout) must land before shared memory goes away
  if (tid == 0 && ulive) (void)mbar_wait(mb_st, 0);
}

template <int MB>
cudaError_t launch_fused_mb(const FusedArgs &a, const LaunchCtx &lc) {
  const FusedSmem<MB> L(a.rows_in, a.rows_out, a.H, a.Vd);
  if (L.total > 226 * 1024) return cudaErrorInvalidValue;
  static size_t configured = 0;  // the kernel also has a little static shared memory
  if (configured < L.total) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_fused_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
    if (e != cudaSuccess) return e;
    configured = L.total;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(lc.num_sms, 1, 1);
  cfg.blockDim = dim3(kThreadsF, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel<MB>, a);
}

}  // namespace

// Whether the fused kernel covers this shape on this GPU, and the per-CTA row
// shares it would use (one CTA per SM).
bool fused_plan(FusedArgs &a, int num_sms) {
  if (a.D != kDF || a.B < 1 || a.B > 2 || a.H % 256 || a.Vd % 256 || a.Hv > num_sms) return false;
  a.rows_in = ((a.Nin + num_sms - 1) / num_sms + 1) & ~1;
  a.rows_out = ((a.H + num_sms - 1) / num_sms + 1) & ~1;
  if (a.B * a.Hv > num_sms) return false;
  const size_t need = a.B == 1 ? FusedSmem<1>(a.rows_in, a.rows_out, a.H, a.Vd).total
                               : FusedSmem<2>(a.rows_in, a.rows_out, a.H, a.Vd).total;
  return need <= 226 * 1024;
}

cudaError_t launch_fused(const FusedArgs &a, const LaunchCtx &lc) {
  return a.B == 1 ? launch_fused_mb<1>(a, lc) : launch_fused_mb<2>(a, lc);
}

}  // namespace gdn
