// Prefill of one sequence: the decode arithmetic applied to T tokens, split
// into token-parallel stages around the one sequential part, the recurrence.
//
//   prep      (token, key head)  conv + SiLU of q, k and the group's v channels,
//                                 q/k L2 norm, beta and alpha = exp(g)
//   recur     (value head, rows) S kept in registers across all T tokens
//   gnorm     (token)            z-gated RMSNorm + NVFP4 quantisation of y
//   conv_tail (channel)          the slot's conv state after the last token
#include "common.cuh"

namespace gdn {


namespace {

// raw conv input of channel `ch` at token `tau` (tau < 0 reads the state)
GDN_DEV float conv_in(const PrefillArgs &a, int tau, int ch) {
  if (tau >= 0) return bf16_bits_to_f32(a.proj[(size_t)tau * a.ld + ch]);
  return bf16_bits_to_f32(a.conv_state[(size_t)(a.Kc - 1 + tau) * a.C + ch]);
}

// one CTA per (token, key head); blockDim = 128
__global__ void __launch_bounds__(128) prep_kernel(PrefillArgs a) {
  extern __shared__ float sm[];
  const int t = blockIdx.x, kh = blockIdx.y;
  const int D = a.D, G = a.Hv / a.Hk;
  float *sq = sm, *sk = sm + D;
  const int nch = 2 * D + G * D;
  for (int i = threadIdx.x; i < nch; i += blockDim.x) {
    int ch;
    if (i < D) ch = kh * D + i;
    else if (i < 2 * D) ch = a.Hk * D + kh * D + (i - D);
    else ch = 2 * a.Hk * D + kh * G * D + (i - 2 * D);
    float pre = 0.0f;
    for (int j = 0; j < a.Kc; ++j)
      pre = fmaf(bf16_bits_to_f32(a.conv_w[(size_t)ch * a.Kc + j]), conv_in(a, t - (a.Kc - 1) + j, ch), pre);
    const float y = siluf_(pre);
    if (i < 2 * D) sm[i] = y;
    else a.v[((size_t)t * a.Hv + kh * G) * D + (i - 2 * D)] = y;
  }
  __syncthreads();
  // norms exactly as the decode kernel takes them: lane-local sums over D/32
  // consecutive elements, then the warp butterfly (warp 0: q, warp 1: k)
  __shared__ float ss[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < 2) {
    const float *src = warp == 0 ? sq : sk;
    const int epl = D / 32;
    float p = 0.0f;
    for (int e = 0; e < epl; ++e) p = fmaf(src[lane * epl + e], src[lane * epl + e], p);
    p = warp_sum(p);
    if (lane == 0) ss[warp] = p;
  }
  __syncthreads();
  const float rq = (1.0f / sqrtf(ss[0] + a.l2_eps)) * (1.0f / sqrtf((float)D));
  const float rk = 1.0f / sqrtf(ss[1] + a.l2_eps);
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    a.qn[((size_t)t * a.Hk + kh) * D + i] = sq[i] * rq;
    a.kn[((size_t)t * a.Hk + kh) * D + i] = sk[i] * rk;
  }
  if (threadIdx.x < G) {
    const int h = kh * G + threadIdx.x;
    const uint16_t *ba = a.proj + (size_t)t * a.ld + 2 * a.Hk * D + 2 * a.Hv * D;
    const float bt = sigmoidf_(bf16_bits_to_f32(ba[h]));
    const float g = -expf(a.A_log[h]) * softplusf_(bf16_bits_to_f32(ba[a.Hv + h]) + a.dt_bias[h]);
    a.beta[(size_t)t * a.Hv + h] = bt;
    a.alpha[(size_t)t * a.Hv + h] = expf(g);
  }
}

constexpr int kRPW = 8;

// one warp owns kRPW rows of one value head's state for the whole sequence
template <int D>
__global__ void __launch_bounds__(128) recur_kernel(PrefillArgs a) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int wph = D / kRPW;  // warps per head
  const int h = gw / wph;
  if (h >= a.Hv) return;
  const int r0 = (gw % wph) * kRPW;
  const int kh = h / (a.Hv / a.Hk);
  float *S = a.ssm + ((size_t)h * D + r0) * D + lane * EPL;
  float st[kRPW][EPL];
#pragma unroll
  for (int j = 0; j < kRPW; ++j)
#pragma unroll
    for (int e = 0; e < EPL; ++e) st[j][e] = S[(size_t)j * D + e];

  for (int t = 0; t < a.T; ++t) {
    float kr[EPL], qr[EPL];
    const float *kp = a.kn + ((size_t)t * a.Hk + kh) * D + lane * EPL;
    const float *qp = a.qn + ((size_t)t * a.Hk + kh) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) { kr[e] = kp[e]; qr[e] = qp[e]; }
    const float beta = a.beta[(size_t)t * a.Hv + h];
    const float alpha = a.alpha[(size_t)t * a.Hv + h];
    const float *vp = a.v + ((size_t)t * a.Hv + h) * D + r0;
    float kq = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) kq = fmaf(kr[e], qr[e], kq);
    float red[2 * kRPW];
#pragma unroll
    for (int j = 0; j < kRPW; ++j) {
      float dk = 0.0f, dq = 0.0f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        dk = fmaf(st[j][e], kr[e], dk);
        dq = fmaf(st[j][e], qr[e], dq);
      }
      red[j] = dk;
      red[kRPW + j] = dq;
    }
    const float tot = warp_transpose_reduce<2 * kRPW>(red, lane);
    kq = warp_sum(kq);
    float my_o = 0.0f;
#pragma unroll
    for (int j = 0; j < kRPW; ++j) {
      const float Sk = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * kRPW>(j));
      const float Sq = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * kRPW>(kRPW + j));
      const float u = beta * (vp[j] - alpha * Sk);
      const float o = fmaf(u, kq, alpha * Sq);
#pragma unroll
      for (int e = 0; e < EPL; ++e) st[j][e] = fmaf(u, kr[e], alpha * st[j][e]);
      if (lane == j) my_o = o;
    }
    if (lane < kRPW) a.o[((size_t)t * a.Hv + h) * D + r0 + lane] = my_o;
  }
#pragma unroll
  for (int j = 0; j < kRPW; ++j)
#pragma unroll
    for (int e = 0; e < EPL; ++e) S[(size_t)j * D + e] = st[j][e];
}

// one CTA per token; thread i owns 16-block i of y (head i / (D/16))
__global__ void gnorm_kernel(PrefillArgs a) {
  const int t = blockIdx.x;
  const int D = a.D, vd = a.Hv * D;
  const int nblk = vd / 16;
  const int i = min((int)threadIdx.x, nblk - 1);  // block index within the token; spare lanes
                                                   // shadow the last block and store nothing
  const int per_head = D / 16;          // threads per head: 2, 4 or 8 (a power of two)
  const int h = i / per_head, e0 = (i % per_head) * 16;
  const float *op = a.o + ((size_t)t * a.Hv + h) * D + e0;
  const uint16_t *zp = a.proj + (size_t)t * a.ld + 2 * a.Hk * D + vd + h * D + e0;
  float ov[16];
  float p = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    ov[k] = op[k];
    p = fmaf(ov[k], ov[k], p);
  }
  // the head's 16-element group sums added in group order (as in decode)
  const int first = (threadIdx.x & 31) & ~(per_head - 1);
  float tot = 0.0f;
  for (int m = 0; m < per_head; ++m) tot += __shfl_sync(0xffffffffu, p, first + m);
  p = tot;
  const float rstd = 1.0f / sqrtf(p / (float)D + a.rms_eps);
  float y[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) y[k] = ov[k] * rstd * a.norm_w[e0 + k] * siluf_(bf16_bits_to_f32(zp[k]));
  uint32_t lo, hi, s;
  const bool ok = quant_block16(y, a.ts_out, inv6ts_of(a.ts_out), lo, hi, s);
  if ((int)threadIdx.x >= nblk) return;
  if (!ok) flag_status(a.status, GDN_E_NONFINITE);
  const size_t b0 = (size_t)t * vd + h * D + e0;
  *reinterpret_cast<uint2 *>(a.y_codes + (b0 >> 1)) = make_uint2(lo, hi);
  a.y_scales[b0 >> 4] = uint8_t(s);
}

// the slot's conv state after the last token: taps hold inputs T-K+1 .. T-1
__global__ void conv_tail_kernel(PrefillArgs a, uint16_t *tmp) {
  const int n = (a.Kc - 1) * a.C;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int j = i / a.C, ch = i % a.C;
    const int tau = a.T - (a.Kc - 1) + j;
    tmp[i] = tau >= 0 ? a.proj[(size_t)tau * a.ld + ch] : a.conv_state[(size_t)(a.Kc - 1 + tau) * a.C + ch];
  }
}

__global__ void copy_u16_kernel(uint16_t *dst, const uint16_t *src, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

}  // namespace

// The stages between the projections (run by the caller) and the out
// projection. `tmp` holds (K-1)*C BF16 values.
cudaError_t launch_prefill_mix(const PrefillArgs &a, uint16_t *tmp, const LaunchCtx &lc) {
  prep_kernel<<<dim3(a.T, a.Hk), 128, 2 * a.D * sizeof(float), lc.stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // conv state tail is computed from the old state before anything overwrites it
  const int n = (a.Kc - 1) * a.C;
  conv_tail_kernel<<<(n + 255) / 256, 256, 0, lc.stream>>>(a, tmp);
  const int warps = a.Hv * (a.D / kRPW);
  const int ctas = (warps + 3) / 4;
  switch (a.D) {
    case 128: recur_kernel<128><<<ctas, 128, 0, lc.stream>>>(a); break;
    case 64: recur_kernel<64><<<ctas, 128, 0, lc.stream>>>(a); break;
    case 32: recur_kernel<32><<<ctas, 128, 0, lc.stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  const int gthreads = ((a.Hv * a.D / 16) + 31) / 32 * 32;
  gnorm_kernel<<<a.T, gthreads, 0, lc.stream>>>(a);
  copy_u16_kernel<<<(n + 255) / 256, 256, 0, lc.stream>>>(a.conv_state, tmp, n);
  return cudaGetLastError();
}

}  // namespace gdn
