// KDA-style recurrent step: the gated delta rule with one decay per key
// channel (Rocket blog, "Moving the KDA state tile out of shared memory is
// 4.6x at M=8": a 64 x 128 x 128 state per stream, read and written every
// step; its lesson -- keep the state columns in registers, not in a shared
// tile, so many warps stay resident -- is the design here).
//
//   S <- S diag(exp(g));  u = beta (v - S k);  S <- S + u k^T;  o = S q
//
// One CTA per (stream, head, d_v slice); each warp keeps RPW state rows in
// registers, one row over the 32 lanes (EPL consecutive d_k elements per lane,
// so the lane also owns those channels' decays). S k and S q of the decayed
// state are row dot products reduced with one transpose-reduction; then
// o = (S diag(a)) q + u (k . q) and S <- a * S + u k, element-wise in registers.
#include "common.cuh"

namespace gdn {

namespace {

template <int NS>
__host__ __device__ constexpr int kda_rows_per_warp() { return NS == 1 ? 16 : 8; }

template <int D, int NS, bool SB>
__global__ void __launch_bounds__((D / NS / kda_rows_per_warp<NS>()) * 32) kda_step_kernel(KdaArgs a) {
  constexpr int R = D / NS;
  constexpr int RPW = kda_rows_per_warp<NS>();
  constexpr int EPL = D / 32;
  static_assert(R % RPW == 0 && EPL >= 1 && EPL <= 4, "shape");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int mh = blockIdx.y;                  // stream * H + head
  const int row0 = blockIdx.x * R + warp * RPW;
  constexpr size_t kEs = SB ? 2 : 4;
  char *base = static_cast<char *>(a.state) + (((size_t)mh * D + row0) * D + lane * EPL) * kEs;

  // state rows first (the bytes), then this lane's channels of q, k, g
  float st[RPW][EPL];
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const char *p = base + (size_t)j * D * kEs;
    if (SB) {
      uint16_t b[EPL];
      if (EPL == 4) {
        const uint2 t = *reinterpret_cast<const uint2 *>(p);
        b[0] = t.x & 0xFFFFu; b[1 % EPL] = t.x >> 16; b[2 % EPL] = t.y & 0xFFFFu; b[3 % EPL] = t.y >> 16;
      } else if (EPL == 2) {
        const uint32_t t = *reinterpret_cast<const uint32_t *>(p);
        b[0] = t & 0xFFFFu; b[1 % EPL] = t >> 16;
      } else {
        b[0] = *reinterpret_cast<const uint16_t *>(p);
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) st[j][e] = bf16_bits_to_f32(b[e]);
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
  const size_t ch = (size_t)mh * D + lane * EPL;
  float qv[EPL], kv[EPL], al[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    qv[e] = a.q[ch + e];
    kv[e] = a.k[ch + e];
    al[e] = expf(a.g[ch + e]);
  }
  const float beta = a.beta[mh];
  float vr[RPW];
#pragma unroll
  for (int j = 0; j < RPW; ++j) vr[j] = a.v[(size_t)mh * D + row0 + j];

  float kq = 0.0f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) kq = fmaf(kv[e], qv[e], kq);
  kq = warp_sum(kq);

  // (S diag(a)) k and (S diag(a)) q for each row
  float vals[2 * RPW];
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    float dk = 0.0f, dq = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float s = al[e] * st[j][e];
      st[j][e] = s;
      dk = fmaf(s, kv[e], dk);
      dq = fmaf(s, qv[e], dq);
    }
    vals[j] = dk;
    vals[RPW + j] = dq;
  }
  const float tot = warp_transpose_reduce<2 * RPW>(vals, lane);
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    const float Sk = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * RPW>(j));
    const float Sq = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * RPW>(RPW + j));
    const float u = beta * (vr[j] - Sk);
    if (lane == 0) a.o[(size_t)mh * D + row0 + j] = fmaf(u, kq, Sq);
#pragma unroll
    for (int e = 0; e < EPL; ++e) st[j][e] = fmaf(u, kv[e], st[j][e]);
  }
#pragma unroll
  for (int j = 0; j < RPW; ++j) {
    char *p = base + (size_t)j * D * kEs;
    if (SB) {
      uint32_t b[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) b[e] = f32_to_bf16_bits(st[j][e]);
      if (EPL == 4)
        *reinterpret_cast<uint2 *>(p) = make_uint2(b[0] | (b[1 % EPL] << 16), b[2 % EPL] | (b[3 % EPL] << 16));
      else if (EPL == 2)
        *reinterpret_cast<uint32_t *>(p) = b[0] | (b[1 % EPL] << 16);
      else
        *reinterpret_cast<uint16_t *>(p) = (uint16_t)b[0];
    } else if (EPL == 4) {
      *reinterpret_cast<float4 *>(p) = make_float4(st[j][0], st[j][1 % EPL], st[j][2 % EPL], st[j][3 % EPL]);
    } else if (EPL == 2) {
      *reinterpret_cast<float2 *>(p) = make_float2(st[j][0], st[j][1 % EPL]);
    } else {
      *reinterpret_cast<float *>(p) = st[j][0];
    }
  }
}

template <int D, int NS>
cudaError_t launch_kda_t(const KdaArgs &a, cudaStream_t stream) {
  const dim3 grid(NS, a.M * a.H);
  const int threads = (D / NS / kda_rows_per_warp<NS>()) * 32;
  if (a.state_bf16)
    kda_step_kernel<D, NS, true><<<grid, threads, 0, stream>>>(a);
  else
    kda_step_kernel<D, NS, false><<<grid, threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

// Slices per head: spread few streams' state over more CTAs.
cudaError_t launch_kda(const KdaArgs &a, cudaStream_t stream) {
  if (a.M <= 0 || a.H <= 0) return cudaSuccess;
  const int heads = a.M * a.H;
  const int ns = heads < 152 ? 4 : (heads < 608 ? 2 : 1);
  switch (a.D) {
    case 128:
      return ns == 4 ? launch_kda_t<128, 4>(a, stream) : ns == 2 ? launch_kda_t<128, 2>(a, stream)
                                                                 : launch_kda_t<128, 1>(a, stream);
    case 64:
      return ns == 4 ? launch_kda_t<64, 4>(a, stream) : ns == 2 ? launch_kda_t<64, 2>(a, stream)
                                                                : launch_kda_t<64, 1>(a, stream);
    case 32:
      return ns >= 2 ? launch_kda_t<32, 2>(a, stream) : launch_kda_t<32, 1>(a, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
