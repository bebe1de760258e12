// Prefill of one sequence: the decode arithmetic over T tokens, with the gated
// delta rule in 64-token chunks (the WY / UT form; bloomery issue #565, §4,
// #812: the delta rule of a prompt runs in chunks on tensor cores).
//
// Within a chunk with start state S0 and rows i = 1..64 (per value head):
//   Gamma_i = sum_{j<=i} g_j,  D_ij = exp(Gamma_i - Gamma_j)  (j <= i)
//   L_ij = beta_i D_ij (k_i . k_j)  (j < i)
//   (I + L) [W | Ut] = [diag(beta e^Gamma) K | diag(beta) V]
//   U = Ut - W S0^T
//   O_i = e^Gamma_i (S0 q_i) + sum_{j<=i} D_ij (q_i . k_j) u_j
//   S_64 = e^Gamma_64 S0 + sum_j D_64j u_j k_j^T
// which is the token recurrence S <- a S; u = b (v - S k); S <- S + u k^T;
// o = S q rewritten over a chunk (u_i = beta_i (v_i - a_i S_{i-1} k_i)).
// Decays are formed only as exp of non-positive log differences, never as
// ratios, so decays down to -240 per token cannot overflow.
//
//   prep        (32 tokens, head)   conv + SiLU, q/k L2 norm, beta, g
//   chunk_prep  (chunk, value head) k.k and q.k, the triangular solve, W, Ut
//               (for d = 128 with the tcgen05 scan: k.k and q.k as one tcgen05
//               product in split FP16, K^T of the chunk for the scan)
//   chunk_scan  (value head, 32 rows of d_v), sequential over chunks: U, O,
//               and the state slice, kept on chip across chunks (scan_tc.cu:
//               the tcgen05 form)
//   gnorm       (token)             z-gated RMSNorm + NVFP4 quantisation of y
//   conv_tail   (channel)           the slot's conv state after the last token
// The chunk products run on warp-level tensor-core MMA in split TF32 (d = 128;
// FP32 on the CUDA cores for the smaller head sizes and on request).
#include "tc.cuh"

namespace gdn {

namespace {

constexpr int kC = 64;  // chunk length

// prep: one CTA (128 threads) per (64-token tile, group of D channels): the
// group is the q or k channels of one key head, or the v channels of one value
// head; group index 2*Hk + Hv .. handles beta and g. The conv window (tile +
// K-1 earlier tokens) is read once with 16-byte loads; a warp takes a token:
// conv + SiLU of its D channels straight from the window, then (q, k) the L2
// norm with lane-local sums over D/32 consecutive elements and the warp
// butterfly -- the decode kernel's order.
constexpr int kPrepTT = 64;

template <int D>
__global__ void __launch_bounds__(128) prep_kernel(PrefillArgs a) {
  __shared__ __align__(16) uint16_t win[kPrepTT + 3][D];
  const int t0 = blockIdx.x * kPrepTT, grp = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ngrp = 2 * a.Hk + a.Hv;
  if (grp == ngrp) {  // gates: beta and g for the tile's tokens and every value head
    for (int e = tid; e < kPrepTT * a.Hv; e += blockDim.x) {
      const int t = t0 + e / a.Hv, h = e % a.Hv;
      if (t >= a.T) continue;
      const uint16_t *ba = a.proj + (size_t)t * a.ld + 2 * a.Hk * D + 2 * a.Hv * D;
      a.beta[(size_t)h * a.Tp + t] = sigmoidf_(bf16_bits_to_f32(ba[h]));
      a.gl[(size_t)h * a.Tp + t] = -expf(a.A_log[h]) * softplusf_(bf16_bits_to_f32(ba[a.Hv + h]) + a.dt_bias[h]);
    }
    return;
  }
  const int ch0 = grp * D;  // q heads, then k heads, then v heads: the conv channel order
  const int Kc = a.Kc;
  // window rows r = 0 .. TT+Kc-2 hold tokens t0 - (Kc-1) + r (state rows for t < 0)
  constexpr int VPR = D / 8;  // 16-byte vectors per row
  if (a.ld % 8 == 0 && a.C % 8 == 0 && blockDim.x == 128) {  // every row starts 16-byte aligned
    // every load of the window issued before any is stored (read-only loads,
    // so they need not wait for the shared-memory stores)
    constexpr int kWin = ((kPrepTT + 3) * VPR + 127) / 128;
    const int nv = (kPrepTT + Kc - 1) * VPR;
    uint4 val[kWin];
#pragma unroll
    for (int q = 0; q < kWin; ++q) {
      const int e = tid + 128 * q;
      const int r = e / VPR, v = e % VPR;
      const int tau = t0 - (Kc - 1) + r;
      val[q] = make_uint4(0, 0, 0, 0);
      if (e < nv && tau >= 0 && tau < a.T)
        val[q] = __ldg(reinterpret_cast<const uint4 *>(a.proj + (size_t)tau * a.ld + ch0 + v * 8));
      else if (e < nv && tau < 0)
        val[q] = __ldg(reinterpret_cast<const uint4 *>(a.conv_state + (size_t)(Kc - 1 + tau) * a.C + ch0 + v * 8));
    }
#pragma unroll
    for (int q = 0; q < kWin; ++q) {
      const int e = tid + 128 * q;
      if (e < nv) *reinterpret_cast<uint4 *>(&win[e / VPR][(e % VPR) * 8]) = val[q];
    }
  } else {
    for (int e = tid; e < (kPrepTT + Kc - 1) * D; e += blockDim.x) {
      const int r = e / D, c = e % D;
      const int tau = t0 - (Kc - 1) + r;
      uint16_t val = 0;
      if (tau >= 0 && tau < a.T)
        val = a.proj[(size_t)tau * a.ld + ch0 + c];
      else if (tau < 0)
        val = a.conv_state[(size_t)(Kc - 1 + tau) * a.C + ch0 + c];
      win[r][c] = val;
    }
  }
  __syncthreads();
  // warp -> token, lane -> EPL consecutive channels: conv + SiLU straight from
  // the window, then (q, k) the L2 norm with lane-local sums and the warp
  // butterfly -- the decode kernel's order
  constexpr int EPL = D / 32;
  float w[EPL][4];
#pragma unroll
  for (int e = 0; e < EPL; ++e)
#pragma unroll
    for (int j = 0; j < 4; ++j) w[e][j] = j < Kc ? bf16_bits_to_f32(a.conv_w[(size_t)(ch0 + lane * EPL + e) * Kc + j]) : 0.0f;
  const int nq = a.Hk;  // groups 0..Hk-1: q, Hk..2Hk-1: k, then v
  const bool isq = grp < nq, isk = !isq && grp < 2 * nq;
  const bool split_qk = D == 128 && a.Qs && a.Ks;
  float *dst = isq ? a.qn + ((size_t)grp * a.Tp) * D
                   : isk ? a.kn + ((size_t)(grp - nq) * a.Tp) * D : a.v + ((size_t)(grp - 2 * nq) * a.Tp) * D;
  for (int i = warp; i < kPrepTT; i += blockDim.x / 32) {
    const int t = t0 + i;
    float o[EPL];
    if constexpr (EPL == 4) {
      // four channels per lane: one 8-byte window load per tap; SiLU with the
      // fast exponential and an IEEE reciprocal (the kernel is issue-bound)
      float pre[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < Kc) {
          const uint2 wv = *reinterpret_cast<const uint2 *>(&win[i + j][lane * 4]);
          pre[0] = fmaf(w[0][j], __uint_as_float(wv.x << 16), pre[0]);
          pre[1] = fmaf(w[1][j], __uint_as_float(wv.x & 0xFFFF0000u), pre[1]);
          pre[2] = fmaf(w[2][j], __uint_as_float(wv.y << 16), pre[2]);
          pre[3] = fmaf(w[3][j], __uint_as_float(wv.y & 0xFFFF0000u), pre[3]);
        }
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = pre[e] * __frcp_rn(1.0f + __expf(-pre[e]));
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        float pre = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < Kc) pre = fmaf(w[e][j], bf16_bits_to_f32(win[i + j][lane * EPL + e]), pre);
        o[e] = siluf_(pre);
      }
    }
    float r = 1.0f;
    if (isq || isk) {
      float p = 0.0f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) p = fmaf(o[e], o[e], p);
      p = warp_sum(p);
      r = rsqrtf(p + a.l2_eps) * (isq ? rsqrtf((float)D) : 1.0f);
    }
    if (split_qk && (isq || isk)) {
      // the tcgen05 chunk stages' q / k operand: x 2^14 = hi + lo in FP16,
      // zero for the padding tokens past T
      if constexpr (EPL == 4) {
        uint16_t *sp = (isq ? a.Qs + (size_t)grp * a.Tp * D : a.Ks + (size_t)(grp - nq) * a.Tp * D) + (size_t)t * D +
                       lane * EPL;
        const float sc = t < a.T ? r * 16384.0f : 0.0f;
        uint32_t h0, l0, h1, l1;
        split_f16x2(o[0] * sc, o[1] * sc, h0, l0);
        split_f16x2(o[2] * sc, o[3] * sc, h1, l1);
        *reinterpret_cast<uint2 *>(sp) = make_uint2(h0, h1);
        *reinterpret_cast<uint2 *>(sp + (size_t)a.Hk * a.Tp * D) = make_uint2(l0, l1);
      }
    } else if (t < a.T) {
      float *row = dst + (size_t)t * D + lane * EPL;
      if constexpr (EPL == 4) {  // one 16-byte store per lane
        *reinterpret_cast<float4 *>(row) = (isq || isk) ? make_float4(o[0] * r, o[1] * r, o[2] * r, o[3] * r)
                                                        : make_float4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) row[e] = (isq || isk) ? o[e] * r : o[e];
      }
    }
  }
}

// ---------------------------------------------------------------- split-TF32 warp MMA
// (used by chunk_prep and chunk_scan_tc: see the latter's comment)
GDN_DEV uint32_t tf32_of(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
GDN_DEV void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  hi = tf32_of(x);
  lo = tf32_of(x - __uint_as_float(hi));
}
GDN_DEV void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D += A B with A (16x8) as (row g, k t / g+8, t / g, t+4 / g+8, t+4) and B (8x8)
// as (k t / t+4, column g), each given as hi and lo TF32 parts.
GDN_DEV void mma3_split(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], const uint32_t (&bh)[2],
                        const uint32_t (&bl)[2]) {
  mma_tf32(d, al, bh[0], bh[1]);
  mma_tf32(d, ah, bl[0], bl[1]);
  mma_tf32(d, ah, bh[0], bh[1]);
}
GDN_DEV void split4(const float (&f)[4], uint32_t (&h)[4], uint32_t (&l)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) split_tf32(f[i], h[i], l[i]);
}
GDN_DEV void split2(const float (&f)[2], uint32_t (&h)[2], uint32_t (&l)[2]) {
  split_tf32(f[0], h[0], l[0]);
  split_tf32(f[1], h[1], l[1]);
}
// both operands split here
GDN_DEV void mma3(float (&d)[4], const float (&af)[4], const float (&bf)[2]) {
  uint32_t ah[4], al[4], bh[2], bl[2];
  split4(af, ah, al);
  split2(bf, bh, bl);
  mma3_split(d, ah, al, bh, bl);
}


// (I + L) X = R by forward substitution, one column per thread (no barriers):
// columns 0..D-1 give W (R = beta e^Gamma k), D..2D-1 give Ut (R = beta v).
// All right-hand sides are loaded first; rows of L are read 4 at a time.
// K and v rows in shared memory with row stride XLD; L strictly lower, rows
// LLD floats apart (a multiple of 4). BLOCKED: in blocks of 16 rows -- the
// block's own rows in order, then every later row takes the block's
// contribution (independent rows, no dependent chain in the long update);
// else row by row with four partial sums (the warp-MMA kernel's form, which
// measured faster beside that kernel's other phases).
template <int D, int XLD, int LLD = kC, bool BLOCKED = false>
GDN_DEV void chunk_solve(const PrefillArgs &a, const float *KR, const float *VR, const float *Lm, const float *bek,
                         const float *bet, int h, int c, int nc, int tid) {
  if (tid < 2 * D) {
    const int col = tid;
    float X[kC];
#pragma unroll
    for (int i = 0; i < kC; ++i) X[i] = col < D ? bek[i] * KR[i * XLD + col] : bet[i] * VR[i * XLD + (col - D)];
    if constexpr (BLOCKED) {
#pragma unroll
      for (int b0 = 0; b0 < kC; b0 += 16) {
#pragma unroll
        for (int i = b0 + 1; i < b0 + 16; ++i) {
          float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
          for (int j = b0; j < i; j += 2) {
            p0 = fmaf(Lm[i * LLD + j], X[j], p0);
            if (j + 1 < i) p1 = fmaf(Lm[i * LLD + j + 1], X[j + 1], p1);
          }
          X[i] -= p0 + p1;
        }
#pragma unroll
        for (int i = b0 + 16; i < kC; ++i) {
          float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
          for (int j = b0; j < b0 + 16; j += 4) {
            const float4 l = *reinterpret_cast<const float4 *>(Lm + i * LLD + j);
            p0 = fmaf(l.x, X[j], p0);
            p1 = fmaf(l.y, X[j + 1], p1);
            p0 = fmaf(l.z, X[j + 2], p0);
            p1 = fmaf(l.w, X[j + 3], p1);
          }
          X[i] -= p0 + p1;
        }
      }
    } else {
#pragma unroll
      for (int i = 1; i < kC; ++i) {
        // four independent partial sums shorten the dependent FMA chain 4x
        float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
#pragma unroll
        for (int j = 0; j + 3 < i; j += 4) {
          const float4 l = *reinterpret_cast<const float4 *>(Lm + i * LLD + j);
          p0 = fmaf(l.x, X[j], p0);
          p1 = fmaf(l.y, X[j + 1], p1);
          p2 = fmaf(l.z, X[j + 2], p2);
          p3 = fmaf(l.w, X[j + 3], p3);
        }
#pragma unroll
        for (int j = i & ~3; j < i; ++j) p0 = fmaf(Lm[i * LLD + j], X[j], p0);
        X[i] = X[i] - ((p0 + p1) + (p2 + p3));
      }
    }
    float *dst = (col < D ? a.W : a.Ut) + ((size_t)h * nc + c) * kC * D + (col < D ? col : col - D);
#pragma unroll
    for (int i = 0; i < kC; ++i) dst[(size_t)i * D] = X[i];
  }
}

// ---------------------------------------------------------------- chunk_prep
// 16-byte asynchronous copy global -> shared; zero-filled when !valid.
GDN_DEV void cp_async16(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
GDN_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
GDN_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// One CTA (256 threads) per (chunk, value head). Tokens past T count as zero
// (k = q = v = 0, beta = 0, g = 0), which adds nothing to any product.
template <int D>
__global__ void __launch_bounds__(256) chunk_prep_kernel(PrefillArgs a) {
  constexpr int XLD = D + 4;  // padded row stride of K and Q (conflict-free fragment loads)
  extern __shared__ __align__(16) float sm[];
  float *KR = sm;                 // [kC][XLD]: k_i
  float *QR = KR + kC * XLD;      // [kC][XLD]: q_i
  float *Lm = QR + kC * XLD;      // [kC][kC]
  float *gam = Lm + kC * kC;      // [kC]
  float *bet = gam + kC;          // [kC]
  float *bek = bet + kC;          // [kC]: beta_i e^Gamma_i
  const int c = blockIdx.x, h = blockIdx.y;
  const int kh = h / (a.Hv / a.Hk);
  const int t0 = c * kC;
  const int nc = a.Tp / kC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // every load of the staging is issued before any of them is waited on
#pragma unroll
  for (int e = tid; e < kC * D / 4; e += 256) {
    const int i = (4 * e) / D, d = (4 * e) % D;
    const bool live = t0 + i < a.T;
    const float4 kv = live ? *reinterpret_cast<const float4 *>(a.kn + ((size_t)kh * a.Tp + t0 + i) * D + d)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 qv = live ? *reinterpret_cast<const float4 *>(a.qn + ((size_t)kh * a.Tp + t0 + i) * D + d)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4 *>(KR + i * XLD + d) = kv;
    *reinterpret_cast<float4 *>(QR + i * XLD + d) = qv;
  }
  if (tid < kC) {
    const bool live = t0 + tid < a.T;
    bet[tid] = live ? a.beta[(size_t)h * a.Tp + t0 + tid] : 0.0f;
    gam[tid] = live ? a.gl[(size_t)h * a.Tp + t0 + tid] : 0.0f;
  }
  __syncthreads();
  if (tid == 0) {  // cumulative log-decay, in token order, from shared memory
    float acc = 0.0f;
    for (int i = 0; i < kC; ++i) {
      acc += gam[i];
      gam[i] = acc;
    }
  }
  __syncthreads();
  if (tid < kC) a.Gam[((size_t)h * nc + c) * kC + tid] = gam[tid];

  // K K^T (warps 0..3) and Q K^T (warps 4..7) on split-TF32 warp MMA: warp ->
  // one 16-row band of the 64 x 64 product, all eight 8-column tiles
  {
    const int g = lane >> 2, t = lane & 3;
    const int m0 = 16 * (warp & 3);
    const bool isq = warp >= 4;
    const float *X = isq ? QR : KR;
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
#pragma unroll 2
    for (int k0 = 0; k0 < D; k0 += 8) {
      const float af[4] = {X[(m0 + g) * XLD + k0 + t], X[(m0 + g + 8) * XLD + k0 + t], X[(m0 + g) * XLD + k0 + t + 4],
                           X[(m0 + g + 8) * XLD + k0 + t + 4]};
      uint32_t ah[4], al[4];
      split4(af, ah, al);
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float bf[2] = {KR[(8 * n + g) * XLD + k0 + t], KR[(8 * n + g) * XLD + k0 + t + 4]};
        uint32_t bh[2], bl[2];
        split2(bf, bh, bl);
        mma3_split(acc[n], ah, al, bh, bl);
      }
    }
    float *Ag = a.Am + ((size_t)h * nc + c) * kC * kC;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // rows g and g + 8
        const int i = m0 + g + 8 * hh, j0 = 8 * n + 2 * t;
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + e;
          const float dec = j <= i ? expf(gam[i] - gam[j]) : 0.0f;
          const float x = acc[n][2 * hh + e];
          v[e] = isq ? dec * x : (j < i ? bet[i] * dec * x : 0.0f);
        }
        if (isq)
          *reinterpret_cast<float2 *>(Ag + (size_t)i * kC + j0) = make_float2(v[0], v[1]);
        else
          *reinterpret_cast<float2 *>(Lm + i * kC + j0) = make_float2(v[0], v[1]);
      }
    }
  }
  __syncthreads();
  // v of the chunk into Q's rows (Q is consumed), so that the substitution
  // below reads every right-hand side from shared memory
  float *VR = QR;
  for (int e = tid; e < kC * D / 4; e += 256) {
    const int i = (4 * e) / D, d = (4 * e) % D;
    cp_async16(VR + i * XLD + d, a.v + ((size_t)h * a.Tp + t0 + i) * D + d, t0 + i < a.T);
  }
  cp_async_commit();
  if (tid < kC) bek[tid] = bet[tid] * expf(gam[tid]);
  cp_async_wait_all();
  __syncthreads();

  chunk_solve<D, XLD>(a, KR, VR, Lm, bek, bet, h, c, nc, tid);
}

// ---------------------------------------------------------------- chunk_prep on tcgen05
// The products of chunk_prep_kernel<128> (Ut and Gamma in FP32; W, A and K^T
// as the tcgen05 scan's split FP16 operands x s = hi + lo -- W with a
// power-of-two scale per chunk from its largest |W|, A and K^T 2^14), with
// K K^T and Q K^T as one tcgen05 product in split FP16 of prep's q and k:
// they are L2-normalised (|k_i| <= 1, |q_i| <= d^-1/2), so the fixed scale
// 2^14 keeps every element below FP16's largest value and every lo part
// x - FP16(x) of an element larger than 2^-14 normal; x = hi + lo then
// carries 22 significant bits and
//   D = [K_hi; Q_hi] [K_hi; K_lo]^T + [K_lo; Q_lo] [K_hi; K_lo]^T
// (M = 128, N = 128, K = 128; FP32 accumulators in tensor memory) gives in its
// two column halves hi.hi + lo.hi and hi.lo + lo.lo of every k_i . k_j and
// q_i . k_j, which the epilogue adds and scales back exactly (2^-28).
// Operands are K-major with the 128-byte swizzle, loaded by TMA: per 64-wide
// d_k half a [128 rows][64 FP16] sub-tile of 16 KB. After the product the
// [K; Q] tiles hold L and Z = (I + L)^-1, while B' keeps k for the W part.
// 256 threads, two CTAs per SM.
constexpr int kPrepSub = 128 * 128;           // one [128 rows][64 FP16] sub-tile
constexpr int kPrepTile = 2 * kPrepSub;       // a 128 x 128 FP16 operand
constexpr int kPrepSmem = 1024 + 3 * kPrepTile + 4 * kC * 4 + 64;

GDN_DEV void mma_f16_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// byte offset of FP16 element (row, col) in a [rows][64 FP16] tile, 128-byte swizzle
GDN_DEV uint32_t sw16(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

__global__ void __launch_bounds__(256, 2)
    chunk_prep_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         PrefillArgs a) {
  constexpr int D = 128;
  constexpr int kLLD = kC + 4;  // row stride of L and of (I + L)^-1: a lane writes one row, 4-way bank spread
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t *Ahi = sm, *Alo = sm + kPrepTile, *Bp = sm + 2 * kPrepTile;
  // after the first product the [K; Q] tiles hold L, Z = (I + L)^-1, a 16 x 8
  // scratch per warp and Z as the split B operand [Z_hi; Z_lo] of the second
  // product (two [128 rows][32 FP32] sub-tiles, 1024-byte aligned: the first
  // over L once Z is complete, the second after the scratch); B' = [K_hi; K_lo]
  // stays for the W part
  float *Lm = reinterpret_cast<float *>(sm);
  float *Zm = Lm + kC * kLLD;
  float *Mt = Zm + kC * kLLD;
  uint8_t *Zb0 = sm, *Zb1 = sm + 38 * 1024;
  static_assert(38 * 1024 >= (2 * kC * kLLD + 8 * 128) * 4 && kC * kLLD * 4 >= 128 * 128 &&
                    38 * 1024 + 128 * 128 <= 2 * kPrepTile,
                "L, Z, the scratch and the B operand fit in the [K; Q] tiles");
  float *gam = reinterpret_cast<float *>(sm + 3 * kPrepTile);
  float *bet = gam + kC, *bek = bet + kC;
  uint64_t *done = reinterpret_cast<uint64_t *>(bek + kC);
  uint64_t *ld = done + 1;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(done + 2);
  __shared__ float wred[8], ured[8];
  const int c = blockIdx.x, h = blockIdx.y;
  const int kh = h / (a.Hv / a.Hk);
  const int t0 = c * kC;
  const int nc = a.Tp / kC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 8) wred[tid] = ured[tid] = 0.0f;

  if (tid < kC) {
    const bool live = t0 + tid < a.T;
    bet[tid] = live ? a.beta[(size_t)h * a.Tp + t0 + tid] : 0.0f;
    gam[tid] = live ? a.gl[(size_t)h * a.Tp + t0 + tid] : 0.0f;
  }
  if (tid == 0) {
    mbar_init(done, 1);
    mbar_init(ld, 1);
    fence_barrier_init();
    // the [K; Q] operand tiles (hi and lo) and B' = [K_hi; K_lo] by TMA from
    // prep's split q and k (x 2^14 = hi + lo, zero past T): per 64-wide d
    // half, rows 0..63 k and 64..127 q of the A tiles, rows 0..63 k_hi and
    // 64..127 k_lo of B'
    const int yq = kh * a.Tp + t0, ylo = a.Hk * a.Tp;
    mbar_arrive_expect_tx(ld, 12 * 64 * 128);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint8_t *ah = Ahi + q * kPrepSub, *al = Alo + q * kPrepSub, *bp = Bp + q * kPrepSub;
      tma_load_2d(ah, &tmK, 128 * q, yq, ld);
      tma_load_2d(ah + 64 * 128, &tmQ, 128 * q, yq, ld);
      tma_load_2d(al, &tmK, 128 * q, ylo + yq, ld);
      tma_load_2d(al + 64 * 128, &tmQ, 128 * q, ylo + yq, ld);
      tma_load_2d(bp, &tmK, 128 * q, yq, ld);
      tma_load_2d(bp + 64 * 128, &tmK, 128 * q, ylo + yq, ld);
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_holder, 256);
    tmem_relinquish();
  }
  // one CTA per key head writes the scan's K^T operand
  const bool write_q = h % (a.Hv / a.Hk) == 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const bool staged = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(ld, 0u) : 0, 0) != 0;
  if (!staged && tid == 0) flag_status(a.status, GDN_E_TIMEOUT);
  if (tid == 32 && staged) {  // the product: eight K = 16 steps, two MMAs each
    const uint32_t idesc = (1u << 4) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t o = (uint32_t)((k >> 2) * kPrepSub + (k & 3) * 32);
      const uint64_t bd = desc_sw128(smem_u32(Bp + o));
      mma_f16_ss(tmem, desc_sw128(smem_u32(Ahi + o)), bd, idesc, k ? 1u : 0u);
      mma_f16_ss(tmem, desc_sw128(smem_u32(Alo + o)), bd, idesc, 1u);
    }
    tc_commit(done);
  }
  if (tid == 0) {  // cumulative log-decay, in token order, while the product runs
    float acc = 0.0f;
    for (int i = 0; i < kC; ++i) {
      acc += gam[i];
      gam[i] = acc;
    }
  }
  __syncthreads();
  if (tid < kC) {
    a.Gam[((size_t)h * nc + c) * kC + tid] = gam[tid];
    bek[tid] = bet[tid] * expf(gam[tid]);
  }
  // one thread per warp waits; the warp follows it (collective TMEM loads)
  const int ok = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(done, 0u) : 0, 0);
  if (!ok && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
  tc_fence_after();
  // L (rows 0..63, k_i . k_j) and A (rows 64..127, q_i . k_j) from the
  // accumulator: thread = row 32 (warp & 3) + lane, columns 32 (warp >> 2) ..
  if (ok) {
    const int qt = warp & 3, hf = warp >> 2;
    const int m = 32 * qt + lane, j0 = 32 * hf;
    const uint32_t tb = tmem + ((uint32_t)(qt * 32) << 16);
    uint32_t d0[16], d1[16], e0[16], e1[16];
    tmem_ld16(tb + j0, d0);
    tmem_ld16(tb + j0 + 16, d1);
    tmem_ld16(tb + 64 + j0, e0);
    tmem_ld16(tb + 64 + j0 + 16, e1);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      v[k] = __uint_as_float(d0[k]) + __uint_as_float(e0[k]);
      v[16 + k] = __uint_as_float(d1[k]) + __uint_as_float(e1[k]);
    }
    if (m < kC) {
      const int i = m;
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        float l4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = j0 + k + e;
          l4[e] = j < i ? bet[i] * expf(gam[i] - gam[j]) * (v[k + e] * 0x1p-28f) : 0.0f;
        }
        *reinterpret_cast<float4 *>(Lm + i * kLLD + j0 + k) = make_float4(l4[0], l4[1], l4[2], l4[3]);
      }
    } else {
      // A 2^14 = e^(Gamma_i - Gamma_j) (q_i . k_j 2^28) 2^-14, split for the scan
      const int i = m - kC;
      uint16_t *Ag = a.As + ((size_t)h * a.Tp + t0 + i) * kC + j0;
      uint32_t hw[16], lw[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const int j = j0 + k;
        const float x0 = j <= i ? expf(gam[i] - gam[j]) * (v[k] * 0x1p-14f) : 0.0f;
        const float x1 = j + 1 <= i ? expf(gam[i] - gam[j + 1]) * (v[k + 1] * 0x1p-14f) : 0.0f;
        split_f16x2(x0, x1, hw[k / 2], lw[k / 2]);
      }
      uint4 *gh = reinterpret_cast<uint4 *>(Ag), *gl = reinterpret_cast<uint4 *>(Ag + (size_t)a.Hv * a.Tp * kC);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        gh[k] = make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2], hw[4 * k + 3]);
        gl[k] = make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // [W | Ut]^T = R^T Z^T, R = [diag(beta e^Gamma) K | diag(beta) v], one
  // 128-row part at a time: the part's R^T (lanes = d, columns = tokens j) as
  // hi and lo in TMEM columns 128..255 (the MMAs' A operand), the product
  // D[d][n] = R^T Z_hi^T | R^T Z_lo^T in columns 0..127, whose halves the
  // epilogue adds. Tokens past T are zero. A warp stages its lane quarter's
  // rows d for one half of the tokens.
  const int qt = warp & 3, hf = warp >> 2;
  const int d = 32 * qt + lane, j0 = 32 * hf;
  const uint32_t tl = tmem + ((uint32_t)(qt * 32) << 16);
  auto stage_r = [&](int part) {
    float x[32];
    if (part == 0) {
      // k from B' (k 2^14 = hi + lo, exact in FP32); its hi and lo are the
      // scan's K^T operand as they stand
      const uint8_t *bp = Bp + (d >> 6) * kPrepSub;
      uint32_t hw[16], lw[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const int j = j0 + k;
        const uint16_t h0 = *reinterpret_cast<const uint16_t *>(bp + sw16(j, d & 63));
        const uint16_t h1 = *reinterpret_cast<const uint16_t *>(bp + sw16(j + 1, d & 63));
        const uint16_t l0 = *reinterpret_cast<const uint16_t *>(bp + sw16(64 + j, d & 63));
        const uint16_t l1 = *reinterpret_cast<const uint16_t *>(bp + sw16(65 + j, d & 63));
        x[k] = (__half2float(__ushort_as_half(h0)) + __half2float(__ushort_as_half(l0))) * 0x1p-14f;
        x[k + 1] = (__half2float(__ushort_as_half(h1)) + __half2float(__ushort_as_half(l1))) * 0x1p-14f;
        hw[k / 2] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lw[k / 2] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
      if (write_q) {  // K^T 2^14 of the chunk, split, for the scan
        uint16_t *kt = a.KTs + (((size_t)kh * nc + c) * D + d) * kC + j0;
        uint4 *gh = reinterpret_cast<uint4 *>(kt), *gl = reinterpret_cast<uint4 *>(kt + (size_t)a.Hk * nc * D * kC);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          gh[k] = make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2], hw[4 * k + 3]);
          gl[k] = make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
        }
      }
    } else {
      // v of the chunk, bulk-copied into B' once k had been read
      const bool vin = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(ld, 1u) : 0, 0) != 0;
      if (!vin && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
      const float *vs = reinterpret_cast<const float *>(Bp);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int j = j0 + k;
        x[k] = vin && t0 + j < a.T ? vs[j * D + d] : 0.0f;
      }
    }
    uint32_t xh[32], xl[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) split_hi_lo(x[k] * (part == 0 ? bek[j0 + k] : bet[j0 + k]), xh[k], xl[k]);
    tmem_st32(tl + 128 + j0, xh);
    tmem_st32(tl + 192 + j0, xl);
    tmem_st_wait();
    tc_fence_before();
  };
  // Z = (I + L)^-1 by 16 x 16 blocks: the diagonal blocks D_b by forward
  // substitution (one column per thread, warps 0-1), then Z_ib = -D_i
  // sum_{k=b}^{i-1} L_ik Z_kb level by level (i - b = 1, 2, 3; warps 2-7), from
  // the equation (I + L) Z = I read block row by block row. Blocks above the
  // diagonal are zero and never written. The W part's R^T needs only k, so
  // each warp stages it while the other warps work on the inverse.
  if (tid < kC) {
    const int b = tid >> 4, cc = tid & 15, o = 16 * b;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = r == cc ? 1.0f : 0.0f;
#pragma unroll
      for (int s2 = 0; s2 < r; ++s2) acc = fmaf(-Lm[(o + r) * kLLD + o + s2], x[s2], acc);
      x[r] = acc;
      Zm[(o + r) * kLLD + o + cc] = acc;
    }
  } else {
    stage_r(0);
  }
  __syncthreads();
  if (warp < 2) {
    stage_r(0);
  } else {
    // a level's blocks on split-TF32 warp MMA: warp w (2..7) takes block
    // b = (w - 2) / 2, columns 8 ((w - 2) & 1) .. + 7 of it, while b < 4 - lv;
    // M = sum_k L_ik Z_kb (16 x 8) goes through the warp's scratch into B
    // fragments of -D_i M; a named barrier of warps 2-7 between levels
    const int g = lane >> 2, t = lane & 3, wl = warp - 2;
    float *Ms = Mt + warp * 128;
#pragma unroll 1
    for (int lv = 1; lv < 4; ++lv) {
      const int b = wl >> 1;
      if (b < 4 - lv) {
        const int i = b + lv, cb = 16 * b + 8 * (wl & 1), ri = 16 * i;
        float dacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int kc = 16 * b; kc < ri; kc += 8) {
          const float af[4] = {Lm[(ri + g) * kLLD + kc + t], Lm[(ri + g + 8) * kLLD + kc + t],
                               Lm[(ri + g) * kLLD + kc + t + 4], Lm[(ri + g + 8) * kLLD + kc + t + 4]};
          const float bf[2] = {Zm[(kc + t) * kLLD + cb + g], Zm[(kc + t + 4) * kLLD + cb + g]};
          mma3(dacc, af, bf);
        }
        Ms[g * 8 + 2 * t] = dacc[0];
        Ms[g * 8 + 2 * t + 1] = dacc[1];
        Ms[(g + 8) * 8 + 2 * t] = dacc[2];
        Ms[(g + 8) * 8 + 2 * t + 1] = dacc[3];
        __syncwarp();
        float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int s2 = 0; s2 < 16; s2 += 8) {
          const float af[4] = {Zm[(ri + g) * kLLD + ri + s2 + t], Zm[(ri + g + 8) * kLLD + ri + s2 + t],
                               Zm[(ri + g) * kLLD + ri + s2 + t + 4], Zm[(ri + g + 8) * kLLD + ri + s2 + t + 4]};
          const float bf[2] = {Ms[(s2 + t) * 8 + g], Ms[(s2 + t + 4) * 8 + g]};
          mma3(z, af, bf);
        }
        Zm[(ri + g) * kLLD + cb + 2 * t] = -z[0];
        Zm[(ri + g) * kLLD + cb + 2 * t + 1] = -z[1];
        Zm[(ri + g + 8) * kLLD + cb + 2 * t] = -z[2];
        Zm[(ri + g + 8) * kLLD + cb + 2 * t + 1] = -z[3];
        __syncwarp();
      }
      asm volatile("bar.sync 1, 192;" ::: "memory");
    }
  }
  __syncthreads();
  if (tid == 0) {  // k has been read from B': the chunk's v rows (32 KB) over it
    fence_async_shared();
    mbar_arrive_expect_tx(ld, kC * D * 4);
    bulk_g2s(Bp, a.v + ((size_t)h * a.Tp + t0) * D, kC * D * 4, ld);
  }
  // Z as the B operand [Z_hi; Z_lo] (N = 128 rows: row n < 64 is Z_hi[n], row
  // 64 + n is Z_lo[n]; K = the 64 tokens j in two 32-wide swizzled sub-tiles)
  for (int e = tid; e < kC * kC; e += 256) {
    const int n = e >> 6, j = e & 63;
    uint32_t zh, zl;
    split_hi_lo((j >> 4) > (n >> 4) ? 0.0f : Zm[n * kLLD + j], zh, zl);
    uint8_t *sub = (j >> 5) ? Zb1 : Zb0;
    *reinterpret_cast<uint32_t *>(sub + sw_off(n, j & 31)) = zh;
    *reinterpret_cast<uint32_t *>(sub + sw_off(64 + n, j & 31)) = zl;
  }
  fence_async_shared();
  tc_fence_before();
  __syncthreads();
  {
    const uint32_t idesc = idesc_tf32(128);
    auto issue = [&]() {  // D = R^T [Z_hi; Z_lo]^T: eight K = 8 steps, A lo then A hi
      if (tid == 32) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = desc_sw128(smem_u32((kk >> 2) ? Zb1 : Zb0)) + 2 * (kk & 3);
          mma_tf32_ts(tmem, tmem + 192 + 8 * kk, bd, idesc, kk ? 1u : 0u);
          mma_tf32_ts(tmem, tmem + 128 + 8 * kk, bd, idesc, 1u);
        }
        tc_commit(done);
      }
    };
    // this thread's row d of the product, tokens j0 .. j0 + 31 (the halves added)
    auto read_acc = [&](float (&out)[32]) {
      uint32_t p0[16], p1[16], q0[16], q1[16];
      tmem_ld16(tl + j0, p0);
      tmem_ld16(tl + j0 + 16, p1);
      tmem_ld16(tl + 64 + j0, q0);
      tmem_ld16(tl + 64 + j0 + 16, q1);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        out[k] = __uint_as_float(p0[k]) + __uint_as_float(q0[k]);
        out[16 + k] = __uint_as_float(p1[k]) + __uint_as_float(q1[k]);
      }
    };
    auto warp_absmax = [&](const float (&v)[32]) -> float {
      float mx = 0.0f;
#pragma unroll
      for (int k = 0; k < 32; ++k) mx = fmaxf(mx, fabsf(v[k]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      return mx;
    };
    // the W part
    issue();
    const int okw = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(done, 1u) : 0, 0);
    if (!okw && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
    tc_fence_after();
    float wv[32];  // W: tokens j0 + k, kept until the chunk's largest |W| is known
    if (okw) read_acc(wv);
    // the U part's R^T over the W part's (whose product has completed)
    stage_r(1);
    if (okw) {
      const float mx = warp_absmax(wv);
      if (lane == 0) wred[warp] = mx;
    }
    __syncthreads();  // every warp has read the W product and staged its U operand
    issue();
    if (okw) {  // W s = hi + lo, s from the chunk's largest |W|, while the U product runs
      float m = wred[0];
#pragma unroll
      for (int w = 1; w < 8; ++w) m = fmaxf(m, wred[w]);
      const float sw = fp16_scale_for(m);
      if (tid == 0) a.Wsc[(size_t)h * nc + c] = sw;
      uint16_t *wh = a.Ws + ((size_t)h * a.Tp + t0 + j0) * D + d, *wl = wh + (size_t)a.Hv * a.Tp * D;
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        uint32_t hi, lo;
        split_f16x2(wv[k] * sw, wv[k + 1] * sw, hi, lo);
        wh[(size_t)k * D] = (uint16_t)hi;
        wh[(size_t)(k + 1) * D] = (uint16_t)(hi >> 16);
        wl[(size_t)k * D] = (uint16_t)lo;
        wl[(size_t)(k + 1) * D] = (uint16_t)(lo >> 16);
      }
    }
    // the U part: U~ in FP32 and the chunk's largest |U~| (the scan's bound on |U|)
    const int oku = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(done, 0u) : 0, 0);
    if (!oku && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
    tc_fence_after();
    if (oku) {
      float uv[32];
      read_acc(uv);
      float *dst = a.Ut + (((size_t)h * nc + c) * kC + j0) * D + d;
#pragma unroll
      for (int k = 0; k < 32; ++k) dst[(size_t)k * D] = uv[k];
      const float mx = warp_absmax(uv);
      if (lane == 0) ured[warp] = mx;
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      float m = ured[0];
      for (int w = 1; w < 8; ++w) m = fmaxf(m, ured[w]);
      a.Umax[(size_t)h * nc + c] = m;
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------- chunk_scan

// One CTA (512 threads = 16 warps) per (value head, 32 rows of d_v). The state
// slice S[32][D] stays in shared memory across all chunks; lane = row r of the
// slice in every product.
template <int D>
__global__ void __launch_bounds__(512) chunk_scan_kernel(PrefillArgs a) {
  constexpr int R = 32;
  constexpr int NSL = D / R;
  constexpr int SLD = D + 1;  // padded row stride of S (conflict-free lane = row)
  constexpr int RLD = R + 1;
  extern __shared__ __align__(16) float sm[];
  float *Ws = sm;                    // [kC][D]
  float *Qs = Ws + kC * D;           // [kC][D]
  float *Ks = Qs + kC * D;           // [kC][D]
  float *Us = Ks + kC * D;           // [kC][R]  Ut slice, then U
  float *As = Us + kC * R;           // [kC][kC]
  float *Gs = As + kC * kC;          // [kC]
  float *S = Gs + kC;                // [R][SLD]
  float *P = S + R * SLD;            // [2 kC][RLD]: W S0^T then Q S0^T
  float *Cf = P + 2 * kC * RLD;      // [kC][RLD]: e^(Gamma_64 - Gamma_j) u_j

  const int h = blockIdx.x / NSL, r0 = (blockIdx.x % NSL) * R;
  const int kh = h / (a.Hv / a.Hk);
  const int nc = a.Tp / kC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int e = tid; e < R * D; e += blockDim.x) {
    const int r = e / D, d = e % D;
    S[r * SLD + d] = state_load(a.ssm, a.state_bf16, ((size_t)h * D + r0 + r) * D + d);
  }
  auto load_wq = [&](int c) {
    const float *w = a.W + ((size_t)h * nc + c) * kC * D;
    const float *q = a.qn + ((size_t)kh * a.Tp + (size_t)c * kC) * D;
    for (int e = tid; e < kC * D / 4; e += blockDim.x) {
      const int i = (4 * e) / D;
      cp_async16(Ws + 4 * e, w + 4 * e, true);
      cp_async16(Qs + 4 * e, q + 4 * e, c * kC + i < a.T);
    }
  };
  auto load_rest = [&](int c) {
    const float *k = a.kn + ((size_t)kh * a.Tp + (size_t)c * kC) * D;
    for (int e = tid; e < kC * D / 4; e += blockDim.x) {
      const int i = (4 * e) / D;
      cp_async16(Ks + 4 * e, k + 4 * e, c * kC + i < a.T);
    }
    const float *u = a.Ut + ((size_t)h * nc + c) * kC * D + r0;
    for (int e = tid; e < kC * R / 4; e += blockDim.x) {
      const int i = (4 * e) / R, r = (4 * e) % R;
      cp_async16(Us + 4 * e, u + (size_t)i * D + r, true);
    }
    const float *am = a.Am + ((size_t)h * nc + c) * kC * kC;
    for (int e = tid; e < kC * kC / 4; e += blockDim.x) cp_async16(As + 4 * e, am + 4 * e, true);
    if (tid < kC / 4) cp_async16(Gs + 4 * tid, a.Gam + ((size_t)h * nc + c) * kC + 4 * tid, true);
  };
  load_wq(0);
  load_rest(0);
  cp_async_commit();

  for (int c = 0; c < nc; ++c) {
    cp_async_wait_all();
    __syncthreads();
    // P = [W; Q] S0^T: warp w -> rows 8w..8w+7 of [W; Q], lane -> slice row r
    {
      const float *X = warp < 8 ? Ws + (8 * warp) * D : Qs + (8 * (warp - 8)) * D;
      float acc[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[x] = 0.0f;
#pragma unroll 4
      for (int d = 0; d < D; d += 4) {
        const float s0 = S[lane * SLD + d], s1 = S[lane * SLD + d + 1];
        const float s2 = S[lane * SLD + d + 2], s3 = S[lane * SLD + d + 3];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 xv = *reinterpret_cast<const float4 *>(X + x * D + d);
          acc[x] = fmaf(xv.x, s0, fmaf(xv.y, s1, fmaf(xv.z, s2, fmaf(xv.w, s3, acc[x]))));
        }
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) P[(8 * warp + x) * RLD + lane] = acc[x];
    }
    __syncthreads();
    if (c + 1 < nc) {  // W and Q of this chunk are consumed
      load_wq(c + 1);
      cp_async_commit();
    }
    // U = Ut - W S0^T (in place in Us), and the state-update coefficients
    const float gC = Gs[kC - 1];
    for (int e = tid; e < kC * R; e += blockDim.x) {
      const int i = e / R, r = e % R;
      const float u = Us[i * R + r] - P[i * RLD + r];
      Us[i * R + r] = u;
      Cf[i * RLD + r] = expf(gC - Gs[i]) * u;
    }
    __syncthreads();
    // O_i = e^Gamma_i (Q S0^T)_i + sum_{j<=i} A_ij u_j : warp w -> rows 4w..4w+3
    {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int i = 4 * warp + x;
        float acc0 = expf(Gs[i]) * P[(kC + i) * RLD + lane], acc1 = 0.0f;
        int j = 0;
        for (; j + 1 <= i; j += 2) {
          acc0 = fmaf(As[i * kC + j], Us[j * R + lane], acc0);
          acc1 = fmaf(As[i * kC + j + 1], Us[(j + 1) * R + lane], acc1);
        }
        if (j == i) acc0 = fmaf(As[i * kC + j], Us[j * R + lane], acc0);
        const int t = c * kC + i;
        if (t < a.T) a.o[((size_t)t * a.Hv + h) * D + r0 + lane] = acc0 + acc1;
      }
    }
    // S <- e^Gamma_64 S + sum_j coef_j[r] k_j : warp w -> columns 8w..8w+7
    if (warp < D / 8) {
      const float dC = expf(gC);
      float sv[8];
#pragma unroll
      for (int y = 0; y < 8; ++y) sv[y] = dC * S[lane * SLD + 8 * warp + y];
#pragma unroll 4
      for (int j = 0; j < kC; ++j) {
        const float cf = Cf[j * RLD + lane];
        const float4 k0 = *reinterpret_cast<const float4 *>(Ks + j * D + 8 * warp);
        const float4 k1 = *reinterpret_cast<const float4 *>(Ks + j * D + 8 * warp + 4);
        sv[0] = fmaf(cf, k0.x, sv[0]);
        sv[1] = fmaf(cf, k0.y, sv[1]);
        sv[2] = fmaf(cf, k0.z, sv[2]);
        sv[3] = fmaf(cf, k0.w, sv[3]);
        sv[4] = fmaf(cf, k1.x, sv[4]);
        sv[5] = fmaf(cf, k1.y, sv[5]);
        sv[6] = fmaf(cf, k1.z, sv[6]);
        sv[7] = fmaf(cf, k1.w, sv[7]);
      }
#pragma unroll
      for (int y = 0; y < 8; ++y) S[lane * SLD + 8 * warp + y] = sv[y];
    }
    __syncthreads();
    if (c + 1 < nc) {  // K, U, A and Gamma of this chunk are consumed
      load_rest(c + 1);
      cp_async_commit();
    }
  }
  cp_async_wait_all();
  __syncthreads();
  for (int e = tid; e < R * D; e += blockDim.x) {
    const int r = e / D, d = e % D;
    state_store(a.ssm, a.state_bf16, ((size_t)h * D + r0 + r) * D + d, S[r * SLD + d]);
  }
}

// ---------------------------------------------------------------- chunk_scan on tensor cores
// The same chunk recurrence as chunk_scan_kernel for D = 128, with its three
// products on warp-level MMA (mma.sync m16n8k8, TF32 in, FP32 accumulation)
// in the split form x = hi + lo (hi = TF32(x), lo = TF32(x - hi)) and
// a.b ~ hi.hi + hi.lo + lo.hi: about 21 of FP32's 24 mantissa bits per
// product, so chunked prefill stays as precise as the per-token recurrence
// (bloomery issue #565, §10, splits FP32 operands into BF16 parts for the same
// reason); lo terms added first.
//   P = [W; Q] S^T          (128 x 32, K = 128)
//   O = diag(e^Gamma) Pq + A U   (64 x 32, K = 64; A is zero above the diagonal)
//   S <- e^Gamma_64 S + Cf^T K   (32 x 128, K = 64)
// Shared tiles are padded so every fragment load is conflict-free. The state
// slice and the update coefficients are kept pre-split (hi and lo parts next
// to the FP32 state), since eight warps read each of their fragments.
__global__ void __launch_bounds__(512) chunk_scan_tc_kernel(PrefillArgs a) {
  constexpr int D = 128, R = 32, NSL = D / R;
  constexpr int XLD = D + 4;   // W, Q rows
  constexpr int KLD = D + 8;   // K rows (read with the token index across lanes)
  constexpr int SLD = D + 4;   // S rows
  constexpr int ULD = R + 8;   // U, Cf rows
  constexpr int ALD = kC + 4;  // A rows
  constexpr int PLD = R + 1;   // P rows
  extern __shared__ __align__(16) float sm[];
  float *Ws = sm;                    // [kC][XLD]
  float *Qs = Ws + kC * XLD;         // [kC][XLD]
  float *Ks = Qs + kC * XLD;         // [kC][KLD]
  float *Us = Ks + kC * KLD;         // [kC][ULD]  Ut slice, then U
  float *As = Us + kC * ULD;         // [kC][ALD]
  float *Gs = As + kC * ALD;         // [kC]
  float *S = Gs + kC;                // [R][SLD]
  float *P = S + R * SLD;            // [2 kC][PLD]: W S0^T then Q S0^T
  uint32_t *Cfh = reinterpret_cast<uint32_t *>(P + 2 * kC * PLD);  // [kC][ULD]: e^(Gamma_64 - Gamma_j) u_j, hi
  uint32_t *Cfl = Cfh + kC * ULD;                                   // ... lo
  uint32_t *Sh = Cfl + kC * ULD;                                    // [R][SLD]: S, hi
  uint32_t *Sl = Sh + R * SLD;                                      // ... lo

  const int h = blockIdx.x / NSL, r0 = (blockIdx.x % NSL) * R;
  const int kh = h / (a.Hv / a.Hk);
  const int nc = a.Tp / kC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  for (int e = tid; e < R * D; e += blockDim.x) {
    const int r = e / D, d = e % D;
    const float v = state_load(a.ssm, a.state_bf16, ((size_t)h * D + r0 + r) * D + d);
    S[r * SLD + d] = v;
    split_tf32(v, Sh[r * SLD + d], Sl[r * SLD + d]);
  }
  auto load_wq = [&](int c) {
    const float *w = a.W + ((size_t)h * nc + c) * kC * D;
    const float *q = a.qn + ((size_t)kh * a.Tp + (size_t)c * kC) * D;
    for (int e = tid; e < kC * D / 4; e += blockDim.x) {
      const int i = (4 * e) / D, d = (4 * e) % D;
      cp_async16(Ws + i * XLD + d, w + 4 * e, true);
      cp_async16(Qs + i * XLD + d, q + 4 * e, c * kC + i < a.T);
    }
  };
  auto load_rest = [&](int c) {
    const float *k = a.kn + ((size_t)kh * a.Tp + (size_t)c * kC) * D;
    for (int e = tid; e < kC * D / 4; e += blockDim.x) {
      const int i = (4 * e) / D, d = (4 * e) % D;
      cp_async16(Ks + i * KLD + d, k + 4 * e, c * kC + i < a.T);
    }
    const float *u = a.Ut + ((size_t)h * nc + c) * kC * D + r0;
    for (int e = tid; e < kC * R / 4; e += blockDim.x) {
      const int i = (4 * e) / R, r = (4 * e) % R;
      cp_async16(Us + i * ULD + r, u + (size_t)i * D + r, true);
    }
    const float *am = a.Am + ((size_t)h * nc + c) * kC * kC;
    for (int e = tid; e < kC * kC / 4; e += blockDim.x) {
      const int i = (4 * e) / kC, j = (4 * e) % kC;
      cp_async16(As + i * ALD + j, am + 4 * e, true);
    }
    if (tid < kC / 4) cp_async16(Gs + 4 * tid, a.Gam + ((size_t)h * nc + c) * kC + 4 * tid, true);
  };
  load_wq(0);
  load_rest(0);
  cp_async_commit();

  for (int c = 0; c < nc; ++c) {
    cp_async_wait_all();
    __syncthreads();
    // ---- P = [W; Q] S0^T: warp -> one 16-row tile of [W; Q], two 8-column tiles
    {
      const int m0 = 16 * (warp >> 1), n0 = 16 * (warp & 1);
      const float *X = m0 < kC ? Ws + m0 * XLD : Qs + (m0 - kC) * XLD;
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int k0 = 0; k0 < D; k0 += 8) {
        const float af[4] = {X[g * XLD + k0 + t], X[(g + 8) * XLD + k0 + t], X[g * XLD + k0 + t + 4],
                             X[(g + 8) * XLD + k0 + t + 4]};
        uint32_t ah[4], al[4];
        split4(af, ah, al);
        const uint32_t b0h[2] = {Sh[(n0 + g) * SLD + k0 + t], Sh[(n0 + g) * SLD + k0 + t + 4]};
        const uint32_t b0l[2] = {Sl[(n0 + g) * SLD + k0 + t], Sl[(n0 + g) * SLD + k0 + t + 4]};
        const uint32_t b1h[2] = {Sh[(n0 + 8 + g) * SLD + k0 + t], Sh[(n0 + 8 + g) * SLD + k0 + t + 4]};
        const uint32_t b1l[2] = {Sl[(n0 + 8 + g) * SLD + k0 + t], Sl[(n0 + 8 + g) * SLD + k0 + t + 4]};
        mma3_split(d0, ah, al, b0h, b0l);
        mma3_split(d1, ah, al, b1h, b1l);
      }
      P[(m0 + g) * PLD + n0 + 2 * t] = d0[0];
      P[(m0 + g) * PLD + n0 + 2 * t + 1] = d0[1];
      P[(m0 + g + 8) * PLD + n0 + 2 * t] = d0[2];
      P[(m0 + g + 8) * PLD + n0 + 2 * t + 1] = d0[3];
      P[(m0 + g) * PLD + n0 + 8 + 2 * t] = d1[0];
      P[(m0 + g) * PLD + n0 + 8 + 2 * t + 1] = d1[1];
      P[(m0 + g + 8) * PLD + n0 + 8 + 2 * t] = d1[2];
      P[(m0 + g + 8) * PLD + n0 + 8 + 2 * t + 1] = d1[3];
    }
    __syncthreads();
    if (c + 1 < nc) {  // W and Q of this chunk are consumed
      load_wq(c + 1);
      cp_async_commit();
    }
    // ---- U = Ut - W S0^T (in place), and the state-update coefficients
    const float gC = Gs[kC - 1];
    for (int e = tid; e < kC * R; e += blockDim.x) {
      const int i = e / R, r = e % R;
      const float u = Us[i * ULD + r] - P[i * PLD + r];
      Us[i * ULD + r] = u;
      split_tf32(expf(gC - Gs[i]) * u, Cfh[i * ULD + r], Cfl[i * ULD + r]);
    }
    __syncthreads();
    // ---- O = diag(e^Gamma) (Q S0^T) + A U: warp -> one 16 x 8 tile
    {
      const int m0 = 16 * (warp >> 2), n0 = 8 * (warp & 3);
      const float e0 = expf(Gs[m0 + g]), e1 = expf(Gs[m0 + g + 8]);
      float d[4] = {e0 * P[(kC + m0 + g) * PLD + n0 + 2 * t], e0 * P[(kC + m0 + g) * PLD + n0 + 2 * t + 1],
                    e1 * P[(kC + m0 + g + 8) * PLD + n0 + 2 * t], e1 * P[(kC + m0 + g + 8) * PLD + n0 + 2 * t + 1]};
      for (int k0 = 0; k0 < m0 + 16; k0 += 8) {  // A is zero above the diagonal
        const float af[4] = {As[(m0 + g) * ALD + k0 + t], As[(m0 + g + 8) * ALD + k0 + t],
                             As[(m0 + g) * ALD + k0 + t + 4], As[(m0 + g + 8) * ALD + k0 + t + 4]};
        const float bf[2] = {Us[(k0 + t) * ULD + n0 + g], Us[(k0 + t + 4) * ULD + n0 + g]};
        mma3(d, af, bf);
      }
      const int i0 = c * kC + m0 + g, i1 = i0 + 8;
      if (i0 < a.T) {
        a.o[((size_t)i0 * a.Hv + h) * D + r0 + n0 + 2 * t] = d[0];
        a.o[((size_t)i0 * a.Hv + h) * D + r0 + n0 + 2 * t + 1] = d[1];
      }
      if (i1 < a.T) {
        a.o[((size_t)i1 * a.Hv + h) * D + r0 + n0 + 2 * t] = d[2];
        a.o[((size_t)i1 * a.Hv + h) * D + r0 + n0 + 2 * t + 1] = d[3];
      }
    }
    // ---- S <- e^Gamma_64 S + Cf^T K: warp -> one 16-row tile of S, two 8-column tiles
    {
      const float dC = expf(gC);
      const int m0 = 16 * (warp >> 3), n0 = 16 * (warp & 7);
      float d0[4] = {dC * S[(m0 + g) * SLD + n0 + 2 * t], dC * S[(m0 + g) * SLD + n0 + 2 * t + 1],
                     dC * S[(m0 + g + 8) * SLD + n0 + 2 * t], dC * S[(m0 + g + 8) * SLD + n0 + 2 * t + 1]};
      float d1[4] = {dC * S[(m0 + g) * SLD + n0 + 8 + 2 * t], dC * S[(m0 + g) * SLD + n0 + 8 + 2 * t + 1],
                     dC * S[(m0 + g + 8) * SLD + n0 + 8 + 2 * t], dC * S[(m0 + g + 8) * SLD + n0 + 8 + 2 * t + 1]};
#pragma unroll 4
      for (int k0 = 0; k0 < kC; k0 += 8) {
        const uint32_t ah[4] = {Cfh[(k0 + t) * ULD + m0 + g], Cfh[(k0 + t) * ULD + m0 + g + 8],
                                Cfh[(k0 + t + 4) * ULD + m0 + g], Cfh[(k0 + t + 4) * ULD + m0 + g + 8]};
        const uint32_t al[4] = {Cfl[(k0 + t) * ULD + m0 + g], Cfl[(k0 + t) * ULD + m0 + g + 8],
                                Cfl[(k0 + t + 4) * ULD + m0 + g], Cfl[(k0 + t + 4) * ULD + m0 + g + 8]};
        const float b0[2] = {Ks[(k0 + t) * KLD + n0 + g], Ks[(k0 + t + 4) * KLD + n0 + g]};
        const float b1[2] = {Ks[(k0 + t) * KLD + n0 + 8 + g], Ks[(k0 + t + 4) * KLD + n0 + 8 + g]};
        uint32_t bh[2], bl[2];
        split2(b0, bh, bl);
        mma3_split(d0, ah, al, bh, bl);
        split2(b1, bh, bl);
        mma3_split(d1, ah, al, bh, bl);
      }
      const int sidx[8] = {(m0 + g) * SLD + n0 + 2 * t,         (m0 + g) * SLD + n0 + 2 * t + 1,
                           (m0 + g + 8) * SLD + n0 + 2 * t,     (m0 + g + 8) * SLD + n0 + 2 * t + 1,
                           (m0 + g) * SLD + n0 + 8 + 2 * t,     (m0 + g) * SLD + n0 + 8 + 2 * t + 1,
                           (m0 + g + 8) * SLD + n0 + 8 + 2 * t, (m0 + g + 8) * SLD + n0 + 8 + 2 * t + 1};
      const float sv[8] = {d0[0], d0[1], d0[2], d0[3], d1[0], d1[1], d1[2], d1[3]};
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        S[sidx[x]] = sv[x];
        split_tf32(sv[x], Sh[sidx[x]], Sl[sidx[x]]);
      }
    }
    __syncthreads();
    if (c + 1 < nc) {  // K, U, A and Gamma of this chunk are consumed
      load_rest(c + 1);
      cp_async_commit();
    }
  }
  cp_async_wait_all();
  __syncthreads();
  for (int e = tid; e < R * D; e += blockDim.x) {
    const int r = e / D, d = e % D;
    state_store(a.ssm, a.state_bf16, ((size_t)h * D + r0 + r) * D + d, S[r * SLD + d]);
  }
}

// one CTA per token; thread i owns 16-block i of y (head i / (D/16))
__global__ void __launch_bounds__(256, 5) gnorm_kernel(PrefillArgs a) {
  const int t = blockIdx.x;
  const int D = a.D, vd = a.Hv * D;
  const int nblk = vd / 16;
  const int i = min((int)threadIdx.x, nblk - 1);  // block index within the token; spare lanes
                                                   // shadow the last block and store nothing
  const int per_head = D / 16;          // threads per head: 2, 4 or 8 (a power of two)
  const int h = i / per_head, e0 = (i % per_head) * 16;
  const float *op = a.o + ((size_t)t * a.Hv + h) * D + e0;
  const uint16_t *zp = a.proj + (size_t)t * a.ld + 2 * a.Hk * D + vd + h * D + e0;
  // o and the z bits first (z kept packed); the norm weight is read at use
  float y[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // o rows are 64-byte aligned per 16-block
    const float4 o4 = reinterpret_cast<const float4 *>(op)[q];
    y[4 * q] = o4.x; y[4 * q + 1] = o4.y; y[4 * q + 2] = o4.z; y[4 * q + 3] = o4.w;
  }
  uint32_t zw[8];
  if (a.ld % 8 == 0) {  // z rows 16-byte aligned
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 z4 = reinterpret_cast<const uint4 *>(zp)[q];
      zw[4 * q] = z4.x; zw[4 * q + 1] = z4.y; zw[4 * q + 2] = z4.z; zw[4 * q + 3] = z4.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) zw[k] = uint32_t(zp[2 * k]) | (uint32_t(zp[2 * k + 1]) << 16);
  }
  float p = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) p = fmaf(y[k], y[k], p);
  // the head's 16-element group sums added in group order (as in decode)
  const int first = (threadIdx.x & 31) & ~(per_head - 1);
  float tot = 0.0f;
  for (int m = 0; m < per_head; ++m) tot += __shfl_sync(0xffffffffu, p, first + m);
  p = tot;
  const float rstd = 1.0f / sqrtf(p / (float)D + a.rms_eps);
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // the norm weight is 64-byte aligned per 16-block
    const float4 w4 = reinterpret_cast<const float4 *>(a.norm_w + e0)[q];
    const float nw[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = 4 * q + k;
      const float zv = __uint_as_float((j & 1) ? (zw[j >> 1] & 0xFFFF0000u) : (zw[j >> 1] << 16));
      y[j] = y[j] * rstd * nw[k] * siluf_(zv);
    }
  }
  uint32_t lo, hi, s;
  const bool ok = quant_block16(y, a.ts_out, inv6ts_of(a.ts_out), lo, hi, s);
  if ((int)threadIdx.x >= nblk) return;
  if (!ok) flag_status(a.status, GDN_E_NONFINITE);
  const size_t b0 = (size_t)t * vd + h * D + e0;
  *reinterpret_cast<uint2 *>(a.y_codes + (b0 >> 1)) = make_uint2(lo, hi);
  a.y_scales[a.y_sf_tiled ? sf_tiled_offset(t, (h * D + e0) >> 4, vd >> 4) : (b0 >> 4)] = uint8_t(s);
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

template <int D>
cudaError_t launch_chunks(const PrefillArgs &a, const LaunchCtx &lc) {
  const size_t sm_prep = (size_t)(2 * kC * (D + 4) + kC * kC + 3 * kC) * sizeof(float);
  const size_t sm_scan =
      (size_t)(3 * kC * D + kC * 32 + kC * kC + kC + 32 * (D + 1) + 2 * kC * 33 + kC * 33) * sizeof(float);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_prep);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(chunk_scan_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_scan);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int nc = a.Tp / kC;
  if (D == 128 && a.scan_tc == 2) {  // both chunk stages on tcgen05
    if (!a.Qs || !a.Ks || !a.Ws || !a.As || !a.KTs || !a.Wsc || !a.Umax) return cudaErrorInvalidValue;
    static bool configured_p = false;
    if (!configured_p) {
      cudaError_t e = cudaFuncSetAttribute(chunk_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
      if (e != cudaSuccess) return e;
      configured_p = true;
    }
    // prep's split q and k as 2-D byte tensors [2 Hk Tp][2 D]; 64-row boxes of 128 bytes
    CUtensorMap mQ, mK;
    if (!make_map(&mQ, a.Qs, 2ull * a.Hk * a.Tp, (uint64_t)D * 2, kC, 128, true) ||
        !make_map(&mK, a.Ks, 2ull * a.Hk * a.Tp, (uint64_t)D * 2, kC, 128, true))
      return cudaErrorInvalidValue;
    chunk_prep_tc_kernel<<<dim3(nc, a.Hv), 256, kPrepSmem, lc.stream>>>(mQ, mK, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_chunk_scan_umma(a, lc.stream);
  }
  chunk_prep_kernel<D><<<dim3(nc, a.Hv), 256, sm_prep, lc.stream>>>(a);
  if (D == 128 && a.scan_tc) {
    const size_t sm_tc = (size_t)(2 * kC * (D + 4) + kC * (D + 8) + kC * 40 + kC * (kC + 4) + kC + 32 * (D + 4) + 2 * kC * 33 +
                                  2 * kC * 40 + 2 * 32 * (D + 4)) * sizeof(float);
    static bool configured_tc = false;
    if (!configured_tc) {
      cudaError_t e = cudaFuncSetAttribute(chunk_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_tc);
      if (e != cudaSuccess) return e;
      configured_tc = true;
    }
    chunk_scan_tc_kernel<<<a.Hv * (D / 32), 512, sm_tc, lc.stream>>>(a);
  } else {
    chunk_scan_kernel<D><<<a.Hv * (D / 32), 512, sm_scan, lc.stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

// The stages between the projections (run by the caller) and the out
// projection. `tmp` holds (K-1)*C BF16 values.
cudaError_t launch_prefill_mix(const PrefillArgs &a, uint16_t *tmp, const LaunchCtx &lc) {
  const dim3 pg((a.T + kPrepTT - 1) / kPrepTT, 2 * a.Hk + a.Hv + 1);
  switch (a.D) {
    case 128: prep_kernel<128><<<pg, 128, 0, lc.stream>>>(a); break;
    case 64: prep_kernel<64><<<pg, 128, 0, lc.stream>>>(a); break;
    case 32: prep_kernel<32><<<pg, 128, 0, lc.stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // conv state tail is computed from the old state before anything overwrites it
  const int n = (a.Kc - 1) * a.C;
  conv_tail_kernel<<<(n + 255) / 256, 256, 0, lc.stream>>>(a, tmp);
  switch (a.D) {
    case 128: e = launch_chunks<128>(a, lc); break;
    case 64: e = launch_chunks<64>(a, lc); break;
    case 32: e = launch_chunks<32>(a, lc); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  const int gthreads = ((a.Hv * a.D / 16) + 31) / 32 * 32;
  gnorm_kernel<<<a.T, gthreads, 0, lc.stream>>>(a);
  copy_u16_kernel<<<(n + 255) / 256, 256, 0, lc.stream>>>(a.conv_state, tmp, n);
  return cudaGetLastError();
}

}  // namespace gdn
