// In-projection and token mixing of one decode step in one kernel, for up to
// eight rows: NVFP4 quantisation of x, the W4A4 q|k|v|z|b|a rows a key head
// needs, depthwise causal conv + SiLU, q/k L2 norm, the beta/g gates, the gated
// delta rule on the recurrent state, the z-gated RMSNorm and the NVFP4
// quantisation of its output. The out-projection follows as its own kernel:
// each of its rows reads every head's output.
//
// Work split: a thread-block cluster of 8 CTAs per key head. CTA `rank` owns
//  * 16 of the key head's 128 q channels and 16 of its k channels;
//  * R = 128 * G / 8 d_v rows of value head h = kh * G + rank / (8 / G), both
//    its v and z channels and the same rows of that head's state S[h] (stored
//    [d_v][d_k], the pretranspose decode layout of the Rocket blog's entry "A
//    reduction barrier makes Qwen GDN graph replay bit exact").
// Every CTA computes exactly the projection rows its channels need, so the
// key head's 16 + 16 + 2R rows of [qkvz; ba] are read once per cluster (b and
// a, two rows per value head, are read by the head's 8 / G CTAs). The q and k
// conv outputs are pushed to all 8 CTAs through distributed shared memory;
// the RMSNorm's sum of o^2 over a head's d_v rows is pushed to the head's
// CTAs the same way. Two cluster barriers in all; every remote store comes
// before the barrier that publishes it, so no CTA reads a peer that may have
// exited.
//
// Numerics are those of the three-kernel step in the same order: the block
// dot products of the warp-MMA projection kernel (exact block sums, weight
// scales applied by FMA in block order per K quarter, quarters added in
// order), the conv taps, norms, gates, delta rule, row reductions (the same
// lane butterfly) and group sums of the mixing kernel. The two paths give
// bit-identical results.
//
// Dependencies: before griddepcontrol.wait the kernel reads only weights
// (bulk copies into shared memory) and slot ids, and asks L2 to prefetch the
// state rows it will update; state and x are read after the wait. So it may
// start while the preceding kernel still runs, and it lets the next kernel
// (the out-projection, which reads only weights before its own wait) launch at
// once.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace gdn {

namespace {

constexpr int kPmThreads = 256;  // 8 warps
constexpr int kPmD = 128;        // head size

// Shared-memory layout (byte offsets, each a multiple of 128).
struct PmSmem {
  size_t bars, w, ba, xh, part, bsum, proj, q, k, v, o, gsum, total;
  __host__ __device__ PmSmem(int R, int MB, int K) {
    const int NG = 2 + 2 * R / 16;                 // MMA row groups: q, k, v (R/16), z (R/16)
    const size_t unit = (size_t)(K / 256) * 576;   // one (group, K quarter) unit
    auto up = [](size_t x) { return (x + 127) / 128 * 128; };
    bars = 0;
    w = 128;
    ba = up(w + (size_t)NG * 4 * unit);
    xh = up(ba + 2 * (size_t)(K / 2 + K / 16));
    part = up(xh + (size_t)MB * K * 2);
    bsum = up(part + (size_t)NG * 4 * 16 * MB * 4);
    proj = up(bsum + (size_t)2 * MB * (K / 16) * 4 + (size_t)2 * MB * 4 * 4);
    q = up(proj + (size_t)MB * (32 + 2 * R + 2) * 4);
    k = up(q + (size_t)MB * kPmD * 4);
    v = up(k + (size_t)MB * kPmD * 4);
    o = up(v + (size_t)MB * R * 4);
    gsum = up(o + (size_t)MB * R * 4);
    total = up(gsum + (size_t)MB * (kPmD / 16) * 4);
  }
};

template <int R, int MB, bool SB>
__global__ void __launch_bounds__(kPmThreads, 1) proj_mix_kernel(PmArgs a) {
  constexpr int D = kPmD, EPL = D / 32;
  constexpr int NS = D / R;              // CTAs (d_v slices) per value head
  constexpr int G = 8 / NS;              // value heads per key head
  constexpr int NG = 2 + 2 * R / 16;     // MMA row groups of this CTA
  constexpr int NU = NG * 4;             // (group, K quarter) units
  constexpr int UPW = NU / 8;            // units per warp
  constexpr int RPW = R / 8;             // state rows per warp
  constexpr int NP = 32 + 2 * R + 2;     // projection values per row: q16 k16 v z b a
  static_assert(NU % 8 == 0 && R % 16 == 0 && RPW >= 1, "unit split");
  extern __shared__ __align__(128) unsigned char smem[];
  const int K = a.H;
  const PmSmem L(R, MB, K);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);  // 8 warps + the b/a rows
  unsigned char *wsm = smem + L.w;
  unsigned char *bas = smem + L.ba;
  __half *xh = reinterpret_cast<__half *>(smem + L.xh);
  float *part = reinterpret_cast<float *>(smem + L.part);   // [unit][16 rows][MB]
  float *bsum = reinterpret_cast<float *>(smem + L.bsum);   // [2][MB][K/16]
  float *proj = reinterpret_cast<float *>(smem + L.proj);   // [MB][NP]
  float *s_q = reinterpret_cast<float *>(smem + L.q);       // [MB][D] conv outputs of the key head's q
  float *s_k = reinterpret_cast<float *>(smem + L.k);       // [MB][D] and k channels
  float *s_v = reinterpret_cast<float *>(smem + L.v);       // [MB][R] conv outputs of this CTA's v channels
  float *s_o = reinterpret_cast<float *>(smem + L.o);       // [MB][R] delta-rule outputs, later y
  float *s_gsum = reinterpret_cast<float *>(smem + L.gsum); // [MB][D/16] sums of o^2 per 16-row group

  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster.block_rank();
  const int kh = blockIdx.x / 8;
  const int hl = rank / NS, sl = rank % NS;
  const int h = kh * G + hl;
  const int row0 = sl * R;                               // first d_v row of this CTA
  const int Hk = a.Hk, Hv = a.Hv, C = a.C, Kc = a.Kc, B = a.B;
  const int vd = Hv * D;
  const int nkb4 = K >> 6, qkb4 = nkb4 >> 2, nblk = K >> 4;
  const uint32_t cbytes = (uint32_t)qkb4 * 512, sbytes = (uint32_t)qkb4 * 64, ubytes = cbytes + sbytes;
  const size_t group_bytes = (size_t)nkb4 * 576;

  // first [qkvz; ba] row of MMA group g of this CTA
  auto group_row = [&](int g) -> int {
    if (g == 0) return kh * D + rank * 16;                                     // q
    if (g == 1) return Hk * D + kh * D + rank * 16;                            // k
    if (g < 2 + R / 16) return 2 * Hk * D + h * D + row0 + (g - 2) * 16;       // v
    return 2 * Hk * D + vd + h * D + row0 + (g - 2 - R / 16) * 16;             // z
  };

  // ---- before the dependency wait: weights into shared memory, state to L2
  if (lane == 0) {
    mbar_init(bars + warp, 1);
    if (warp == 0) mbar_init(bars + 8, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bars + warp, UPW * ubytes);
#pragma unroll
    for (int i = 0; i < UPW; ++i) {
      const int u = warp + 8 * i, g = u >> 2, q = u & 3;
      const unsigned char *src = a.w_mma + (size_t)(group_row(g) >> 4) * group_bytes;
      unsigned char *dst = wsm + (size_t)u * ubytes;
      bulk_g2s(dst, src + (size_t)q * cbytes, cbytes, bars + warp);
      bulk_g2s(dst + cbytes, src + (size_t)nkb4 * 512 + (size_t)q * sbytes, sbytes, bars + warp);
    }
    if (warp == 0) {  // the b and a rows of value head h, row-major
      const uint32_t cb = (uint32_t)K / 2, sb = (uint32_t)K / 16;
      mbar_arrive_expect_tx(bars + 8, 2 * (cb + sb));
      for (int r = 0; r < 2; ++r) {
        const size_t row = (size_t)a.Nqkvz + (r ? Hv : 0) + h;
        bulk_g2s(bas + r * (cb + sb), a.w_codes + row * cb, cb, bars + 8);
        bulk_g2s(bas + r * (cb + sb) + cb, a.w_scales + row * sb, sb, bars + 8);
      }
    }
  }
  // slot ids are written by no kernel of this library; a row is live when its
  // slot is in range and used by no other row
  __shared__ int s_slot[MB];
  int slot[MB];
  uint32_t live = 0;
  bool bad = false;
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    slot[m] = m < B ? a.slot_ids[m] : -1;
    if (slot[m] >= 0 && slot[m] < a.num_slots) live |= 1u << m;
    if (m < B && (slot[m] < -1 || slot[m] >= a.num_slots)) bad = true;
  }
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int j = 0; j < MB; ++j)
      if (j != m && ((live >> m) & 1) && slot[j] == slot[m]) { live &= ~(1u << m); bad = true; }
  if (tid < MB) s_slot[tid] = slot[tid];
  constexpr size_t kEs = SB ? 2 : 4;
  const size_t head_bytes = (size_t)D * D * kEs;
#pragma unroll
  for (int m = 0; m < MB; ++m)  // this CTA's R state rows of each live row: one contiguous run
    if (tid == m && ((live >> m) & 1))
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char *>(a.ssm_state) +
                   ((size_t)slot[m] * Hv + h) * head_bytes + (size_t)row0 * D * kEs), "r"((uint32_t)(R * D * kEs))
                   : "memory");
  pdl_launch_dependents();
  pdl_wait();

  // ---- x rows -> x_hat (FP16, exact) for the MMA columns
  {
    const float inv6ts = inv6ts_of(a.ts_in);
    for (int jm = tid; jm < B * nblk; jm += kPmThreads) {
      const int m = jm / nblk, j = jm - m * nblk;
      uint32_t lo = 0, hi = 0, s = 0;
      if ((live >> m) & 1) {
        float v[16];
        load_bf16x16(a.x + (size_t)m * K + (size_t)j * 16, v);
        if (!quant_block16(v, a.ts_in, inv6ts, lo, hi, s) && blockIdx.x == 0)
          flag_status(a.status, GDN_E_NONFINITE);
      }
      store_xhat_block(xh + (size_t)m * K + (size_t)j * 16, lo, hi, s);
    }
  }
  // the first live row's state rows, requested now so they arrive under the projections
  const int lr0 = warp * RPW;  // this warp's first state row within the CTA's R
  auto srow = [&](int m) -> const char * {
    return static_cast<const char *>(a.ssm_state) + ((size_t)s_slot[m] * Hv + h) * head_bytes +
           ((size_t)(row0 + lr0) * D + lane * EPL) * kEs;
  };
  float st[RPW][EPL];
  auto load_state = [&](int m, float (&dst)[RPW][EPL]) {
    const char *p = srow(m);
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      if (SB) {
        const uint2 t = *reinterpret_cast<const uint2 *>(p + (size_t)j * D * kEs);
        dst[j][0] = __uint_as_float(t.x << 16);
        dst[j][1] = __uint_as_float(t.x & 0xFFFF0000u);
        dst[j][2] = __uint_as_float(t.y << 16);
        dst[j][3] = __uint_as_float(t.y & 0xFFFF0000u);
      } else {
        const float4 t = *reinterpret_cast<const float4 *>(p + (size_t)j * D * kEs);
        dst[j][0] = t.x; dst[j][1] = t.y; dst[j][2] = t.z; dst[j][3] = t.w;
      }
    }
  };
  __syncthreads();  // x_hat and s_slot complete; barrier initialisation visible to every warp
  if (live) load_state(__ffs(live) - 1, st);

  // ---- projection rows on warp-level MMA: unit u = (group u/4, K quarter u%4)
  const int g8 = lane >> 2, t4 = lane & 3;
  bool ok = mbar_wait(bars + warp, 0);
  if (ok) {
#pragma unroll 1
    for (int i = 0; i < UPW; ++i) {
      const int u = warp + 8 * i, q = u & 3;
      const uint4 *codes = reinterpret_cast<const uint4 *>(wsm + (size_t)u * ubytes);
      const uint32_t *scl = reinterpret_cast<const uint32_t *>(wsm + (size_t)u * ubytes + cbytes);
      const __half *xrow = xh + (size_t)(g8 < B ? g8 : 0) * K + 4 * t4;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int s = 0; s < qkb4; ++s) {
        const uint4 c4 = codes[s * 32 + lane];
        float swg[4], swg8[4];
        e4m3x4_to_f32(scl[s * 16 + g8], swg);
        e4m3x4_to_f32(scl[s * 16 + g8 + 8], swg8);
        const int kb0 = (q * qkb4 + s) * 4;
        const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __half2 hv[4];
          e2m1x8_to_h2x4(cw[j], hv);
          const uint32_t af[4] = {*reinterpret_cast<uint32_t *>(&hv[0]), *reinterpret_cast<uint32_t *>(&hv[2]),
                                  *reinterpret_cast<uint32_t *>(&hv[1]), *reinterpret_cast<uint32_t *>(&hv[3])};
          uint32_t b0 = 0, b1 = 0;
          if (g8 < B) {
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
      float *pu = part + (size_t)u * 16 * MB;
      const int c0 = 2 * t4, c1 = 2 * t4 + 1;
      if (c0 < MB) { pu[g8 * MB + c0] = acc[0]; pu[(g8 + 8) * MB + c0] = acc[2]; }
      if (c1 < MB) { pu[g8 * MB + c1] = acc[1]; pu[(g8 + 8) * MB + c1] = acc[3]; }
    }
  }
  // ---- the b and a rows: exact block sums on the CUDA cores, then the same
  // FMA chains (blocks in order per K quarter, quarters in order)
  const bool ok_ba = mbar_wait(bars + 8, 0);
  ok = ok && ok_ba;
  if (ok_ba) {
    const int cb = K / 2, sb = K / 16;
    for (int it = tid; it < 2 * B * nblk; it += kPmThreads) {
      const int r = it / (B * nblk), rem = it - r * B * nblk, m = rem / nblk, j = rem - m * nblk;
      const uint2 c = *reinterpret_cast<const uint2 *>(bas + r * (cb + sb) + j * 8);
      __half2 wv[8];
      e2m1x8_to_h2x4(c.x, *reinterpret_cast<__half2(*)[4]>(&wv[0]));
      e2m1x8_to_h2x4(c.y, *reinterpret_cast<__half2(*)[4]>(&wv[4]));
      const __half2 *xv = reinterpret_cast<const __half2 *>(xh + (size_t)m * K + (size_t)j * 16);
      float sum = 0.0f;  // products exact in FP32, their sum exact (multiples of one quantum)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 w2 = __half22float2(wv[e]), x2 = __half22float2(xv[e]);
        sum = fmaf(w2.x, x2.x, sum);
        sum = fmaf(w2.y, x2.y, sum);
      }
      bsum[(r * MB + m) * nblk + j] = sum;
    }
  }
  __syncthreads();
  // the b and a rows' quarter chains: one thread per (row, m, quarter), its
  // block sums and scales in registers, then the FMAs in block order
  float *bpart = bsum + (size_t)2 * MB * nblk;  // [2][MB][4], after the block sums
  if (tid < 2 * B * 4) {
    const int r = tid / (B * 4), rem = tid - r * B * 4, m = rem >> 2, q = rem & 3;
    const int nq = nblk >> 2;  // blocks per quarter, a multiple of 4
    const float4 *bs = reinterpret_cast<const float4 *>(bsum + (size_t)(r * MB + m) * nblk + q * nq);
    const uint32_t *scw = reinterpret_cast<const uint32_t *>(bas + r * (K / 2 + K / 16) + K / 2 + q * nq);
    float acc = 0.0f;
#pragma unroll 4
    for (int j4 = 0; j4 < nq / 4; ++j4) {
      const float4 b4 = bs[j4];
      float sw[4];
      e4m3x4_to_f32(scw[j4], sw);
      acc = fmaf(b4.x, sw[0], acc);
      acc = fmaf(b4.y, sw[1], acc);
      acc = fmaf(b4.z, sw[2], acc);
      acc = fmaf(b4.w, sw[3], acc);
    }
    bpart[(r * MB + m) * 4 + q] = acc;
  }
  __syncthreads();
  // combine: projection value n of row m = ((q0 + q1) + q2) + q3, scaled, BF16
  {
    const float tsq = a.ts_in * a.ts_qkvz;
    for (int i = tid; i < B * (NG * 16 + 2); i += kPmThreads) {
      const int m = i / (NG * 16 + 2), n = i - m * (NG * 16 + 2);
      float y;
      if (n < NG * 16) {
        const int g = n >> 4, r = n & 15;
        const float *p0 = part + (size_t)(g * 4) * 16 * MB + r * MB + m;
        const size_t qs = (size_t)16 * MB;
        y = (((p0[0] + p0[qs]) + p0[2 * qs]) + p0[3 * qs]) * tsq;
      } else {  // b (n = NG*16) or a: the quarter sums in order
        const float *qv = bpart + ((n - NG * 16) * MB + m) * 4;
        y = (((qv[0] + qv[1]) + qv[2]) + qv[3]) * (a.ts_in * a.ts_ba);
      }
      proj[m * NP + n] = bf16_bits_to_f32(f32_to_bf16_bits(y));
    }
  }
  __syncthreads();

  // ---- conv + SiLU of this CTA's channels: q 16, k 16 (pushed to every CTA of
  // the cluster), v R (kept); the conv state of these channels shifts in place
  for (int i = tid; i < B * (32 + R); i += kPmThreads) {
    const int m = i / (32 + R), c = i - m * (32 + R);
    if (!((live >> m) & 1)) continue;
    int ch, pidx;
    if (c < 16) { ch = kh * D + rank * 16 + c; pidx = c; }
    else if (c < 32) { ch = Hk * D + kh * D + rank * 16 + (c - 16); pidx = c; }
    else { ch = 2 * Hk * D + h * D + row0 + (c - 32); pidx = c; }
    uint16_t *cst = a.conv_state + (size_t)s_slot[m] * (Kc - 1) * C + ch;
    uint16_t tap[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) tap[j] = j < Kc - 1 ? cst[(size_t)j * C] : uint16_t(0);
    const uint16_t xn = f32_to_bf16_bits(proj[m * NP + pidx]);
    float pre = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < Kc) {
        const uint16_t bits = j < Kc - 1 ? tap[j < 3 ? j : 2] : xn;
        pre = fmaf(bf16_bits_to_f32(a.conv_w[(size_t)ch * Kc + j]), bf16_bits_to_f32(bits), pre);
      }
    }
    for (int j = 0; j < Kc - 2; ++j) cst[(size_t)j * C] = tap[j + 1 < 3 ? j + 1 : 2];
    cst[(size_t)(Kc - 2) * C] = xn;
    const float out = siluf_(pre);
    if (c < 32) {
      float *dst = (c < 16 ? s_q : s_k) + m * D + rank * 16 + (c & 15);
#pragma unroll 1
      for (int r2 = 0; r2 < 8; ++r2) *cluster.map_shared_rank(dst, r2) = out;
    } else {
      s_v[m * R + (c - 32)] = out;
    }
  }
  cluster.sync();  // every CTA's q/k conv outputs have landed

  // ---- per row: normalised q, k, gates, the delta rule on this warp's rows
  const float A_log = a.A_log[h], dt_bias = a.dt_bias[h];
#pragma unroll 1
  for (int m = 0; m < B; ++m) {
    if (!((live >> m) & 1)) continue;
    float nxt[RPW][EPL];
    const uint32_t later = live >> (m + 1);
    const int mn = later ? m + __ffs(later) : -1;  // the next live row
    if (mn >= 0) load_state(mn, nxt);
    float kr[EPL], qr[EPL];
    float ssk = 0.0f, ssq = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kr[e] = s_k[m * D + lane * EPL + e];
      qr[e] = s_q[m * D + lane * EPL + e];
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
    const float beta = sigmoidf_(proj[m * NP + 32 + 2 * R]);
    const float g = -expf(A_log) * softplusf_(proj[m * NP + 32 + 2 * R + 1] + dt_bias);
    const float alpha = expf(g);
    float vals[2 * RPW];
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      float dk = 0.0f, dq = 0.0f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        dk = fmaf(st[j][e], kr[e], dk);
        dq = fmaf(st[j][e], qr[e], dq);
      }
      vals[j] = dk;
      vals[RPW + j] = dq;
    }
    const float tot = warp_transpose_reduce<2 * RPW>(vals, lane);
    char *sw = const_cast<char *>(srow(m));
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
      const float Sk = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * RPW>(j));
      const float Sq = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * RPW>(RPW + j));
      // S <- alpha S; u = beta (v - S k); S <- S + u k^T; o = S q
      const float u = beta * (s_v[m * R + lr0 + j] - alpha * Sk);
      const float o = fmaf(u, kq, alpha * Sq);
#pragma unroll
      for (int e = 0; e < EPL; ++e) st[j][e] = fmaf(u, kr[e], alpha * st[j][e]);
      if (lane == 0) s_o[m * R + lr0 + j] = o;
      if (SB) {
        uint32_t b[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) b[e] = f32_to_bf16_bits(st[j][e]);
        *reinterpret_cast<uint2 *>(sw + (size_t)j * D * kEs) = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
      } else {
        *reinterpret_cast<float4 *>(sw + (size_t)j * D * kEs) = make_float4(st[j][0], st[j][1], st[j][2], st[j][3]);
      }
    }
    if (mn >= 0) {
#pragma unroll
      for (int j = 0; j < RPW; ++j)
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[j][e] = nxt[j][e];
    }
  }
  __syncthreads();  // s_o complete

  // ---- sums of o^2 per 16-row group, pushed to the head's NS CTAs
  for (int i = tid; i < B * (R / 16); i += kPmThreads) {
    const int m = i / (R / 16), grp = i - m * (R / 16);
    if (!((live >> m) & 1)) continue;
    float p = 0.0f;
    for (int r = 0; r < 16; ++r) p = fmaf(s_o[m * R + grp * 16 + r], s_o[m * R + grp * 16 + r], p);
    float *dst = s_gsum + m * (D / 16) + sl * (R / 16) + grp;
#pragma unroll 1
    for (int s2 = 0; s2 < NS; ++s2) *cluster.map_shared_rank(dst, hl * NS + s2) = p;
  }
  cluster.sync();

  // ---- gated RMSNorm -> y, NVFP4 blocks of 16 rows (row-major scales)
  for (int i = tid; i < B * R; i += kPmThreads) {
    const int m = i / R, r = i - m * R;
    if (!((live >> m) & 1)) continue;
    float sumsq = 0.0f;
    for (int gi = 0; gi < D / 16; ++gi) sumsq += s_gsum[m * (D / 16) + gi];
    const float rstd = 1.0f / sqrtf(sumsq / (float)D + a.rms_eps);
    const float nw = a.norm_w[row0 + r];
    const float zv = proj[m * NP + 32 + R + r];
    s_o[m * R + r] = s_o[m * R + r] * rstd * nw * siluf_(zv);
  }
  __syncthreads();
  for (int i = tid; i < B * (R / 16); i += kPmThreads) {
    const int m = i / (R / 16), blk = i - m * (R / 16);
    const size_t e0 = (size_t)m * vd + h * D + row0 + blk * 16;
    uint32_t lo = 0, hi = 0, s = 0;
    if ((live >> m) & 1) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = s_o[m * R + blk * 16 + e];
      if (!quant_block16(v, a.ts_out, inv6ts_of(a.ts_out), lo, hi, s)) flag_status(a.status, GDN_E_NONFINITE);
    }
    *reinterpret_cast<uint2 *>(a.y_codes + (e0 >> 1)) = make_uint2(lo, hi);  // padding rows: zeros
    a.y_scales[e0 >> 4] = uint8_t(s);
  }
  if (bad && tid == 0 && blockIdx.x == 0) flag_status(a.status, GDN_E_RANGE);
  if (!ok) {
    if (lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
    // copies that were not waited for must land before shared memory goes away
    if (lane == 0) (void)mbar_wait(bars + warp, 0);
    if (tid == 0) (void)mbar_wait(bars + 8, 0);
  }
}

template <int R, int MB, bool SB>
cudaError_t launch_pm_t(const PmArgs &a, const LaunchCtx &lc) {
  const PmSmem L(R, MB, a.H);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(proj_mix_kernel<R, MB, SB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L.total);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hk * 8, 1, 1);
  cfg.blockDim = dim3(kPmThreads, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 8;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, proj_mix_kernel<R, MB, SB>, a);
}

template <int R, int MB>
cudaError_t launch_pm_r(const PmArgs &a, const LaunchCtx &lc) {
  return a.state_bf16 ? launch_pm_t<R, MB, true>(a, lc) : launch_pm_t<R, MB, false>(a, lc);
}

template <int R>
cudaError_t launch_pm_b(const PmArgs &a, const LaunchCtx &lc) {
  if (a.B <= 1) return launch_pm_r<R, 1>(a, lc);
  if (a.B <= 2) return launch_pm_r<R, 2>(a, lc);
  if (a.B <= 4) return launch_pm_r<R, 4>(a, lc);
  return launch_pm_r<R, 8>(a, lc);
}

}  // namespace

bool proj_mix_ok(int H, int Hk, int Hv, int D, int Kc, int B) {
  if (D != kPmD || B < 1 || B > 8 || H % 256 || H > 2048 || Kc < 2 || Kc > 4) return false;
  const int G = Hv / Hk;
  return (G == 1 || G == 2) && Hv % Hk == 0;
}

cudaError_t launch_proj_mix(const PmArgs &a, const LaunchCtx &lc) {
  if (!proj_mix_ok(a.H, a.Hk, a.Hv, kPmD, a.Kc, a.B)) return cudaErrorInvalidValue;
  return (a.Hv / a.Hk == 2) ? launch_pm_b<32>(a, lc) : launch_pm_b<16>(a, lc);
}

}  // namespace gdn
