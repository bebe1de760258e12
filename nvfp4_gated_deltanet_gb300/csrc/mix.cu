// Token mixing of one decode step, fused: depthwise causal conv + SiLU, q/k L2
// norm, the beta/g gates, the gated delta rule on the FP32 state, the z-gated
// RMSNorm and the NVFP4 quantisation of its output.
//
// Work split: one CTA per (row b, value head h, slice of NS) owns R = D/NS rows
// of that head's state S[h] (stored [d_v][d_k], Rocket blog "A reduction
// barrier makes Qwen GDN graph replay bit exact": FlashInfer's pretranspose
// decode layout). Each warp keeps RPW state rows in registers, one row spread
// over the 32 lanes, so S k and S q are row dot products.
//
// A thread-block cluster groups the G = Hv/Hk value heads of one key head and
// their NS slices. It serves two purposes:
//  * the q/k conv state of the key head is read by all G*NS CTAs and written
//    back by cluster rank 0 only after every CTA has passed a cluster barrier
//    that follows its reads;
//  * the RMSNorm needs sum(o^2) over all d_v rows of a head: slices exchange
//    their partial sums through distributed shared memory in a fixed order.
//
// Shared-memory reductions keep the value in a register and pass a barrier
// before the shared slot is reused (the lesson of the same Rocket entry).
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace gdn {

namespace {

// State rows per warp: 16 when one CTA holds a whole head, 8 for half a head,
// 4 for a quarter (eight warps per CTA at d = 128 whatever the slicing: the
// smallest batches have the fewest CTAs, and their latency chain -- conv,
// norms, the row reductions -- shortens with more warps in flight). The row
// dot products reduce over the lanes in the same butterfly order whatever the
// rows per warp, so the results do not depend on it.
template <int NS>
__host__ __device__ constexpr int rows_per_warp() { return NS == 1 ? 16 : (NS == 2 ? 8 : 4); }


template <int D, int NS, bool SB, bool STR>
__global__ void __launch_bounds__((D / NS / rows_per_warp<NS>()) * 32, STR ? 4 : (NS == 1 ? 2 : 0)) mix_kernel(MixArgs a) {
  constexpr int kRPW = rows_per_warp<NS>();
  constexpr int R = D / NS;
  constexpr int WARPS = R / kRPW;
  constexpr int THREADS = WARPS * 32;
  constexpr int EPL = D / 32;
  constexpr int NCH = 2 * D + R;                        // conv channels this CTA needs
  constexpr int CPT = (NCH + THREADS - 1) / THREADS;    // channels per thread
  static_assert(R % 16 == 0 && WARPS >= 1 && R <= THREADS, "slice must hold whole quantisation blocks");

  __shared__ float s_q[D], s_k[D], s_v[R], s_o[R];
  __shared__ uint16_t s_qk_new[3][2 * D];  // new conv state of the q/k channels (K_conv <= 4)
  __shared__ float s_gsum[D / 16];         // sums of o^2 over the head's 16-row groups

  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.Hv / a.Hk;
  const int h = blockIdx.x / NS, split = blockIdx.x % NS;
  const int kh = h / G;
  const int b = blockIdx.y;
  const int io = a.io_mul ? b * a.io_mul + a.io_add : b;  // row of the q|k|v|z, b|a and y buffers
  const int row0 = split * R;  // first d_v row of this slice
  const int vd = a.Hv * D;
  const int C = a.C, Kc = a.Kc;

  // ---- loads that do not depend on the preceding kernel come first. With
  // programmatic dependent launch this kernel starts once the projection
  // kernel has passed its own griddepcontrol.wait, so everything earlier in
  // the stream (slot ids, the previous step's state writes) is complete;
  // only the projections themselves may still be in flight.
  int ch[CPT];
  float cw[CPT][4];
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int t = tid + c * THREADS;
    int q = 0;
    if (t < D) q = kh * D + t;                                  // q
    else if (t < 2 * D) q = a.Hk * D + kh * D + (t - D);        // k
    else if (t < NCH) q = 2 * a.Hk * D + h * D + row0 + (t - 2 * D);  // v
    ch[c] = q;
#pragma unroll
    for (int j = 0; j < 4; ++j) cw[c][j] = (t < NCH && j < Kc) ? bf16_bits_to_f32(a.conv_w[(size_t)q * Kc + j]) : 0.0f;
  }
  const float A_log = a.A_log[h], dt_bias = a.dt_bias[h];
  const float nw = tid < R ? a.norm_w[row0 + tid] : 0.0f;
  const int slot = a.slot_ids[b];
  bool live = slot >= 0 && slot < a.num_slots;
  bool bad = slot < -1 || slot >= a.num_slots;
  if (live) {  // a slot used by two rows: refuse both (each warp checks, B/32 loads per lane)
    bool dup = false;
    for (int j = lane; j < a.B; j += 32) dup |= (j != b && a.slot_ids[j] == slot);
    if (__any_sync(0xffffffffu, dup)) { bad = true; live = false; }
  }
  // state: conv taps and this warp's rows of S. A plain step reads and writes
  // the slot's state; a verify pass reads row b's from *_src (or the slot) and
  // writes it to *_dst, leaving the slot untouched.
  uint16_t *cst_slot = a.conv_state + (size_t)(live ? slot : 0) * (Kc - 1) * C;
  const uint16_t *cst_rd = a.conv_src ? a.conv_src + (size_t)b * a.conv_row_stride : cst_slot;
  uint16_t *cst = a.conv_dst ? a.conv_dst + (size_t)b * a.conv_row_stride : cst_slot;  // written
  uint16_t tap[CPT][3];
  const int lr0 = warp * kRPW;
  // this lane's EPL consecutive d_k elements of each of the warp's rows: FP32,
  // or BF16 bits when SB (loaded to FP32, stored rounded to nearest even)
  constexpr size_t kEs = SB ? 2 : 4;
  const size_t s_rel = (((size_t)h * D + row0 + lr0) * D + lane * EPL) * kEs;
  const size_t s_slot = (size_t)(live ? slot : 0) * a.Hv * D * D * kEs;
  const char *s_rd = (a.ssm_src ? static_cast<const char *>(a.ssm_src) + (size_t)b * a.ssm_row_stride * kEs
                                : static_cast<const char *>(a.ssm_state) + s_slot) + s_rel;
  char *s_wr = (a.ssm_dst ? static_cast<char *>(a.ssm_dst) + (size_t)b * a.ssm_row_stride * kEs
                          : static_cast<char *>(a.ssm_state) + s_slot) + s_rel;
  const float *S = reinterpret_cast<const float *>(s_rd);
  const uint16_t *Sb = reinterpret_cast<const uint16_t *>(s_rd);
  // STR: the state streams. This warp's rows are asked of L2 here and pass
  // through registers 4 at a time after the wait, so the CTAs stay light
  // enough (4 per SM) that a grid of more CTAs than two per SM is resident at
  // once; with the rows held in registers from here such a grid ran as two
  // waves (c16 31.0 -> 26.8 us per layer-step streamed; c8, whose grid fits,
  // 21.9 held against 23.8 streamed).
  constexpr bool STREAM = STR;
  constexpr int RB = STREAM ? 4 : kRPW;  // state rows in registers at a time
  float st[RB][EPL];
  auto load_row = [&](int j, float (&dst)[EPL]) {
    if (SB) {
      uint16_t b[EPL];
      if (EPL == 4) {
        const uint2 t = *reinterpret_cast<const uint2 *>(Sb + (size_t)j * D);
        b[0] = t.x & 0xFFFFu; b[1 % EPL] = t.x >> 16; b[2 % EPL] = t.y & 0xFFFFu; b[3 % EPL] = t.y >> 16;
      } else if (EPL == 2) {
        const uint32_t t = *reinterpret_cast<const uint32_t *>(Sb + (size_t)j * D);
        b[0] = t & 0xFFFFu; b[1 % EPL] = t >> 16;
      } else {
        b[0] = Sb[(size_t)j * D];
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) dst[e] = bf16_bits_to_f32(b[e]);
    } else if (EPL == 4) {
      float4 t4 = *reinterpret_cast<const float4 *>(S + (size_t)j * D);
      dst[0] = t4.x; dst[1 % EPL] = t4.y; dst[2 % EPL] = t4.z; dst[3 % EPL] = t4.w;
    } else if (EPL == 2) {
      float2 t2 = *reinterpret_cast<const float2 *>(S + (size_t)j * D);
      dst[0] = t2.x; dst[1 % EPL] = t2.y;
    } else {
      dst[0] = S[(size_t)j * D];
    }
  };
  if (live) {
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
      for (int j = 0; j < 3; ++j)
        tap[c][j] = (tid + c * THREADS < NCH && j < Kc - 1) ? cst_rd[(size_t)j * C + ch[c]] : uint16_t(0);
    if (STREAM) {
      if (lane == 0)  // this warp's rows: one contiguous run (lane 0's offset is the row start)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s_rd), "r"((uint32_t)(kRPW * D * kEs))
                     : "memory");
    } else {
#pragma unroll
      for (int j = 0; j < kRPW; ++j) {
        if (SB) {
          uint16_t b[EPL];
          if (EPL == 4) {
            const uint2 t = *reinterpret_cast<const uint2 *>(Sb + (size_t)j * D);
            b[0] = t.x & 0xFFFFu; b[1 % EPL] = t.x >> 16; b[2 % EPL] = t.y & 0xFFFFu; b[3 % EPL] = t.y >> 16;
          } else if (EPL == 2) {
            const uint32_t t = *reinterpret_cast<const uint32_t *>(Sb + (size_t)j * D);
            b[0] = t & 0xFFFFu; b[1 % EPL] = t >> 16;
          } else {
            b[0] = Sb[(size_t)j * D];
          }
#pragma unroll
          for (int e = 0; e < EPL; ++e) st[j][e] = bf16_bits_to_f32(b[e]);
        } else if (EPL == 4) {
          float4 t4 = *reinterpret_cast<const float4 *>(S + (size_t)j * D);
          st[j][0] = t4.x; st[j][1 % EPL] = t4.y; st[j][2 % EPL] = t4.z; st[j][3 % EPL] = t4.w;
        } else if (EPL == 2) {
          float2 t2 = *reinterpret_cast<const float2 *>(S + (size_t)j * D);
          st[j][0] = t2.x; st[j][1 % EPL] = t2.y;
        } else {
          st[j][0] = S[(size_t)j * D];
        }
      }
    }
  }

  // ---- the projections come from the preceding kernel
  pdl_wait();
  pdl_launch_dependents();
  const uint16_t *xin = a.qkvz + (size_t)io * a.ld_qkvz;
  if (bad && tid == 0 && blockIdx.x == 0) flag_status(a.status, GDN_E_RANGE);
  if (!live) {  // padding: zero y for this slice, touch no state (whole cluster agrees)
    for (int i = tid; i < R; i += blockDim.x) {
      if (a.y_f32) a.y_f32[(size_t)io * vd + h * D + row0 + i] = 0.0f;
      if (a.y_codes && (i & 1) == 0) a.y_codes[((size_t)io * vd + h * D + row0 + i) >> 1] = 0;
      if (a.y_scales && (i & 15) == 0) {
        const int blk = (h * D + row0 + i) >> 4;
        a.y_scales[a.y_sf_tiled ? sf_tiled_offset(io, blk, vd >> 4) : ((size_t)io * vd >> 4) + blk] = 0;
      }
    }
    return;
  }
  uint16_t xn[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) xn[c] = (tid + c * THREADS < NCH) ? xin[ch[c]] : uint16_t(0);
  const float zv = tid < R ? bf16_bits_to_f32(xin[2 * a.Hk * D + vd + h * D + row0 + tid]) : 0.0f;
  const uint16_t *bain = a.ba + (size_t)io * a.ld_ba;
  const float b_raw = bf16_bits_to_f32(bain[h]);
  const float a_raw = bf16_bits_to_f32(bain[a.Hv + h]);
  // the gates need nothing else: start them before the conv
  const float beta = sigmoidf_(b_raw);
  const float g = -expf(A_log) * softplusf_(a_raw + dt_bias);
  const float alpha = expf(g);

  // ---- conv + SiLU for q, k (key head kh, all D) and v (this slice)
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int t = tid + c * THREADS;
    if (t < NCH) {
      float pre = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < Kc) {
          const uint16_t bits = j < Kc - 1 ? tap[c][j < 3 ? j : 2] : xn[c];
          pre = fmaf(cw[c][j], bf16_bits_to_f32(bits), pre);
        }
      }
      const float out = siluf_(pre);
      if (t < D) s_q[t] = out;
      else if (t < 2 * D) s_k[t - D] = out;
      else s_v[t - 2 * D] = out;
      // new state: taps shift by one, newest raw input last
      if (t < 2 * D) {
        for (int j = 0; j < Kc - 2; ++j) s_qk_new[j][t] = tap[c][j + 1 < 3 ? j + 1 : 2];
        s_qk_new[Kc - 2][t] = xn[c];
      } else {  // v channels belong to this CTA alone
        for (int j = 0; j < Kc - 2; ++j) cst[(size_t)j * C + ch[c]] = tap[c][j + 1 < 3 ? j + 1 : 2];
        cst[(size_t)(Kc - 2) * C + ch[c]] = xn[c];
      }
    }
  }
  __syncthreads();

  // ---- per-warp: normalised q, k in registers; k.q; gates
  float kr[EPL], qr[EPL];
  float ssk = 0.0f, ssq = 0.0f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    kr[e] = s_k[lane * EPL + e];
    qr[e] = s_q[lane * EPL + e];
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

  // ---- the delta rule on this warp's rows, RB at a time
  auto store_row = [&](int j, const float (&src)[EPL]) {
    float *Sf = reinterpret_cast<float *>(s_wr);
    uint16_t *Sw = reinterpret_cast<uint16_t *>(s_wr);
    if (SB) {
      uint32_t b[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) b[e] = f32_to_bf16_bits(src[e]);
      if (EPL == 4)
        *reinterpret_cast<uint2 *>(Sw + (size_t)j * D) = make_uint2(b[0] | (b[1 % EPL] << 16), b[2 % EPL] | (b[3 % EPL] << 16));
      else if (EPL == 2)
        *reinterpret_cast<uint32_t *>(Sw + (size_t)j * D) = b[0] | (b[1 % EPL] << 16);
      else
        Sw[(size_t)j * D] = (uint16_t)b[0];
    } else if (EPL == 4) {
      *reinterpret_cast<float4 *>(Sf + (size_t)j * D) = make_float4(src[0], src[1 % EPL], src[2 % EPL], src[3 % EPL]);
    } else if (EPL == 2) {
      *reinterpret_cast<float2 *>(Sf + (size_t)j * D) = make_float2(src[0], src[1 % EPL]);
    } else {
      Sf[(size_t)j * D] = src[0];
    }
  };
  if constexpr (STREAM) {
  #pragma unroll 1
    for (int j0 = 0; j0 < kRPW; j0 += RB) {
      if (STREAM) {
#pragma unroll
        for (int jj = 0; jj < RB; ++jj) load_row(j0 + jj, st[jj]);
      }
      float vals[2 * RB];
#pragma unroll
      for (int jj = 0; jj < RB; ++jj) {
        float dk = 0.0f, dq = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          dk = fmaf(st[jj][e], kr[e], dk);
          dq = fmaf(st[jj][e], qr[e], dq);
        }
        vals[jj] = dk;
        vals[RB + jj] = dq;
      }
      // the same lane butterfly for every value whatever RB is: each row's
      // totals do not depend on how many rows are reduced together
      const float tot = warp_transpose_reduce<2 * RB>(vals, lane);
#pragma unroll
      for (int jj = 0; jj < RB; ++jj) {
        const float Sk = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * RB>(jj));
        const float Sq = __shfl_sync(0xffffffffu, tot, reduce_owner<2 * RB>(RB + jj));
        // S <- alpha S; u = beta (v - S k); S <- S + u k^T; o = S q
        //   => (alpha S) k = alpha Sk, o = alpha Sq + u (k . q)
        const float u = beta * (s_v[lr0 + j0 + jj] - alpha * Sk);
        const float o = fmaf(u, kq, alpha * Sq);
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[jj][e] = fmaf(u, kr[e], alpha * st[jj][e]);
        if (lane == 0) s_o[lr0 + j0 + jj] = o;
      }
#pragma unroll
      for (int jj = 0; jj < RB; ++jj) store_row(j0 + jj, st[jj]);
    }
  } else {
    // ---- the delta rule on this warp's rows
    {
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
        // S <- alpha S; u = beta (v - S k); S <- S + u k^T; o = S q
        //   => (alpha S) k = alpha Sk, o = alpha Sq + u (k . q)
        const float u = beta * (s_v[lr0 + j] - alpha * Sk);
        const float o = fmaf(u, kq, alpha * Sq);
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[j][e] = fmaf(u, kr[e], alpha * st[j][e]);
        if (lane == 0) s_o[lr0 + j] = o;
      }
      float *Sf = reinterpret_cast<float *>(s_wr);
      uint16_t *Sw = reinterpret_cast<uint16_t *>(s_wr);
#pragma unroll
      for (int j = 0; j < kRPW; ++j) {
        if (SB) {
          uint32_t b[EPL];
#pragma unroll
          for (int e = 0; e < EPL; ++e) b[e] = f32_to_bf16_bits(st[j][e]);
          if (EPL == 4)
            *reinterpret_cast<uint2 *>(Sw + (size_t)j * D) = make_uint2(b[0] | (b[1 % EPL] << 16), b[2 % EPL] | (b[3 % EPL] << 16));
          else if (EPL == 2)
            *reinterpret_cast<uint32_t *>(Sw + (size_t)j * D) = b[0] | (b[1 % EPL] << 16);
          else
            Sw[(size_t)j * D] = (uint16_t)b[0];
        } else if (EPL == 4) {
          *reinterpret_cast<float4 *>(Sf + (size_t)j * D) =
              make_float4(st[j][0], st[j][1 % EPL], st[j][2 % EPL], st[j][3 % EPL]);
        } else if (EPL == 2) {
          *reinterpret_cast<float2 *>(Sf + (size_t)j * D) = make_float2(st[j][0], st[j][1 % EPL]);
        } else {
          Sf[(size_t)j * D] = st[j][0];
        }
      }
    }
  }

  __syncthreads();  // s_o complete

  // ---- sum of o^2 over the head in one fixed order whatever NS is: 16-row
  // group sums (rows in order), then the D/16 group sums in order. Every slice
  // pushes its group sums into the shared memory of all slices of the head
  // (remote stores before the one cluster barrier), so after the barrier each
  // CTA reads only its own shared memory and nobody reads a peer that may have
  // exited.
  if (tid < R / 16) {
    float p = 0.0f;
    for (int i = 0; i < 16; ++i) p = fmaf(s_o[tid * 16 + i], s_o[tid * 16 + i], p);
    if (NS > 1) {
      const int gbase = (h % G) * NS;
      for (int s2 = 0; s2 < NS; ++s2) *cluster.map_shared_rank(&s_gsum[split * (R / 16) + tid], gbase + s2) = p;
    } else {
      s_gsum[tid] = p;
    }
  }
  // One cluster barrier: every slice's group sums have landed, and every CTA
  // of the key head has read the shared q/k conv state (its reads came first).
  if (G * NS > 1) cluster.sync(); else __syncthreads();
  if (cluster.block_rank() == 0) {  // the q/k conv state of this key head
    for (int t = tid; t < 2 * D; t += blockDim.x) {
      const int q = t < D ? kh * D + t : a.Hk * D + kh * D + (t - D);
      for (int j = 0; j < Kc - 1; ++j) cst[(size_t)j * C + q] = s_qk_new[j][t];
    }
  }
  float sumsq = 0.0f;
  for (int gi = 0; gi < D / 16; ++gi) sumsq += s_gsum[gi];
  const float rstd = 1.0f / sqrtf(sumsq / (float)D + a.rms_eps);

  // ---- gated RMSNorm -> y (FP32), then NVFP4 blocks of 16 rows, each block
  // by 16 lanes: shuffle max, then every lane converts its own element -- the
  // operations of quant_block16, so the same bits
  float y = 0.0f;
  if (tid < R) {
    y = s_o[tid] * rstd * nw * siluf_(zv);
    if (a.y_f32) a.y_f32[(size_t)io * vd + h * D + row0 + tid] = y;
  }
  if (a.y_codes && warp < (R + 31) / 32) {  // whole warps (R is a multiple of 16)
    float amax = fabsf(y);
    int finite = amax <= 3.402823466e38f;  // false for NaN and +inf
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o, 16));
      finite &= __shfl_xor_sync(0xffffffffu, finite, o, 16);
    }
    uint32_t sc = 0, code2 = 0;
    const float yn = __shfl_down_sync(0xffffffffu, y, 1, 16);
    if (finite) {
      sc = e4m3_from_f32(__fmul_rn(amax, inv6ts_of(a.ts_out)));
      const float sv = e4m3_to_f32(sc);
      if (sv != 0.0f) {
        const float rr = __frcp_rn(__fmul_rn(sv, a.ts_out));
        code2 = e2m1x2_from_f32(__fmul_rn(y, rr), __fmul_rn(yn, rr));
      }
    }
    uint32_t lo = 0, hi = 0;  // the block's 8 code bytes (lanes 0, 2, .., 14 of the 16)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = __shfl_sync(0xffffffffu, code2, 2 * i, 16);
      if (i < 4) lo |= b << (8 * i); else hi |= b << (8 * (i - 4));
    }
    if (tid < R && (tid & 15) == 0) {
      if (!finite) flag_status(a.status, GDN_E_NONFINITE);
      const size_t e0 = (size_t)io * vd + h * D + row0 + tid;
      *reinterpret_cast<uint2 *>(a.y_codes + (e0 >> 1)) = make_uint2(lo, hi);
      const int blk = (h * D + row0 + tid) >> 4;
      a.y_scales[a.y_sf_tiled ? sf_tiled_offset(io, blk, vd >> 4) : (e0 >> 4)] = uint8_t(sc);
    }
  }
}

template <int D, int NS, bool SB, bool STR>
cudaError_t launch_dn_t(const MixArgs &a, const LaunchCtx &lc) {
  const int G = a.Hv / a.Hk;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hv * NS, a.B, 1);
  cfg.blockDim = dim3((D / NS / rows_per_warp<NS>()) * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = G * NS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mix_kernel<D, NS, SB, STR>, a);
}

template <int D, int NS, bool STR>
cudaError_t launch_dn_s(const MixArgs &a, const LaunchCtx &lc) {
  return a.state_bf16 ? launch_dn_t<D, NS, true, STR>(a, lc) : launch_dn_t<D, NS, false, STR>(a, lc);
}

template <int D, int NS>
cudaError_t launch_dn(const MixArgs &a, const LaunchCtx &lc) {
  if constexpr (NS == 1)
    if ((long long)a.Hv * a.B > 2LL * lc.num_sms) return launch_dn_s<D, NS, true>(a, lc);
  return launch_dn_s<D, NS, false>(a, lc);
}

}  // namespace

// Slices per head: more CTAs when the batch is small (the state traffic of one
// row is spread over more SMs), bounded by the portable cluster size 8.
// Measured on GB300 (us per layer-step, full-width layer / two-way head
// slice): c1 13.2 with two slices vs 13.6 with four and 14.6 with one; c2 14.5
// vs 14.9 / 15.0; c4 equal for one and two; the two-way slice's c1 (16 value
// heads) 12.1 with four vs 13.0 with two; c8 and larger batches best with one.
cudaError_t launch_mix(const MixArgs &a, const LaunchCtx &lc) {
  if (a.B <= 0) return cudaSuccess;
  const int G = a.Hv / a.Hk;
  int ns = a.slices > 0 ? a.slices : (a.Hv * a.B <= 16 ? 4 : (a.B <= 4 ? 2 : 1));
  while (ns > 1 && G * ns > 8) ns >>= 1;
  if (G > 8) return cudaErrorInvalidValue;
  switch (a.D) {
    case 128:
      if (ns == 4) return launch_dn<128, 4>(a, lc);
      if (ns == 2) return launch_dn<128, 2>(a, lc);
      return launch_dn<128, 1>(a, lc);
    case 64:
      if (ns >= 4) return launch_dn<64, 4>(a, lc);
      if (ns == 2) return launch_dn<64, 2>(a, lc);
      return launch_dn<64, 1>(a, lc);
    case 32:
      if (ns >= 2) return launch_dn<32, 2>(a, lc);
      return launch_dn<32, 1>(a, lc);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
