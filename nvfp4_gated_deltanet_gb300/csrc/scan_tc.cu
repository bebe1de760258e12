// The sequential part of chunked prefill -- the scan over 64-token chunks --
// on the fifth-generation tensor cores: tcgen05.mma .kind::tf32 with FP32
// accumulators in tensor memory (bloomery issue #565, §4, #812: the delta
// rule of a prompt runs in chunks on tensor cores; §10 keeps FP32 precision
// by splitting each operand into narrower parts).
//
// One CTA per (value head, R rows of d_v). With S the slice of the state,
// per chunk (W, Ut, A, Gamma from chunk_prep; q, k normalised):
//   P   = [Q; W] S^T                      M = 128 (64 q rows, 64 W rows), N = R, K = d
//   U   = Ut - P_W,  Cf_j = e^(Gamma_64 - Gamma_j) u_j
//   O   = diag(e^Gamma) P_Q + A U         M = 128 (rows past 64 unused), N = R, K = 64
//   S^T <- e^Gamma_64 S^T + K^T Cf        M = 128 (d_k), N = R, K = 64
// The state lives in the registers of the eight epilogue warps, transposed:
// a thread of TMEM lane e holds S[r0 + r][e] for half of the slice's R rows,
// exactly its lane and columns of the update's accumulator, so no state
// element moves between threads. Every product runs in split TF32, x = hi + lo with
// hi = TF32(x) and lo = TF32(x - hi) (round to nearest), as
// a.b ~ hi.hi + lo.hi + hi.lo + lo.lo accumulated in FP32 -- at least the
// 21-bit precision of the warp-level chunk scan. The A operand (the chunk's
// 128-row tiles) sits in tensor memory as hi and lo columns; the B operand
// (S, U, Cf: R rows) is [B_hi; B_lo], N = 2R, from shared memory (K-major,
// 128-byte swizzle), so one K step is two MMAs (A_hi B'^T and A_lo B'^T) and
// the epilogue adds the accumulator's two column halves.
//
// Warp roles (448 threads):
//   warps 0..7   epilogue (two per TMEM lane quarter, each half of the
//                slice's rows): TMEM -> registers, U / Cf / S operand tiles
//                (split) into shared memory, outputs, the state
//   warp 8       TMEM allocation; one thread issues the MMAs
//   warp 9       one thread streams the chunk's [Q; W], A and K^T tiles by
//                TMA (128-byte swizzle) into a ring of 32 KB FP32 landing
//                slots, and asks L2 to prefetch the next chunk
//   warps 10..13 split each landed tile into hi and lo and store both into a
//                tensor-memory slot (tcgen05.st), where the MMAs read their
//                A operand: only the small B operands (S, U, Cf) are read from
//                shared memory, once per MMA
// Every mbarrier wait is bounded; a wait that gives up sets the status word
// (GDN_E_TIMEOUT) and a shared abort flag that ends every role's loop.
#include <cuda.h>

#include "tc.cuh"

namespace gdn {

namespace {

constexpr int kC = 64, kD = 128;
constexpr int kLand = 5;                  // FP32 landing slots in shared memory
constexpr int kLandBytes = 2 * 128 * 128; // two [128 rows][32 floats] sub-tiles
constexpr int kTSlots = 2;                // A-operand slots in tensor memory
constexpr int kTSlotCols = 128;           // hi: 64 columns (K = 64), lo: the next 64
constexpr int kTSlot0 = 192;              // first slot column; accumulators below
constexpr int kEpiWarps = 8;              // two per TMEM lane quarter
constexpr int kSplitWarps = 4;            // one per TMEM lane quarter
constexpr int kScanThreads = 32 * (kEpiWarps + 2 + kSplitWarps);
constexpr int kUsesPerChunk = 4;          // [Q; W] d_k 0..63 and 64..127, K^T, A (K = 64 each)

template <int R>
struct ScanLayout {
  static constexpr int kSub = R * 128;                  // one [R][32 floats] sub-tile
  static constexpr int kRing = kLand * kLandBytes;
  static constexpr int kS = 2 * 4 * kSub;               // S: per 32-wide d_k sub-tile, hi rows then lo rows
  static constexpr int kU = 2 * 2 * kSub;               // U^T: per 32-token sub-tile, hi rows then lo rows
  static constexpr int kCf = kU;                        // Cf^T hi, lo
  static constexpr int kBars = 256;
  static constexpr int kBytes = 1024 + kRing + kS + kU + kCf + kBars;
  static_assert(kSub % 1024 == 0, "sub-tiles stay 1024-byte aligned");
  static_assert(kBytes <= 227 * 1024, "one CTA per SM");
  static_assert(6 * R <= kTSlot0, "accumulators (2R columns each) below the A slots");
};

// D (+)= A B'^T over K = 64 (eight K = 8 steps) with A = hi + lo in tensor
// memory (hi at column a, lo at a + 64) and B' = [B_hi; B_lo] from shared
// memory (N = 2R rows: the hi rows, then the lo rows; b(j) gives the
// descriptor of K step j): columns 0..R-1 of D collect hi.hi + lo.hi and
// columns R..2R-1 hi.lo + lo.lo, which the epilogue adds -- the split
// product in two MMAs per K step. `first` starts the accumulator.
template <typename BD>
GDN_DEV void mma_split_ts(uint32_t d, uint32_t a, BD b, uint32_t idesc, bool first) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint64_t bd = b(j);
    mma_tf32_ts(d, a + 64 + 8 * j, bd, idesc, (first && j == 0) ? 0u : 1u);
    mma_tf32_ts(d, a + 8 * j, bd, idesc, 1u);
  }
}
// The ring's use u in the MMA thread's order: chunk c consumes [Q; W] d_k
// 0..63 and 64..127, then (from c = 1) the previous chunk's A, then its own
// K^T; the last chunk's A comes last. kind: 0, 1 = [Q; W] halves, 2 = K^T,
// 3 = A.
GDN_DEV void ring_use(uint32_t u, int nc, int &kind, int &chunk) {
  if (u < 3) {
    kind = u < 2 ? (int)u : 2;
    chunk = 0;
    return;
  }
  const int c = 1 + (int)((u - 3) / 4), q = (int)((u - 3) % 4);
  if (c == nc) {
    kind = 3;
    chunk = nc - 1;
  } else {
    kind = q < 2 ? q : (q == 2 ? 3 : 2);
    chunk = q == 2 ? c - 1 : c;
  }
}
GDN_DEV void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Bounded wait that also gives up when another role has given up.
GDN_DEV bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag, int32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 2000u)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1u;
      flag_status(status, GDN_E_TIMEOUT);
      return false;
    }
  }
  return true;
}
// The same, decided by lane 0 for the whole warp (collective TMEM accesses
// that follow run with all 32 lanes or none).
GDN_DEV bool warp_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag, int32_t *status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_flag, status) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int R>
__global__ void __launch_bounds__(kScanThreads, 1)
    chunk_scan_umma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmKT,
                           PrefillArgs a) {
  using L = ScanLayout<R>;
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = sm;
  uint8_t *sS = sm + L::kRing;           // S as [R][d_k]: per d_k sub-tile q, hi at 2q, lo at 2q + 1
  uint8_t *sU = sS + L::kS;              // U^T as [R][token]: per token sub-tile, hi then lo
  uint8_t *sCf = sU + L::kU;             // Cf^T, the same layout
  uint64_t *landed = reinterpret_cast<uint64_t *>(sCf + L::kCf);  // TMA -> splitters
  uint64_t *sfree = landed + kLand;                                  // splitters -> TMA
  uint64_t *tfull = sfree + kLand;                                   // splitters -> MMA
  uint64_t *tempty = tfull + kTSlots;                                // MMA -> splitters
  // per chunk: S tile written (all epilogue warps) -> P = [Q; W] S^T done ->
  // Cf tile written (W-row warps) -> state update product done; U tile
  // written (W-row warps) and the previous chunk's output read (Q-row warps)
  // -> A U done
  uint64_t *s_ready = tempty + kTSlots, *p_done = s_ready + 1, *cf_ready = s_ready + 2, *s_acc_done = s_ready + 3,
           *u_ready = s_ready + 4, *o_free = s_ready + 5, *o_done = s_ready + 6, *fin = s_ready + 7;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(s_ready + 8);
  volatile uint32_t *abort_flag = tmem_holder + 1;

  constexpr int NSL = kD / R;
  const int h = blockIdx.x / NSL, r0 = (blockIdx.x % NSL) * R;
  const int kh = h / (a.Hv / a.Hk);
  const int nc = a.Tp / kC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kLand; ++s) {
      mbar_init(landed + s, 1);
      mbar_init(sfree + s, 32 * kSplitWarps);
    }
    for (int t = 0; t < kTSlots; ++t) {
      mbar_init(tfull + t, 32 * kSplitWarps);
      mbar_init(tempty + t, 1);
    }
    mbar_init(s_ready, 32 * kEpiWarps);
    mbar_init(p_done, 1);
    mbar_init(cf_ready, 16 * kEpiWarps);
    mbar_init(s_acc_done, 1);
    mbar_init(u_ready, 16 * kEpiWarps);
    mbar_init(o_free, 16 * kEpiWarps);
    mbar_init(o_done, 1);
    mbar_init(fin, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kEpiWarps) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp < kEpiWarps) {
    // ------------------------------------------------ epilogue: thread = TMEM lane e of its warp's
    // quarter, and one half of the slice's rows (accumulator columns) hf.
    // Lanes 0..63 are the q rows of P and of O, lanes 64..127 the W rows of P;
    // every lane is d_k = e of the state update.
    constexpr int RH = R / 2;
    const int qt = warp & 3, hf = warp >> 2;
    const bool wrow = qt >= 2;
    const int e = 32 * qt + lane, i = e & 63;
    const uint32_t lane_base = tmem + ((uint32_t)(qt * 32) << 16) + RH * hf;
    float Sv[RH];  // S[r0 + RH hf + r][e]
#pragma unroll
    for (int r = 0; r < RH; ++r)
      Sv[r] = state_load(a.ssm, a.state_bf16, ((size_t)h * kD + r0 + RH * hf + r) * kD + e);
    float pq[RH];  // q rows: e^Gamma_i (S q_i) of the chunk whose output is pending
    bool ok = true;
    // q rows: the output of chunk cc = e^Gamma (S q) + A U, once A U is done
    auto emit_o = [&](int cc) -> bool {
      if (!warp_wait(o_done, (uint32_t)(cc & 1), abort_flag, a.status)) return false;
      tc_fence_after();
      uint32_t oa[RH], oa1[RH];
      tmem_ld16(lane_base + 2 * R, oa);
      tmem_ld16(lane_base + 3 * R, oa1);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(o_free);
      const int t = cc * kC + i;
      if (t < a.T) {
        float *op = a.o + ((size_t)t * a.Hv + h) * kD + r0 + RH * hf;
        float ov[RH];
#pragma unroll
        for (int k = 0; k < RH; ++k) ov[k] = pq[k] + (__uint_as_float(oa[k]) + __uint_as_float(oa1[k]));
#pragma unroll
        for (int k = 0; k < RH; k += 4)
          *reinterpret_cast<float4 *>(op + k) = make_float4(ov[k], ov[k + 1], ov[k + 2], ov[k + 3]);
      }
      return true;
    };
    for (int c = 0; c < nc; ++c) {
      // (a) S -> the B operand of P (thread e owns column e of its rows)
      {
        uint8_t *hi = sS + 2 * qt * L::kSub, *lo = hi + L::kSub;
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          uint32_t vh, vl;
          split_hi_lo(Sv[r], vh, vl);
          const uint32_t off = sw_off(RH * hf + r, lane);
          *reinterpret_cast<uint32_t *>(hi + off) = vh;
          *reinterpret_cast<uint32_t *>(lo + off) = vl;
        }
        fence_async_shared();
        tc_fence_before();
        mbar_arrive(s_ready);
      }
      if (!wrow && c > 0 && !emit_o(c - 1)) { ok = false; break; }
      const float *gam = a.Gam + ((size_t)h * nc + c) * kC;
      const float gi = gam[i], gC = gam[kC - 1];
      if (wrow) {
        // (b) W rows: U = Ut - W S^T, the update coefficients Cf = e^(Gamma_64 - Gamma_i) U
        float ut[RH];
        const float4 *up = reinterpret_cast<const float4 *>(a.Ut + (((size_t)h * nc + c) * kC + i) * kD + r0 + RH * hf);
#pragma unroll
        for (int j = 0; j < RH / 4; ++j) {
          const float4 v = up[j];
          ut[4 * j] = v.x; ut[4 * j + 1] = v.y; ut[4 * j + 2] = v.z; ut[4 * j + 3] = v.w;
        }
        const float dc = expf(gC - gi);
        if (!warp_wait(p_done, (uint32_t)(c & 1), abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t pr[RH], pr1[RH];
        tmem_ld16(lane_base, pr);
        tmem_ld16(lane_base + R, pr1);
        tmem_ld_wait();
        const int sub = i >> 5, col = i & 31;
        float u[RH];
#pragma unroll
        for (int k = 0; k < RH; ++k) u[k] = ut[k] - (__uint_as_float(pr[k]) + __uint_as_float(pr1[k]));
        {  // Cf first: the state update is the next chunk's dependency
          uint8_t *ch = sCf + 2 * sub * L::kSub, *cl = ch + L::kSub;
#pragma unroll
          for (int k = 0; k < RH; ++k) {
            uint32_t vh, vl;
            split_hi_lo(dc * u[k], vh, vl);
            const uint32_t off = sw_off(RH * hf + k, col);
            *reinterpret_cast<uint32_t *>(ch + off) = vh;
            *reinterpret_cast<uint32_t *>(cl + off) = vl;
          }
          fence_async_shared();
          tc_fence_before();
          mbar_arrive(cf_ready);
        }
        // the U tile is free once the previous chunk's A U is done
        if (c > 0 && !warp_wait(o_done, (uint32_t)((c - 1) & 1), abort_flag, a.status)) { ok = false; break; }
        {
          uint8_t *uh = sU + 2 * sub * L::kSub, *ul = uh + L::kSub;
#pragma unroll
          for (int k = 0; k < RH; ++k) {
            uint32_t vh, vl;
            split_hi_lo(u[k], vh, vl);
            const uint32_t off = sw_off(RH * hf + k, col);
            *reinterpret_cast<uint32_t *>(uh + off) = vh;
            *reinterpret_cast<uint32_t *>(ul + off) = vl;
          }
          fence_async_shared();
          mbar_arrive(u_ready);
        }
      } else {
        // (b) q rows: e^Gamma_i (S q_i), kept until the chunk's A U is done
        const float di = expf(gi);
        if (!warp_wait(p_done, (uint32_t)(c & 1), abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t pr[RH], pr1[RH];
        tmem_ld16(lane_base, pr);
        tmem_ld16(lane_base + R, pr1);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < RH; ++k) pq[k] = di * (__uint_as_float(pr[k]) + __uint_as_float(pr1[k]));
      }
      // (c) the state update
      if (!warp_wait(s_acc_done, (uint32_t)(c & 1), abort_flag, a.status)) { ok = false; break; }
      tc_fence_after();
      const float dC = expf(gC);
      {
        uint32_t sa[RH], sa1[RH];
        tmem_ld16(lane_base + 4 * R, sa);
        tmem_ld16(lane_base + 5 * R, sa1);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < RH; ++k) Sv[k] = fmaf(dC, Sv[k], __uint_as_float(sa[k]) + __uint_as_float(sa1[k]));
      }
    }
    if (ok && !wrow && nc > 0 && !emit_o(nc - 1)) ok = false;
    if (ok) {
#pragma unroll
      for (int r = 0; r < RH; ++r)
        state_store(a.ssm, a.state_bf16, ((size_t)h * kD + r0 + RH * hf + r) * kD + e, Sv[r]);
    }
  } else if (warp == kEpiWarps) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_tf32(2 * R);
      const uint32_t bS = smem_u32(sS), bU = smem_u32(sU), bC = smem_u32(sCf);
      uint32_t u = 0;
      bool ok = true;
      // use u: A operand in tensor-memory slot u % kTSlots, filled by the splitters
      auto take = [&](uint32_t &col) -> bool {
        const int t = (int)(u % kTSlots);
        if (!wait_or_abort(tfull + t, (u / kTSlots) & 1u, abort_flag, a.status)) return false;
        tc_fence_after();
        col = tmem + kTSlot0 + t * kTSlotCols;
        return true;
      };
      auto give = [&]() {
        tc_commit(tempty + (u % kTSlots));
        ++u;
      };
      // O = A U of chunk cc, once its U tile is written and the q rows have
      // read chunk cc - 1's O
      auto au = [&](int cc) -> bool {
        if (!wait_or_abort(u_ready, (uint32_t)(cc & 1), abort_flag, a.status)) return false;
        if (cc > 0 && !wait_or_abort(o_free, (uint32_t)((cc - 1) & 1), abort_flag, a.status)) return false;
        tc_fence_after();
        uint32_t acol;
        if (!take(acol)) return false;
        mma_split_ts(
            tmem + 2 * R, acol, [&](int j) { return desc_sw128(bU + 2 * (j / 4) * L::kSub) + 2 * (j & 3); }, idesc,
            true);
        give();
        tc_commit(o_done);
        return true;
      };
      for (int c = 0; c < nc && ok; ++c) {
        if (!wait_or_abort(s_ready, (uint32_t)(c & 1), abort_flag, a.status)) break;
        tc_fence_after();
        // P = [Q; W] S^T: d_k 0..63, then 64..127 (S sub-tiles 2 i + j / 4)
        for (int i = 0; i < 2; ++i) {
          uint32_t acol;
          if (!take(acol)) { ok = false; break; }
          mma_split_ts(
              tmem, acol, [&](int j) { return desc_sw128(bS + 2 * (2 * i + j / 4) * L::kSub) + 2 * (j & 3); }, idesc,
              i == 0);
          give();
        }
        if (!ok) break;
        tc_commit(p_done);
        // the previous chunk's O = A U (A's rows in lanes 0..63), while the
        // W-row warps compute this chunk's Cf
        if (c > 0 && !au(c - 1)) break;
        // S_acc = K^T Cf: the next chunk's dependency
        if (!wait_or_abort(cf_ready, (uint32_t)(c & 1), abort_flag, a.status)) break;
        tc_fence_after();
        {
          uint32_t acol;
          if (!take(acol)) break;
          mma_split_ts(
              tmem + 4 * R, acol, [&](int j) { return desc_sw128(bC + 2 * (j / 4) * L::kSub) + 2 * (j & 3); }, idesc,
              true);
          give();
        }
        tc_commit(s_acc_done);
        if (c == nc - 1) au(c);
      }
      // every MMA issued has completed before the CTA may leave
      tc_commit(fin);
      mbar_wait(fin, 0u);
    }
  } else if (warp == kEpiWarps + 1) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t total = (uint32_t)nc * kUsesPerChunk;
      for (uint32_t u = 0; u < total; ++u) {
        const int s = (int)(u % kLand);
        if (u >= (uint32_t)kLand && !wait_or_abort(sfree + s, ((u / kLand) - 1u) & 1u, abort_flag, a.status)) break;
        int q, c;
        ring_use(u, nc, q, c);
        if (q == 0 && c + 1 < nc) {  // the next chunk's operands and Ut rows into L2
          const int n = c + 1;
          prefetch_l2(a.qn + ((size_t)kh * a.Tp + (size_t)n * kC) * kD, kC * kD * 4);
          prefetch_l2(a.W + ((size_t)h * nc + n) * kC * kD, kC * kD * 4);
          prefetch_l2(a.Am + ((size_t)h * nc + n) * kC * kC, kC * kC * 4);
          prefetch_l2(a.KT + ((size_t)kh * nc + n) * kD * kC, kD * kC * 4);
          prefetch_l2(a.Ut + ((size_t)h * nc + n) * kC * kD, kC * kD * 4);
        }
        // two [128 rows][32 floats] sub-tiles: K columns 0..31 and 32..63 of the use
        uint8_t *d0 = ring + s * kLandBytes, *d1 = d0 + kLandBytes / 2;
        mbar_arrive_expect_tx(landed + s, q == 3 ? kLandBytes / 2 : kLandBytes);
        if (q < 2) {         // [Q; W], d_k columns 64 q .. 64 q + 63
          const int yq = kh * a.Tp + c * kC, yw = (h * nc + c) * kC;
          tma_load_2d(d0, &tmQ, 256 * q, yq, landed + s);
          tma_load_2d(d0 + 64 * 128, &tmW, 256 * q, yw, landed + s);
          tma_load_2d(d1, &tmQ, 256 * q + 128, yq, landed + s);
          tma_load_2d(d1 + 64 * 128, &tmW, 256 * q + 128, yw, landed + s);
        } else if (q == 2) { // K^T: 128 rows of d_k
          tma_load_2d(d0, &tmKT, 0, (kh * nc + c) * kD, landed + s);
          tma_load_2d(d1, &tmKT, 128, (kh * nc + c) * kD, landed + s);
        } else {             // A: 64 rows
          tma_load_2d(d0, &tmA, 0, (h * nc + c) * kC, landed + s);
          tma_load_2d(d1, &tmA, 128, (h * nc + c) * kC, landed + s);
        }
      }
    }
  } else {
    // ------------------------------------------------ splitters (one warp per TMEM lane quarter)
    // thread = row m of the use (its TMEM lane); both 32-wide halves of the
    // use's K columns in turn
    const int qt = warp & 3;
    const int m = 32 * qt + lane;
    const uint32_t tlane = (uint32_t)(qt * 32) << 16;
    const uint32_t total = (uint32_t)nc * kUsesPerChunk;
    for (uint32_t u = 0; u < total; ++u) {
      const int s = (int)(u % kLand), t = (int)(u % kTSlots);
      int q, cq;
      ring_use(u, nc, q, cq);
      const bool live = !(q == 3 && m >= kC);  // A has 64 rows; lanes 64..127 of its slot are never read out
      if (u >= (uint32_t)kTSlots && !warp_wait(tempty + t, ((u / kTSlots) - 1u) & 1u, abort_flag, a.status)) break;
      if (!warp_wait(landed + s, (u / kLand) & 1u, abort_flag, a.status)) break;
      if (live) {
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t vh[32], vl[32];
          const uint8_t *src = ring + s * kLandBytes + hf * (kLandBytes / 2) + m * 128;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + ((c4 ^ (m & 7)) << 4));
            split_hi_lo(x.x, vh[4 * c4], vl[4 * c4]);
            split_hi_lo(x.y, vh[4 * c4 + 1], vl[4 * c4 + 1]);
            split_hi_lo(x.z, vh[4 * c4 + 2], vl[4 * c4 + 2]);
            split_hi_lo(x.w, vh[4 * c4 + 3], vl[4 * c4 + 3]);
          }
          const uint32_t col = tmem + tlane + kTSlot0 + t * kTSlotCols + 32 * hf;
          tmem_st32(col, vh);
          tmem_st32(col + 64, vl);
        }
      }
      mbar_arrive(sfree + s);  // the landing slot has been read
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(tfull + t);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kEpiWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// The tcgen05 chunk scan for d = 128 (slices of 32 rows of d_v per CTA).
// Needs chunk_prep's W, Ut, Am, Gam and KT.
cudaError_t launch_chunk_scan_umma(const PrefillArgs &a, cudaStream_t stream) {
  constexpr int R = 32;
  if (a.D != kD || !a.KT) return cudaErrorInvalidValue;
  const uint64_t nc = (uint64_t)a.Tp / kC;
  CUtensorMap mQ, mW, mA, mKT;
  if (!make_map(&mQ, a.qn, (uint64_t)a.Hk * a.Tp, kD * 4, kC, 128, true) ||
      !make_map(&mW, a.W, (uint64_t)a.Hv * a.Tp, kD * 4, kC, 128, true) ||
      !make_map(&mA, a.Am, (uint64_t)a.Hv * a.Tp, kC * 4, kC, 128, true) ||
      !make_map(&mKT, a.KT, (uint64_t)a.Hk * nc * kD, kC * 4, kD, 128, true))
    return cudaErrorInvalidValue;
  const int smem = ScanLayout<R>::kBytes;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(chunk_scan_umma_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  chunk_scan_umma_kernel<R><<<a.Hv * (kD / R), kScanThreads, smem, stream>>>(mQ, mW, mA, mKT, a);
  return cudaGetLastError();
}

}  // namespace gdn
