// The sequential part of chunked prefill -- the scan over 64-token chunks --
// on the fifth-generation tensor cores: tcgen05.mma .kind::f16 with FP32
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
// element moves between threads.
//
// Every product runs in split FP16: an operand block x with a power-of-two
// scale s (its largest |x s| below 2^14) is x s = hi + lo, hi = FP16(x s),
// lo = FP16(x s - hi), 22 significant bits, and
// a.b ~ (hi.hi + lo.hi + hi.lo + lo.lo) / (s_a s_b) accumulated in FP32. The
// A operands (q, W, A, K^T: 128-row tiles) come split from chunk_prep -- q, A
// and K^T with the fixed 2^14, each chunk's W with its own scale -- and are
// read by the MMAs straight from shared memory; the B operands (S, U and Cf:
// R rows) are split here with a scale from the tile's largest magnitude (Cf
// shares U's: |Cf| <= |U|) and laid out as [B_hi; B_lo], N = 2R, so one K step
// is two MMAs (A_hi B'^T and A_lo B'^T) and the epilogue adds the
// accumulator's two column halves and multiplies by the exact inverse scales.
//
// Warp roles (320 threads):
//   warps 0..7   epilogue (two per TMEM lane quarter, each half of the
//                slice's rows): TMEM -> registers, U / Cf / S operand tiles
//                (split) into shared memory, outputs, the state
//   warp 8       TMEM allocation; one thread issues the MMAs
//   warp 9       one thread streams the chunk's split [Q; W], A and K^T tiles
//                by TMA (128-byte swizzle) into a ring of 32 KB slots (hi
//                16 KB, lo 16 KB), and asks L2 to prefetch the next chunk
// Every mbarrier wait is bounded; a wait that gives up sets the status word
// (GDN_E_TIMEOUT) and a shared abort flag that ends every role's loop.
#include <cuda.h>

#include "tc.cuh"

namespace gdn {

namespace {

constexpr int kC = 64, kD = 128;
constexpr int kLand = 6;                  // operand slots in shared memory
constexpr int kLandBytes = 32 * 1024;     // hi [128 rows][64 FP16], then lo
constexpr int kLoOff = 16 * 1024;         // the lo tile within a slot
constexpr float kFixedScale = 16384.0f;   // 2^14: q, k and A are bounded by 1 (|q_i| <= d^-1/2, |k_i| = 1)
constexpr int kEpiWarps = 8;              // two per TMEM lane quarter
constexpr int kScanThreads = 32 * (kEpiWarps + 2);
constexpr int kUsesPerChunk = 4;          // [Q; W] d_k 0..63 and 64..127, K^T, A (K = 64 each)
static_assert(kLand >= kUsesPerChunk, "a chunk's uses are held together until its slots are released");

template <int R>
struct ScanLayout {
  static constexpr int kSub = 2 * R * 128;              // one [2R][64 FP16] sub-tile: hi rows, then lo rows
  static constexpr int kRing = kLand * kLandBytes;
  static constexpr int kS = 2 * kSub;                   // S: two 64-wide d_k sub-tiles
  static constexpr int kU = kSub;                       // U^T: the 64 tokens
  static constexpr int kCf = kU;                        // Cf^T hi, lo
  static constexpr int kBars = 512;
  static constexpr int kBytes = 1024 + kRing + kS + kU + kCf + kBars;
  static_assert(kSub % 1024 == 0, "sub-tiles stay 1024-byte aligned");
  static_assert(kBytes <= 227 * 1024, "one CTA per SM");
  static_assert(6 * R <= 256, "three accumulators of 2R columns");
};

// byte offset of FP16 element (row, col) in a [rows][64 FP16] tile, 128-byte swizzle
GDN_DEV uint32_t sw_off16(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}
// Instruction descriptor of kind::f16 with FP16 A and B, FP32 accumulator,
// both K-major, M = 128, N = n.
GDN_DEV uint32_t idesc_f16(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
GDN_DEV void mma_f16_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (+)= A B'^T over K = 64 (four K = 16 steps) with A = hi + lo in a ring
// slot (hi tile at `slot`, lo tile kLoOff further) and B' = [B_hi; B_lo]
// (N = 2R; b(j): the descriptor of K step j): columns 0..R-1 of D collect
// hi.hi + lo.hi and R..2R-1 hi.lo + lo.lo, which the epilogue adds -- the split
// product in two MMAs per 16-wide K step. `first` starts the accumulator.
template <typename BD>
GDN_DEV void mma_split(uint32_t d, uint32_t slot, BD b, uint32_t idesc, bool first) {
  const uint64_t ah = desc_sw128(slot), al = desc_sw128(slot + kLoOff);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t bd = b(j);
    mma_f16_ss(d, al + 2 * j, bd, idesc, (first && j == 0) ? 0u : 1u);
    mma_f16_ss(d, ah + 2 * j, bd, idesc, 1u);
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

// 1 / s for a power of two s = 2^k, |k| <= 126: the exponent negated (exact)
GDN_DEV float inv_pow2(float s) { return __uint_as_float((254u << 23) - __float_as_uint(s)); }

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

// The largest of v over the eight epilogue warps: lane 0 of each warp posts
// its warp's largest value in red[warp] and arrives on `bar` (count 8), waits
// for the phase, and reads all eight; the warp takes lane 0's result. red is
// double-buffered by the caller (a warp writes the next buffer only after
// every warp has arrived at this phase, i.e. has read the previous one), and
// the phase parity alternates the same way.
GDN_DEV bool epi_max(float v, float *red, uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                     int32_t *status, float &out) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  int ok = 0;
  float m = 0.0f;
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = v;
    mbar_arrive(bar);
    ok = wait_or_abort(bar, parity, abort_flag, status) ? 1 : 0;
    if (ok) {
      m = red[0];
#pragma unroll
      for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
    }
  }
  out = __shfl_sync(0xffffffffu, m, 0);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Rows row0 .. row0 + RH - 1 of a split B tile [2R][64 FP16] (hi rows, lo
// rows R further on), column `col` of this lane, the value of row row0 + r
// being v[r] s. Neighbouring lanes (col even, col + 1) pair up so that each
// 32-bit store holds two neighbouring columns: the even lane writes row r and
// the odd lane row r + 4 of each group of eight, which fall on disjoint halves
// of the 128-byte swizzle -- every store is one conflict-free wavefront.
template <int R, int RH>
GDN_DEV void put_split_rows(uint8_t *tile, int row0, int col, const float (&v)[RH], float s, int lane) {
  static_assert(RH % 8 == 0, "rows in groups of eight");
  const bool odd = (lane & 1) != 0;
#pragma unroll
  for (int g = 0; g < RH; g += 8)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = g + j;
      const float other = __shfl_xor_sync(0xffffffffu, odd ? v[r] : v[r + 4], 1);
      const float x0 = odd ? other : v[r], x1 = odd ? v[r + 4] : other;
      uint32_t hi, lo;
      split_f16x2(x0 * s, x1 * s, hi, lo);
      const uint32_t off = sw_off16(row0 + r + (odd ? 4 : 0), col & ~1);
      *reinterpret_cast<uint32_t *>(tile + off) = hi;
      *reinterpret_cast<uint32_t *>(tile + off + R * 128) = lo;
    }
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
  uint8_t *tS = sm + L::kRing;           // S as [R][d_k]: d_k 0..63, then 64..127
  uint8_t *tU = tS + L::kS;              // U^T as [R][token]
  uint8_t *tCf = tU + L::kU;             // Cf^T, the same layout
  uint64_t *landed = reinterpret_cast<uint64_t *>(tCf + L::kCf);  // TMA -> MMA
  uint64_t *sfree = landed + kLand;                                  // MMA -> TMA
  // per chunk: S tile written (all epilogue warps) -> P = [Q; W] S^T done ->
  // Cf tile written (W-row warps) -> state update product done; U tile
  // written (W-row warps) and the previous chunk's output read (Q-row warps)
  // -> A U done
  uint64_t *s_ready = sfree + kLand, *p_done = s_ready + 1, *cf_ready = s_ready + 2, *s_acc_done = s_ready + 3,
           *u_ready = s_ready + 4, *o_free = s_ready + 5, *o_done = s_ready + 6, *fin = s_ready + 7,
           *redbar = s_ready + 8;  // the epilogue warps' tile-maximum reductions
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(s_ready + 9);
  volatile uint32_t *abort_flag = tmem_holder + 1;
  float *red = reinterpret_cast<float *>(s_ready + 10);  // two buffers of eight

  constexpr int NSL = kD / R;
  const int h = blockIdx.x / NSL, r0 = (blockIdx.x % NSL) * R;
  const int kh = h / (a.Hv / a.Hk);
  const int nc = a.Tp / kC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kLand; ++s) {
      mbar_init(landed + s, 1);
      mbar_init(sfree + s, 1);
    }
    mbar_init(s_ready, 32 * kEpiWarps);
    mbar_init(p_done, 1);
    mbar_init(cf_ready, 16 * kEpiWarps);
    mbar_init(s_acc_done, 1);
    mbar_init(u_ready, 16 * kEpiWarps);
    mbar_init(o_free, 16 * kEpiWarps);
    mbar_init(o_done, 1);
    mbar_init(fin, 1);
    mbar_init(redbar, kEpiWarps);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kEpiWarps) {
    tmem_alloc(tmem_holder, 256);
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
    // every lane is d_k = e of the state update. Operand tiles carry a
    // power-of-two scale each: q, k and A the fixed 2^14, the chunk's W rows
    // the scale chunk_prep chose for them, S and U (Cf shares U's) one found
    // here from the tile's largest magnitude; the accumulators are unscaled
    // exactly by the inverse powers of two.
    constexpr int RH = R / 2;
    const int qt = warp & 3, hf = warp >> 2;
    const bool wrow = qt >= 2;
    const int e = 32 * qt + lane, i = e & 63;
    const uint32_t lane_base = tmem + ((uint32_t)(qt * 32) << 16) + RH * hf;
    float Sv[RH];  // S[r0 + RH hf + r][e]
#pragma unroll
    for (int r = 0; r < RH; ++r)
      Sv[r] = state_load(a.ssm, a.state_bf16, ((size_t)h * kD + r0 + RH * hf + r) * kD + e);
    float pq[RH];       // q rows: e^Gamma_i (S q_i) of the chunk whose output is pending
    float iO = 1.0f;    // and the inverse scale of its A U
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
        for (int k = 0; k < RH; ++k) ov[k] = fmaf(__uint_as_float(oa[k]) + __uint_as_float(oa1[k]), iO, pq[k]);
#pragma unroll
        for (int k = 0; k < RH; k += 4)
          *reinterpret_cast<float4 *>(op + k) = make_float4(ov[k], ov[k + 1], ov[k + 2], ov[k + 3]);
      }
      return true;
    };
    // A chunk's scalars (largest |Ut|, W scale, Gamma_i, Gamma_64) and, in the
    // W-row warps, its Ut row are loaded one chunk ahead: their latency from
    // L2 would otherwise sit on the chain from one chunk to the next.
    float n_um = 0.0f, n_ws = 1.0f, n_gi = 0.0f, n_gC = 0.0f;
    float4 n_ut[RH / 4];
    auto load_next = [&](int cc) {
      const size_t hc = (size_t)h * nc + cc;
      n_um = a.Umax[hc];
      n_ws = a.Wsc[hc];
      n_gi = a.Gam[hc * kC + i];
      n_gC = a.Gam[hc * kC + kC - 1];
      if (wrow) {
        const float4 *up = reinterpret_cast<const float4 *>(a.Ut + (hc * kC + i) * kD + r0 + RH * hf);
#pragma unroll
        for (int j = 0; j < RH / 4; ++j) n_ut[j] = up[j];
      }
    };
    if (nc > 0) load_next(0);
    for (int c = 0; c < nc; ++c) {
      const float umax = n_um, wsc = n_ws, gi = n_gi, gC = n_gC;
      float ut[RH];
#pragma unroll
      for (int j = 0; j < RH / 4; ++j) {
        ut[4 * j] = n_ut[j].x; ut[4 * j + 1] = n_ut[j].y; ut[4 * j + 2] = n_ut[j].z; ut[4 * j + 3] = n_ut[j].w;
      }
      // (a) S -> the B operand of P (thread e owns column e of its rows), with
      // the scale of the slice's largest |S|. U's scale (Cf shares it) comes
      // from a bound known here, |U| <= max|Ut| + d max|W| max|S| with
      // max|W| < 2^14 / Wsc: a loose bound costs no precision while the
      // scaled tile's largest value stays above 2^-3, so no reduction over U
      // (which would hold the W-row warps until the q-row warps are free).
      float sS, sU;
      {
        float mx = 0.0f;
#pragma unroll
        for (int r = 0; r < RH; ++r) mx = fmaxf(mx, fabsf(Sv[r]));
        float smax;
        if (!epi_max(mx, red + 8 * (c & 1), redbar, (uint32_t)(c & 1), abort_flag, a.status, smax)) {
          ok = false;
          break;
        }
        sS = fp16_scale_for(smax);
        sU = fp16_scale_for(fmaf((float)kD * kFixedScale * inv_pow2(wsc), smax, umax));
        put_split_rows<R, RH>(tS + (qt >> 1) * L::kSub, RH * hf, 32 * (qt & 1) + lane, Sv, sS, lane);
        fence_async_shared();
        tc_fence_before();
        mbar_arrive(s_ready);
      }
      if (c + 1 < nc) load_next(c + 1);
      const float iS = inv_pow2(sS);
      if (!wrow && c > 0 && !emit_o(c - 1)) { ok = false; break; }
      if (wrow) {
        // (b) W rows: U = Ut - W S^T, the update coefficients Cf = e^(Gamma_64 - Gamma_i) U
        const float iWS = iS * inv_pow2(wsc);
        const float dc = expf(gC - gi);
        if (!warp_wait(p_done, (uint32_t)(c & 1), abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t pr[RH], pr1[RH];
        tmem_ld16(lane_base, pr);
        tmem_ld16(lane_base + R, pr1);
        tmem_ld_wait();
        float u[RH], cf[RH];
#pragma unroll
        for (int k = 0; k < RH; ++k) {
          u[k] = fmaf(-(__uint_as_float(pr[k]) + __uint_as_float(pr1[k])), iWS, ut[k]);
          cf[k] = dc * u[k];
        }
        // Cf first: the state update is the next chunk's dependency
        put_split_rows<R, RH>(tCf, RH * hf, i, cf, sU, lane);
        fence_async_shared();
        tc_fence_before();
        mbar_arrive(cf_ready);
        // the U tile is free once the previous chunk's A U is done
        if (c > 0 && !warp_wait(o_done, (uint32_t)((c - 1) & 1), abort_flag, a.status)) { ok = false; break; }
        put_split_rows<R, RH>(tU, RH * hf, i, u, sU, lane);
        fence_async_shared();
        mbar_arrive(u_ready);
      } else {
        // (b) q rows: e^Gamma_i (S q_i), kept until the chunk's A U is done
        const float di = expf(gi) * (iS * (1.0f / kFixedScale));
        if (!warp_wait(p_done, (uint32_t)(c & 1), abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t pr[RH], pr1[RH];
        tmem_ld16(lane_base, pr);
        tmem_ld16(lane_base + R, pr1);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < RH; ++k) pq[k] = di * (__uint_as_float(pr[k]) + __uint_as_float(pr1[k]));
      }
      const float iK = (1.0f / kFixedScale) * inv_pow2(sU);  // K^T Cf and A U: 2^14 s_U
      iO = iK;
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
        for (int k = 0; k < RH; ++k)
          Sv[k] = fmaf(dC, Sv[k], (__uint_as_float(sa[k]) + __uint_as_float(sa1[k])) * iK);
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
      const uint32_t idesc = idesc_f16(2 * R);
      const uint32_t bS = smem_u32(tS), bU = smem_u32(tU), bC = smem_u32(tCf);
      uint32_t u = 0, ug = 0;
      bool ok = true;
      // use u: the A operand in ring slot u % kLand, landed by TMA
      auto take = [&](uint32_t &slot) -> bool {
        const int t = (int)(u % kLand);
        if (!wait_or_abort(landed + t, (u / kLand) & 1u, abort_flag, a.status)) return false;
        tc_fence_after();
        slot = smem_u32(ring + t * kLandBytes);
        ++u;
        return true;
      };
      // A chunk's slots are released together once its state-update product
      // has completed, so the TMA refills land while the epilogue updates the
      // state rather than under the MMAs (measured 2.26 -> 2.22 ms at
      // T = 16384); a chunk holds at most kUsesPerChunk <= kLand slots.
      auto give_all = [&]() {
        for (; ug < u; ++ug) tc_commit(sfree + (ug % kLand));
      };
      // O = A U of chunk cc, once its U tile is written and the q rows have
      // read chunk cc - 1's O
      auto au = [&](int cc) -> bool {
        if (!wait_or_abort(u_ready, (uint32_t)(cc & 1), abort_flag, a.status)) return false;
        if (cc > 0 && !wait_or_abort(o_free, (uint32_t)((cc - 1) & 1), abort_flag, a.status)) return false;
        tc_fence_after();
        uint32_t acol;
        if (!take(acol)) return false;
        mma_split(tmem + 2 * R, acol, [&](int j) { return desc_sw128(bU) + 2 * j; }, idesc, true);
        tc_commit(o_done);
        return true;
      };
      for (int c = 0; c < nc && ok; ++c) {
        if (!wait_or_abort(s_ready, (uint32_t)(c & 1), abort_flag, a.status)) break;
        tc_fence_after();
        // P = [Q; W] S^T: d_k 0..63, then 64..127 (S sub-tile hk)
        for (int hk = 0; hk < 2; ++hk) {
          uint32_t acol;
          if (!take(acol)) { ok = false; break; }
          mma_split(tmem, acol, [&](int j) { return desc_sw128(bS + hk * L::kSub) + 2 * j; }, idesc, hk == 0);
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
          mma_split(tmem + 4 * R, acol, [&](int j) { return desc_sw128(bC) + 2 * j; }, idesc, true);
        }
        tc_commit(s_acc_done);
        give_all();
        if (c == nc - 1) au(c);
      }
      give_all();
      // every MMA issued has completed before the CTA may leave
      tc_commit(fin);
      mbar_wait(fin, 0u);
    }
  } else if (warp == kEpiWarps + 1) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t total = (uint32_t)nc * kUsesPerChunk;
      const int qlo = a.Hk * a.Tp, wlo = a.Hv * a.Tp;  // rows of the lo blocks
      const int klo = a.Hk * nc * kD;
      for (uint32_t u = 0; u < total; ++u) {
        const int s = (int)(u % kLand);
        if (u >= (uint32_t)kLand && !wait_or_abort(sfree + s, ((u / kLand) - 1u) & 1u, abort_flag, a.status)) break;
        int q, c;
        ring_use(u, nc, q, c);
        if (q == 0 && c + 1 < nc) {  // the next chunk's operands and Ut rows into L2
          const size_t n = (size_t)c + 1;
          const size_t qrow = (size_t)kh * a.Tp + n * kC, wrow = (size_t)h * a.Tp + n * kC;
          prefetch_l2(a.Qs + qrow * kD, kC * kD * 2);
          prefetch_l2(a.Qs + (qrow + qlo) * kD, kC * kD * 2);
          prefetch_l2(a.Ws + wrow * kD, kC * kD * 2);
          prefetch_l2(a.Ws + (wrow + wlo) * kD, kC * kD * 2);
          prefetch_l2(a.As + wrow * kC, kC * kC * 2);
          prefetch_l2(a.As + (wrow + wlo) * kC, kC * kC * 2);
          const size_t krow = ((size_t)kh * nc + n) * kD;
          prefetch_l2(a.KTs + krow * kC, kD * kC * 2);
          prefetch_l2(a.KTs + (krow + klo) * kC, kD * kC * 2);
          prefetch_l2(a.Ut + wrow * kD, kC * kD * 4);
        }
        uint8_t *hi = ring + s * kLandBytes, *lo = hi + kLoOff;
        mbar_arrive_expect_tx(landed + s, q == 3 ? kLandBytes / 2 : kLandBytes);
        if (q < 2) {         // [Q; W], d_k columns 64 q .. 64 q + 63: rows 0..63 q, 64..127 W
          const int yq = kh * a.Tp + c * kC, yw = h * a.Tp + c * kC;
          tma_load_2d(hi, &tmQ, 128 * q, yq, landed + s);
          tma_load_2d(hi + 64 * 128, &tmW, 128 * q, yw, landed + s);
          tma_load_2d(lo, &tmQ, 128 * q, qlo + yq, landed + s);
          tma_load_2d(lo + 64 * 128, &tmW, 128 * q, wlo + yw, landed + s);
        } else if (q == 2) { // K^T: 128 rows of d_k
          const int yk = (kh * nc + c) * kD;
          tma_load_2d(hi, &tmKT, 0, yk, landed + s);
          tma_load_2d(lo, &tmKT, 0, klo + yk, landed + s);
        } else {             // A: 64 rows (the slot's rows 64..127 are never read out)
          const int ya = h * a.Tp + c * kC;
          tma_load_2d(hi, &tmA, 0, ya, landed + s);
          tma_load_2d(lo, &tmA, 0, wlo + ya, landed + s);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kEpiWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

// The tcgen05 chunk scan for d = 128 (slices of 32 rows of d_v per CTA).
// Needs chunk_prep_tc's split Qs (from prep), Ws, As, KTs, its FP32 Ut, Gam and the per-chunk Wsc, Umax.
cudaError_t launch_chunk_scan_umma(const PrefillArgs &a, cudaStream_t stream) {
  constexpr int R = 32;
  if (a.D != kD || !a.Qs || !a.Ws || !a.As || !a.KTs || !a.Wsc || !a.Umax) return cudaErrorInvalidValue;
  const uint64_t nc = (uint64_t)a.Tp / kC;
  // FP16 operands as 2-D byte tensors; boxes of 128-byte rows (64 FP16)
  CUtensorMap mQ, mW, mA, mKT;
  if (!make_map(&mQ, a.Qs, 2ull * a.Hk * a.Tp, kD * 2, kC, 128, true) ||
      !make_map(&mW, a.Ws, 2ull * a.Hv * a.Tp, kD * 2, kC, 128, true) ||
      !make_map(&mA, a.As, 2ull * a.Hv * a.Tp, kC * 2, kC, 128, true) ||
      !make_map(&mKT, a.KTs, 2ull * a.Hk * nc * kD, kC * 2, kD, 128, true))
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
