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
// The state lives in the registers of the four epilogue warps, transposed:
// thread e (TMEM lane e) holds S[r0 + r][e] for the slice's R rows, which is
// exactly the lane of the update's accumulator, so no state element moves
// between threads. Every product runs in split TF32: x = hi + lo and
// a.b ~ lo.hi + hi.lo + hi.hi, accumulated in FP32, about 21 of FP32's 24
// mantissa bits -- the arithmetic of the warp-level chunk scan, here as
// tcgen05 MMAs reading both operands from shared memory (K-major, 128-byte
// swizzle). For the operands the CTA computes (S, U, Cf), hi = TF32(x) and
// lo = TF32(x - hi) by round-to-nearest; for the streamed chunk operands hi is
// x itself read as TF32 (its low 13 bits dropped) and lo = x - trunc(x).
//
// Warp roles (448 threads):
//   warps 0..3   epilogue: TMEM -> registers, U / Cf / S operand tiles (split)
//                into shared memory, outputs, the state
//   warp 4       TMEM allocation; one thread issues the MMAs
//   warp 5       one thread streams the chunk's [Q; W], A and K^T tiles by
//                TMA (128-byte swizzle) into a ring of 32 KB slots, and asks
//                L2 to prefetch the next chunk
//   warps 6..13  write the lo part of each landed FP32 tile beside it (the
//                tile itself is the hi part: the tensor core reads an FP32
//                word as TF32 by dropping its 13 low mantissa bits)
// Every mbarrier wait is bounded; a wait that gives up sets the status word
// (GDN_E_TIMEOUT) and a shared abort flag that ends every role's loop.
#include <cuda.h>

#include "tc.cuh"

namespace gdn {

namespace {

constexpr int kC = 64, kD = 128;
constexpr int kSlots = 5;                 // operand ring slots
constexpr int kHalf = 128 * 128;          // bytes of one [128 rows][32 floats] tile
constexpr int kSplitWarps = 8;
constexpr int kScanThreads = 32 * (6 + kSplitWarps);
constexpr int kUsesPerChunk = 7;          // ring uses: 4 of [Q; W], 1 of A (both halves), 2 of K^T

template <int R>
struct ScanLayout {
  static constexpr int kSub = R * 128;                  // one [R][32 floats] sub-tile
  static constexpr int kRing = kSlots * 2 * kHalf;      // hi + lo per slot
  static constexpr int kS = 2 * 4 * kSub;               // S hi, lo: four d_k sub-tiles each
  static constexpr int kU = 2 * 2 * kSub;               // U^T hi, lo: two token sub-tiles each
  static constexpr int kCf = kU;                        // Cf^T hi, lo
  static constexpr int kBars = 256;
  static constexpr int kBytes = 1024 + kRing + kS + kU + kCf + kBars;
  static_assert(kSub % 1024 == 0, "sub-tiles stay 1024-byte aligned");
  static_assert(kBytes <= 227 * 1024, "one CTA per SM");
};

GDN_DEV uint32_t tf32_bits(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
GDN_DEV void split_hi_lo(float x, uint32_t &hi, uint32_t &lo) {
  hi = tf32_bits(x);
  lo = tf32_bits(x - __uint_as_float(hi));
}
// byte offset of element (row, col) in a [rows][32 floats] tile, 128-byte swizzle
GDN_DEV uint32_t sw_off(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 2) ^ (row & 7)) << 4) | ((col & 3) << 2)));
}
// Instruction descriptor of kind::tf32: FP32 accumulator, TF32 A and B, both
// K-major, M = 128, N = n.
GDN_DEV uint32_t idesc_tf32(int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
GDN_DEV void mma_tf32(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (+)= A B^T in split precision over one 32-wide K sub-tile (four K = 8 steps):
// lo.hi, hi.lo, hi.hi per step; `first` starts the accumulator.
GDN_DEV void mma_split_sub(uint32_t d, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl, uint32_t idesc, bool first) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    mma_tf32(d, al + 2 * k, bh + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
    mma_tf32(d, ah + 2 * k, bl + 2 * k, idesc, 1u);
    mma_tf32(d, ah + 2 * k, bh + 2 * k, idesc, 1u);
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
  uint8_t *sS = sm + L::kRing;           // S as [R][d_k]: hi sub-tiles 0..3, lo 4..7
  uint8_t *sU = sS + L::kS;              // U^T as [R][token]: hi 0..1, lo 2..3
  uint8_t *sCf = sU + L::kU;             // Cf^T, the same layout
  uint64_t *landed = reinterpret_cast<uint64_t *>(sCf + L::kCf);  // TMA -> splitters
  uint64_t *full = landed + kSlots;                                  // splitters -> MMA
  uint64_t *empty = full + kSlots;                                   // MMA -> TMA
  uint64_t *s_ready = empty + kSlots, *p_done = s_ready + 1, *u_ready = s_ready + 2, *acc_done = s_ready + 3,
           *fin = s_ready + 4;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(s_ready + 5);
  volatile uint32_t *abort_flag = tmem_holder + 1;

  constexpr int NSL = kD / R;
  const int h = blockIdx.x / NSL, r0 = (blockIdx.x % NSL) * R;
  const int kh = h / (a.Hv / a.Hk);
  const int nc = a.Tp / kC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // the second half of the A product reads 64 rows past its operand (rows
  // whose products are never read); the ring starts zeroed so they are finite
  for (int i = tid; i < L::kRing / 16; i += kScanThreads) reinterpret_cast<uint4 *>(ring)[i] = make_uint4(0, 0, 0, 0);
  fence_async_shared();
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(landed + s, 1);
      mbar_init(full + s, 32 * kSplitWarps);
      mbar_init(empty + s, 1);
    }
    mbar_init(s_ready, 128);
    mbar_init(p_done, 1);
    mbar_init(u_ready, 128);
    mbar_init(acc_done, 1);
    mbar_init(fin, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_holder, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp < 4) {
    // ------------------------------------------------ epilogue: thread e = TMEM lane e
    const int e = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float Sv[R];  // S[r0 + r][e]
#pragma unroll
    for (int r = 0; r < R; ++r) Sv[r] = state_load(a.ssm, a.state_bf16, ((size_t)h * kD + r0 + r) * kD + e);
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
      // (a) S -> the B operand of P (thread e owns column e of every row)
      {
        uint8_t *hi = sS + warp * L::kSub, *lo = sS + (4 + warp) * L::kSub;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          uint32_t vh, vl;
          split_hi_lo(Sv[r], vh, vl);
          const uint32_t off = sw_off(r, lane);
          *reinterpret_cast<uint32_t *>(hi + off) = vh;
          *reinterpret_cast<uint32_t *>(lo + off) = vl;
        }
        fence_async_shared();
        tc_fence_before();
        mbar_arrive(s_ready);
      }
      const float *gam = a.Gam + ((size_t)h * nc + c) * kC;
      const int i = e & 63;
      const float gi = gam[i], gC = gam[kC - 1];
      // (b) rows 64..127 of P are W S^T: U = Ut - W S^T and the update coefficients
      if (e >= 64) {
        float ut[R];
        const float4 *up = reinterpret_cast<const float4 *>(a.Ut + (((size_t)h * nc + c) * kC + i) * kD + r0);
#pragma unroll
        for (int j = 0; j < R / 4; ++j) {
          const float4 v = up[j];
          ut[4 * j] = v.x; ut[4 * j + 1] = v.y; ut[4 * j + 2] = v.z; ut[4 * j + 3] = v.w;
        }
        const float dc = expf(gC - gi);
        if (!warp_wait(p_done, (uint32_t)(c & 1), abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        const int sub = i >> 5, col = i & 31;
        uint8_t *uh = sU + sub * L::kSub, *ul = sU + (2 + sub) * L::kSub;
        uint8_t *ch = sCf + sub * L::kSub, *cl = sCf + (2 + sub) * L::kSub;
#pragma unroll
        for (int p0 = 0; p0 < R; p0 += 16) {
          uint32_t pr[16];
          tmem_ld16(lane_base + p0, pr);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int r = p0 + k;
            const float u = ut[r] - __uint_as_float(pr[k]);
            const uint32_t off = sw_off(r, col);
            uint32_t vh, vl;
            split_hi_lo(u, vh, vl);
            *reinterpret_cast<uint32_t *>(uh + off) = vh;
            *reinterpret_cast<uint32_t *>(ul + off) = vl;
            split_hi_lo(dc * u, vh, vl);
            *reinterpret_cast<uint32_t *>(ch + off) = vh;
            *reinterpret_cast<uint32_t *>(cl + off) = vl;
          }
        }
        fence_async_shared();
      }
      tc_fence_before();
      mbar_arrive(u_ready);
      // (c) outputs of rows 0..63 and the state update
      if (!warp_wait(acc_done, (uint32_t)(c & 1), abort_flag, a.status)) { ok = false; break; }
      tc_fence_after();
      if (e < 64) {
        const int t = c * kC + i;
        const float di = expf(gi);
        float *op = a.o + ((size_t)t * a.Hv + h) * kD + r0;
#pragma unroll
        for (int p0 = 0; p0 < R; p0 += 16) {
          uint32_t pq[16], oa[16];
          tmem_ld16(lane_base + p0, pq);
          tmem_ld16(lane_base + R + p0, oa);
          tmem_ld_wait();
          if (t < a.T) {
#pragma unroll
            for (int k = 0; k < 16; k += 4)
              *reinterpret_cast<float4 *>(op + p0 + k) =
                  make_float4(fmaf(di, __uint_as_float(pq[k]), __uint_as_float(oa[k])),
                              fmaf(di, __uint_as_float(pq[k + 1]), __uint_as_float(oa[k + 1])),
                              fmaf(di, __uint_as_float(pq[k + 2]), __uint_as_float(oa[k + 2])),
                              fmaf(di, __uint_as_float(pq[k + 3]), __uint_as_float(oa[k + 3])));
          }
        }
      }
      const float dC = expf(gC);
#pragma unroll
      for (int p0 = 0; p0 < R; p0 += 16) {
        uint32_t sa[16];
        tmem_ld16(lane_base + 2 * R + p0, sa);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) Sv[p0 + k] = fmaf(dC, Sv[p0 + k], __uint_as_float(sa[k]));
      }
    }
    if (ok) {
#pragma unroll
      for (int r = 0; r < R; ++r) state_store(a.ssm, a.state_bf16, ((size_t)h * kD + r0 + r) * kD + e, Sv[r]);
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_tf32(R);
      uint32_t u = 0;
      bool ok = true;
      for (int c = 0; c < nc && ok; ++c) {
        if (!wait_or_abort(s_ready, (uint32_t)(c & 1), abort_flag, a.status)) break;
        tc_fence_after();
        // P = [Q; W] S^T over four 32-wide d_k sub-tiles
        for (int q = 0; q < 4; ++q, ++u) {
          const int s = (int)(u % kSlots);
          if (!wait_or_abort(full + s, (u / kSlots) & 1u, abort_flag, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + s * 2 * kHalf);
          const uint32_t sb = smem_u32(sS + q * L::kSub);
          mma_split_sub(tmem, desc_sw128(sa), desc_sw128(sa + kHalf), desc_sw128(sb), desc_sw128(sb + 4 * L::kSub),
                        idesc, q == 0);
          tc_commit(empty + s);
        }
        if (!ok) break;
        tc_commit(p_done);
        if (!wait_or_abort(u_ready, (uint32_t)(c & 1), abort_flag, a.status)) break;
        tc_fence_after();
        // O = A U (one slot: A's token halves as rows 0..63 and 64..127), then
        // S_acc = K^T Cf (K^T in two token halves)
        for (int q = 0; q < 3; ++q, ++u) {
          const int s = (int)(u % kSlots);
          if (!wait_or_abort(full + s, (u / kSlots) & 1u, abort_flag, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + s * 2 * kHalf);
          if (q == 0) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t ar = sa + hh * (64 * 128), sb = smem_u32(sU + hh * L::kSub);
              mma_split_sub(tmem + R, desc_sw128(ar), desc_sw128(ar + kHalf), desc_sw128(sb),
                            desc_sw128(sb + 2 * L::kSub), idesc, hh == 0);
            }
          } else {
            const uint32_t sb = smem_u32(sCf + (q - 1) * L::kSub);
            mma_split_sub(tmem + 2 * R, desc_sw128(sa), desc_sw128(sa + kHalf), desc_sw128(sb),
                          desc_sw128(sb + 2 * L::kSub), idesc, q == 1);
          }
          tc_commit(empty + s);
        }
        if (!ok) break;
        tc_commit(acc_done);
      }
      // every MMA issued has completed before the CTA may leave
      tc_commit(fin);
      mbar_wait(fin, 0u);
    }
  } else if (warp == 5) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t total = (uint32_t)nc * kUsesPerChunk;
      for (uint32_t u = 0; u < total; ++u) {
        const int s = (int)(u % kSlots);
        if (u >= (uint32_t)kSlots && !wait_or_abort(empty + s, ((u / kSlots) - 1u) & 1u, abort_flag, a.status)) break;
        const int c = (int)(u / kUsesPerChunk), q = (int)(u % kUsesPerChunk);
        if (q == 0 && c + 1 < nc) {  // the next chunk's operands and Ut rows into L2
          const int n = c + 1;
          prefetch_l2(a.qn + ((size_t)kh * a.Tp + (size_t)n * kC) * kD, kC * kD * 4);
          prefetch_l2(a.W + ((size_t)h * nc + n) * kC * kD, kC * kD * 4);
          prefetch_l2(a.Am + ((size_t)h * nc + n) * kC * kC, kC * kC * 4);
          prefetch_l2(a.KT + ((size_t)kh * nc + n) * kD * kC, kD * kC * 4);
          prefetch_l2(a.Ut + ((size_t)h * nc + n) * kC * kD, kC * kD * 4);
        }
        uint8_t *hi = ring + s * 2 * kHalf;
        mbar_arrive_expect_tx(landed + s, kHalf);
        if (q < 4) {         // [Q; W], d_k columns 32 q .. 32 q + 31
          tma_load_2d(hi, &tmQ, q * 128, kh * a.Tp + c * kC, landed + s);
          tma_load_2d(hi + 64 * 128, &tmW, q * 128, (h * nc + c) * kC, landed + s);
        } else if (q == 4) { // A, token halves as rows 0..63 and 64..127
          tma_load_2d(hi, &tmA, 0, (h * nc + c) * kC, landed + s);
          tma_load_2d(hi + 64 * 128, &tmA, 128, (h * nc + c) * kC, landed + s);
        } else {             // K^T, tokens 32 (q - 5) .. + 31
          tma_load_2d(hi, &tmKT, (q - 5) * 128, (kh * nc + c) * kD, landed + s);
        }
      }
    }
  } else {
    // ------------------------------------------------ splitters (warps 6..13)
    // each thread takes the 16-byte pieces id = lt + 256 k of the slot's
    // [128 rows][32 floats] tile (row id / 8, 16-byte chunk id % 8) and writes
    // lo = x - trunc(x) at the same place of the lo tile
    const int lt = tid - 192;
    const uint32_t total = (uint32_t)nc * kUsesPerChunk;
    for (uint32_t u = 0; u < total; ++u) {
      const int s = (int)(u % kSlots);
      if (!warp_wait(landed + s, (u / kSlots) & 1u, abort_flag, a.status)) break;
      uint8_t *hi = ring + s * 2 * kHalf, *lo = hi + kHalf;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int id = lt + 256 * k, row = id >> 3, c4 = id & 7;
        const uint32_t off = (uint32_t)(row * 128 + ((c4 ^ (row & 7)) << 4));
        const float4 x = *reinterpret_cast<const float4 *>(hi + off);
        uint4 vl;
        vl.x = __float_as_uint(x.x - __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u));
        vl.y = __float_as_uint(x.y - __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u));
        vl.z = __float_as_uint(x.z - __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u));
        vl.w = __float_as_uint(x.w - __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u));
        *reinterpret_cast<uint4 *>(lo + off) = vl;
      }
      fence_async_shared();
      mbar_arrive(full + s);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
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
