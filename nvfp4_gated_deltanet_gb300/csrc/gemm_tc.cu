// Block-scaled W4A4 GEMM on the 5th-generation tensor cores:
// tcgen05.mma .kind::mxf4nvf4 .scale_vec::4X (E2M1 operands, one UE4M3 scale
// per 16 elements), FP32 accumulators in tensor memory.
//
//   D[m][n] = sum_k W_hat[m][k] * X_hat[n][k],   stored as C[n][m]
//
// W (the weights) is the MMA's A operand: 128 rows per CTA tile. X (the
// activations: decode rows or prompt tokens) is the B operand: BN rows. Both
// are K-major NVFP4 with row-major codes [rows][K/2] and scales [rows][K/16].
//
// Per CTA (6 warps):
//   warp 0      TMA producer: code tiles (128 B x rows, 128-byte swizzle) and
//               the scales of this K tile (tiled atoms, or row-major rows),
//               into a ring of S stages
//   warp 1      tensor-memory allocation, then one thread issues tcgen05.mma,
//               committing each stage back to the producer
//   warps 2..5  put each stage's scales into TMEM with tcgen05.st (each warp
//               its lane quarter; row-major scale rows are first rearranged
//               into 512-byte atoms, row r at byte (r%32)*16 + (r/32)*4 +
//               k-block, the layout tcgen05.cp.32x128b.warpx4 would copy), so
//               the MMA thread issues nothing but MMAs; then the epilogue:
//               TMEM -> registers -> scaled BF16/FP32 stores
// Split-K over a thread-block cluster of KS CTAs: ranks != 0 push their FP32
// partial tile into rank 0's shared memory before one cluster barrier; rank 0
// adds them in rank order (deterministic, no atomics).
//
// Decode form (b_bf16 set): the weight tiles of every K step of the CTA are
// requested before griddepcontrol.wait, and warps 2..5 quantise the BF16
// activation rows themselves, after the wait, into the swizzled B tiles and
// the tiled scale atoms -- no separate quantisation kernel, no B loads.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cooperative_groups.h>

#include "tc.cuh"

namespace cg = cooperative_groups;

namespace gdn {

// ---------------------------------------------------------------- tensor maps (host)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D byte tensor [rows][row_bytes] (row stride = row_bytes), box [box_rows][box_bytes].
bool make_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t row_bytes, uint32_t box_rows,
              uint32_t box_bytes, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int kThreads = 192;
constexpr int kATile = 128 * 128;  // 128 rows x 128 bytes (256 E2M1 values)
constexpr int kSFAtom = 512;       // scales of 128 rows x one K=64 step
constexpr int kTmemCols = 256;     // accumulator at column 0, scales from column 128

// ---------------------------------------------------------------- PTX wrappers
GDN_DEV void tc_cp_scales(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
GDN_DEV void tc_mma_nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

// 32 rows x 16 bytes, no swizzle: 8-row core matrices 128 bytes apart.
GDN_DEV uint64_t desc_scales(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// Instruction descriptor: E2M1 x E2M1, K-major A and B, UE4M3 scales,
// N = BN, M = 128, dense.
template <int BN>
GDN_DEV uint32_t idesc_nvf4() {
  return (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | (0u << 23) | ((uint32_t)(128 >> 4) << 24);
}

template <int BN>
struct Layout {
  static constexpr int kB = BN * 128;                 // B codes
  static constexpr int kSfaRows = 128 * 16;           // row-major scale rows of this K tile
  static constexpr int kSfbRows = (BN * 16 + 127) / 128 * 128;
  static constexpr int kAtoms = 4 * kSFAtom;          // 4 K=64 steps
  static constexpr int kStage = (kATile + kB + kSfaRows + kSfbRows + 2 * kAtoms + 1023) / 1024 * 1024;
  static_assert(kATile % 1024 == 0 && kB % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
};

template <int BN, int KS, int S>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB, TcArgs a) {
  using L = Layout<BN>;
  // accumulators in tensor memory: one, or four for narrow tiles (columns
  // 0 .. 4*BN-1; the scales start at column 128)
  constexpr int kAcc = BN <= 32 ? 4 : 1;
  static_assert(kAcc * BN <= 128, "accumulators overlap the scale columns");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char *stage0 = sm;
  float *part = reinterpret_cast<float *>(sm + (size_t)S * L::kStage);
  uint64_t *full = reinterpret_cast<uint64_t *>(part + (KS > 1 ? (KS - 1) * 128 * BN : 0));
  uint64_t *sfready = full + S;  // [S] the stage's scales are in TMEM (one arrival per warp 2..5)
  uint64_t *empty = sfready + S;
  uint64_t *accum = empty + S;
  uint64_t *bready = accum + 1;  // decode form: the quantised B tiles are in place
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bready + 1);
  auto stA = [&](int s) { return stage0 + (size_t)s * L::kStage; };
  auto stB = [&](int s) { return stA(s) + kATile; };
  auto stSA = [&](int s) { return stB(s) + L::kB; };
  auto stSB = [&](int s) { return stSA(s) + L::kSfaRows; };
  auto stAtA = [&](int s) { return stSB(s) + L::kSfbRows; };
  auto stAtB = [&](int s) { return stAtA(s) + L::kAtoms; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x / KS, ks = blockIdx.x % KS;
  const int nt = blockIdx.y;
  const int nkt = (a.K >> 8) / KS;
  const int kt0 = ks * nkt;
  const bool bq = a.b_bf16 != nullptr;
  const bool tiled = a.sfa_tiled != nullptr && (a.sfb_tiled != nullptr || bq);
  if (a.early_trigger) pdl_launch_dependents();
  if (bq && (BN != 16 || nkt > S || !a.sfa_tiled || !a.a_const)) {  // host-side contract broken: refuse, uniformly
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) flag_status(a.status, GDN_E_SHAPE);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(sfready + s, 4);
      mbar_init(empty + s, 1);
    }
    mbar_init(accum, 1);
    mbar_init(bready, 128);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t bytes = bq ? kATile + 4 * kSFAtom
                           : tiled ? kATile + L::kB + 2 * 4 * kSFAtom : kATile + L::kB + 128 * 16 + BN * 16;
      const int ksteps = a.K >> 6;
      const int nsf = (nt * BN) >> 7;  // 128-row tile of the activation scales (BN < 128: one N tile)
      auto load_a = [&](int i, int s) {
        if (a.a_tiles)
          bulk_g2s(stA(s), a.a_tiles + ((size_t)mt * (a.K >> 8) + kt0 + i) * kATile, kATile, full + s);
        else
          tma_load_2d(stA(s), &tmA, (kt0 + i) * 128, mt * 128, full + s);
        if (tiled)
          bulk_g2s(stAtA(s), a.sfa_tiled + ((size_t)mt * ksteps + (size_t)(kt0 + i) * 4) * kSFAtom, 4 * kSFAtom, full + s);
        else
          tma_load_2d(stSA(s), &tmSA, (kt0 + i) * 16, mt * 128, full + s);
      };
      auto load_b = [&](int i, int s) {
        tma_load_2d(stB(s), &tmB, (kt0 + i) * 128, nt * BN, full + s);
        if (tiled)
          bulk_g2s(stAtB(s), a.sfb_tiled + ((size_t)nsf * ksteps + (size_t)(kt0 + i) * 4) * kSFAtom, 4 * kSFAtom, full + s);
        else
          tma_load_2d(stSB(s), &tmSB, (kt0 + i) * 16, nt * BN, full + s);
      };
      const int pre = a.a_const ? min(S, nkt) : 0;
      for (int i = 0; i < pre; ++i) {  // weights do not depend on the preceding kernel
        mbar_arrive_expect_tx(full + i, bytes);
        load_a(i, i);
      }
      if (!bq) {
        pdl_wait();
        if (!a.early_trigger) pdl_launch_dependents();
      }
      for (int i = 0; i < (bq ? 0 : pre); ++i) load_b(i, i);
      for (int i = pre; i < nkt; ++i) {
        const int s = i % S, u = i / S;
        if (u > 0 && !mbar_wait(empty + s, (uint32_t)((u - 1) & 1))) { ok = false; break; }
        mbar_arrive_expect_tx(full + s, bytes);
        load_a(i, s);
        load_b(i, s);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4<BN>();
      if (bq && !mbar_wait(bready, 0)) ok = false;
      for (int i = 0; i < (ok ? nkt : 0); ++i) {
        const int s = i % S, u = i / S;
        if (!mbar_wait(full + s, (uint32_t)(u & 1)) || !mbar_wait(sfready + s, (uint32_t)(u & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa = tmem + 128 + 32 * s, sfb = sfa + 16;
        const uint64_t ad = desc_sw128(smem_u32(stA(s))), bd = desc_sw128(smem_u32(stB(s)));
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // K = 64 per MMA: 32 bytes further along the swizzled rows
          // narrow tiles rotate over kAcc accumulators so consecutive MMAs do
          // not wait on each other's result; the epilogue adds them in order
          const int step = i * 4 + j, acc = step % kAcc;
          tc_mma_nvf4(tmem + acc * BN, ad + 2 * j, bd + 2 * j, idesc, sfa + 4 * j, sfb + 4 * j, step >= kAcc);
        }
        tc_commit(empty + s);
      }
      tc_commit(accum);
    }
  } else {
    const int t = threadIdx.x - 64;  // 0..127
    const int qw = warp & 3;         // TMEM lane quarter this warp may access
    // this warp's lane quarter of stage s's scales, from the stage's atoms:
    // per 64-wide K step the 16-byte atom row `lane` (the layout
    // tcgen05.cp.32x128b.warpx4 would give), A at column 128 + 32 s, B 16 on
    auto put_scales = [&](int s) {
      uint32_t va[16], vb[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 x = *reinterpret_cast<const uint4 *>(stAtA(s) + j * kSFAtom + lane * 16);
        const uint4 y = *reinterpret_cast<const uint4 *>(stAtB(s) + j * kSFAtom + lane * 16);
        va[4 * j] = x.x; va[4 * j + 1] = x.y; va[4 * j + 2] = x.z; va[4 * j + 3] = x.w;
        vb[4 * j] = y.x; vb[4 * j + 1] = y.y; vb[4 * j + 2] = y.z; vb[4 * j + 3] = y.w;
      }
      const uint32_t base = tmem + ((uint32_t)(qw * 32) << 16) + 128 + 32 * s;
      tmem_st16(base, va);
      tmem_st16(base + 16, vb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfready + s);
    };
    // ------------------------------------------------ decode form: quantise B
    if constexpr (BN == 16) if (bq) {
      pdl_wait();  // the activation rows come from the preceding kernel
      if (t == 0 && !a.early_trigger) pdl_launch_dependents();
      const float inv6ts = inv6ts_of(a.ts_b);
      bool finite = true;
      // one 32-element piece (two 16-blocks, 16 code bytes) per item: 8 per
      // row of a 256-wide K tile; consecutive threads walk along a row. All
      // of a thread's loads are issued before any quantisation (no load waits
      // behind another), rows' liveness comes from one slot lookup per row.
      // (x rows of padding slots exist in memory: they are read, then dropped)
      constexpr int kMaxItems = (4 * BN * 8 + 127) / 128;
      const int nitems = nkt * BN * 8;
      uint4 xv[kMaxItems][4];
      int slot[kMaxItems];
#pragma unroll
      for (int j = 0; j < kMaxItems; ++j) {
        const int idx = t + j * 128;
        const int i = idx / (BN * 8), r = (idx >> 3) % BN, c = idx & 7;
        const int n = nt * BN + r;
        const bool in = idx < nitems && n < a.Nb;
        slot[j] = in ? (a.b_row_slot ? a.b_row_slot[n] : 0) : -1;
        const uint4 *src = reinterpret_cast<const uint4 *>(a.b_bf16 + (size_t)n * a.K + (size_t)(kt0 + i) * 256 + c * 32);
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) xv[j][q2] = in ? src[q2] : make_uint4(0, 0, 0, 0);
      }
      bool live[kMaxItems];
#pragma unroll
      for (int j = 0; j < kMaxItems; ++j)
        live[j] = slot[j] >= 0 && (a.b_row_slot == nullptr || slot[j] < a.b_num_slots);
#pragma unroll
      for (int j = 0; j < kMaxItems; ++j) {
        const int idx = t + j * 128;
        if (idx >= nitems) break;
        const int i = idx / (BN * 8), r = (idx >> 3) % BN, c = idx & 7;
        uint32_t lo[2] = {0, 0}, hi[2] = {0, 0}, sc[2] = {0, 0};
        if (live[j]) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[16];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              const uint4 w4 = xv[j][half * 2 + q2];
              const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                v[8 * q2 + 2 * k] = __uint_as_float(w[k] << 16);
                v[8 * q2 + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
              }
            }
            finite &= quant_block16(v, a.ts_b, inv6ts, lo[half], hi[half], sc[half]);
          }
        }
        // codes: row r of the tile is 128 bytes, its 16-byte chunks swizzled by r % 8
        *reinterpret_cast<uint4 *>(stB(i) + r * 128 + ((c ^ (r & 7)) << 4)) = make_uint4(lo[0], hi[0], lo[1], hi[1]);
        // scales: blocks 2c, 2c+1 of the tile = K step c/2, blocks (2c)%4, (2c)%4+1
        *reinterpret_cast<uint16_t *>(stAtB(i) + (c >> 1) * kSFAtom + (r & 31) * 16 + ((r & 127) >> 5) * 4 + ((2 * c) & 3)) =
            (uint16_t)(sc[0] | (sc[1] << 8));
      }
      if (!finite && blockIdx.x == 0) flag_status(a.status, GDN_E_NONFINITE);
      fence_async_shared();  // generic-proxy writes -> visible to tcgen05.mma / tcgen05.cp
      mbar_arrive(bready);
    }
    // ------------------------------------------------ scales -> TMEM
    if (tiled) {  // atoms copied in by the producer (and, decode form, B's written above)
      if (bq) asm volatile("bar.sync 1, 128;" ::: "memory");  // every warp's B atoms are in place
      for (int i = 0; i < nkt; ++i) {
        const int s = i % S, u = i / S;
        // lane 0 waits and the warp follows it: the collective TMEM stores run
        // with all 32 lanes (or none)
        const int got = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(full + s, (uint32_t)(u & 1)) : 0, 0);
        __syncwarp();
        if (!got) { ok = false; break; }
        put_scales(s);
      }
    }
    volatile uint32_t *sflag = tmem_holder + 1;
    for (int i = 0; i < (tiled ? 0 : nkt); ++i) {  // row-major scales: rearrange into atoms first
      const int s = i % S, u = i / S;
      // one thread waits, the four warps follow it (the named barriers stay matched)
      if (t == 0) *sflag = mbar_wait(full + s, (uint32_t)(u & 1)) ? 1u : 0u;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (*sflag == 0) { ok = false; break; }
      const uint4 va = *reinterpret_cast<const uint4 *>(stSA(s) + t * 16);
      uint32_t *atA = reinterpret_cast<uint32_t *>(stAtA(s) + (t & 31) * 16 + (t >> 5) * 4);
      atA[0 * kSFAtom / 4] = va.x;
      atA[1 * kSFAtom / 4] = va.y;
      atA[2 * kSFAtom / 4] = va.z;
      atA[3 * kSFAtom / 4] = va.w;
      if (t < BN) {
        const uint4 vb = *reinterpret_cast<const uint4 *>(stSB(s) + t * 16);
        uint32_t *atB = reinterpret_cast<uint32_t *>(stAtB(s) + (t & 31) * 16 + (t >> 5) * 4);
        atB[0 * kSFAtom / 4] = vb.x;
        atB[1 * kSFAtom / 4] = vb.y;
        atB[2 * kSFAtom / 4] = vb.z;
        atB[3 * kSFAtom / 4] = vb.w;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the stage's atoms are complete
      put_scales(s);
    }
    // ------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    float acc[BN];
    if (ok && mbar_wait(accum, 0)) {
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float part4[kAcc][16];
#pragma unroll
        for (int p = 0; p < kAcc; ++p) {
          uint32_t r[16];
          tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + p * BN + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) part4[p][c] = __uint_as_float(r[c]);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float v = part4[0][c];
          if (kAcc == 4) v = (part4[0][c] + part4[1][c]) + (part4[2][c] + part4[3][c]);
          acc[c0 + c] = v;
        }
      }
    } else {
      ok = false;
#pragma unroll
      for (int c = 0; c < BN; ++c) acc[c] = 0.0f;
    }
    if (KS > 1 && ks != 0) {
      float *dst = cg::this_cluster().map_shared_rank(part, 0) + (size_t)(ks - 1) * 128 * BN;
#pragma unroll
      for (int c = 0; c < BN; ++c) dst[c * 128 + row] = acc[c];
    }
    if (KS > 1) cg::this_cluster().sync();  // partials have landed in rank 0
    if (KS == 1 || ks == 0) {
      for (int p = 0; p < KS - 1; ++p)
#pragma unroll
        for (int c = 0; c < BN; ++c) acc[c] += part[((size_t)p * BN + c) * 128 + row];
      const int m = mt * 128 + row;
      const float ts = (m < a.a_split ? a.ts_a0 : a.ts_a1) * a.ts_b;
      // Stage the tile as [BN][128] in shared memory (the pipeline stages are
      // idle once the accumulator is complete), then write whole rows of C
      // with 16-byte stores.
      const int esz = a.c_is_bf16 ? 2 : 4;
      const bool vec = (a.ldc * esz) % 16 == 0 && (a.Ma % 8) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.c) & 15u) == 0;
      if (vec) {
        unsigned char *tile = stage0;
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const float y = acc[c] * ts;
          if (a.c_is_bf16)
            reinterpret_cast<uint16_t *>(tile)[c * 128 + row] = f32_to_bf16_bits(y);
          else
            reinterpret_cast<float *>(tile)[c * 128 + row] = y;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
        const int t = threadIdx.x - 64;
        const int per_row = 128 * esz / 16;  // 16-byte chunks per tile row
        for (int idx = t; idx < BN * per_row; idx += 128) {
          const int cl = idx / per_row, ch = idx % per_row;
          const int n = nt * BN + cl, m0 = mt * 128 + ch * (16 / esz);
          if (n < a.Nb && m0 < a.Ma)
            *reinterpret_cast<uint4 *>(static_cast<unsigned char *>(a.c) + ((size_t)n * a.ldc + m0) * esz) =
                *reinterpret_cast<const uint4 *>(tile + ((size_t)cl * 128 + ch * (16 / esz)) * esz);
        }
      } else if (m < a.Ma) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int n = nt * BN + c;
          if (n < a.Nb) {
            const float y = acc[c] * ts;
            if (a.c_is_bf16)
              static_cast<uint16_t *>(a.c)[(size_t)n * a.ldc + m] = f32_to_bf16_bits(y);
            else
              static_cast<float *>(a.c)[(size_t)n * a.ldc + m] = y;
          }
        }
      }
    }
  }
  if (warp < 2 && KS > 1) cg::this_cluster().sync();  // the same cluster barrier, producer/MMA warps
  if (!ok && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- persistent form
// Large problems (prefill, large batches) with both operands' scales tiled and
// BF16 output: one CTA per SM walks the 128 x 128 output tiles (tile =
// blockIdx.x + i * gridDim.x, weight tiles fastest, so the CTAs in flight share
// the activation tile). The shared-memory ring of S stages runs on across tile
// boundaries -- the producer fetches the next tile's operands while the MMAs of
// this one drain -- and two TMEM accumulators (columns 0 and 128) let the
// epilogue of tile i overlap the MMAs of tile i + 1. Scales of stage s sit at
// TMEM column 256 + 32 s, written by four scale warps with tcgen05.st, so the
// MMA thread issues only MMAs. Warps: 0 producer, 1 MMA, 2..5 epilogue (each
// tile staged as [128 tokens][128 rows] BF16 in a buffer of its own), 6..9
// scales.
constexpr int kWThreads = 320;  // persistent forms: producer, MMA, 4 epilogue and 4 scale warps
constexpr int kPStage = kATile + 128 * 128 + 2 * 4 * kSFAtom;  // A codes | B codes | A atoms | B atoms
constexpr int kPStaging = 128 * 128 * 2;
constexpr int kPTmemCols = 512;
static_assert(kPStage % 1024 == 0, "stages stay 1024-byte aligned");

template <int S>
constexpr size_t persist_smem_bytes() {
  return 1024 + (size_t)S * kPStage + kPStaging + (3 * S + 4) * 8 + 16;
}

template <int S>
__global__ void __launch_bounds__(kWThreads, 1)
    gemm_nvf4_persist_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             TcArgs a) {
  static_assert(256 + 32 * S <= kPTmemCols, "scale columns exceed the allocation");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char *staging = sm + (size_t)S * kPStage;
  uint64_t *full = reinterpret_cast<uint64_t *>(staging + kPStaging);
  uint64_t *empty = full + S;
  uint64_t *sready = empty + S;  // [S] the stage's scales are in TMEM (4 warp arrivals)
  uint64_t *tfull = sready + S;  // [2] accumulator b complete (tcgen05.commit)
  uint64_t *tempty = tfull + 2;  // [2] accumulator b drained by the epilogue (128 arrivals)
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(tempty + 2);
  auto stA = [&](int s) { return sm + (size_t)s * kPStage; };
  auto stB = [&](int s) { return stA(s) + kATile; };
  auto stAtA = [&](int s) { return stB(s) + 128 * 128; };
  auto stAtB = [&](int s) { return stAtA(s) + 4 * kSFAtom; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (a.Ma + 127) >> 7, n_tiles = (a.Nb + 127) >> 7;
  const int ntiles = m_tiles * n_tiles;
  const int nkt = a.K >> 8;      // 256-wide K tiles per output tile
  const int ksteps = a.K >> 6;   // 64-wide MMA steps
  if (a.early_trigger) pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
      mbar_init(sready + s, 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 128);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kPTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      constexpr uint32_t bytes = kPStage;
      auto load_a = [&](int mt, int kt, int s) {
        if (a.a_tiles)
          bulk_g2s(stA(s), a.a_tiles + ((size_t)mt * nkt + kt) * kATile, kATile, full + s);
        else
          tma_load_2d(stA(s), &tmA, kt * 128, mt * 128, full + s);
        bulk_g2s(stAtA(s), a.sfa_tiled + ((size_t)mt * ksteps + (size_t)kt * 4) * kSFAtom, 4 * kSFAtom, full + s);
      };
      auto load_b = [&](int nt, int kt, int s) {
        tma_load_2d(stB(s), &tmB, kt * 128, nt * 128, full + s);
        bulk_g2s(stAtB(s), a.sfb_tiled + ((size_t)nt * ksteps + (size_t)kt * 4) * kSFAtom, 4 * kSFAtom, full + s);
      };
      const int t0 = blockIdx.x;
      // the first tile's weights do not depend on the preceding kernel
      const int pre = (a.a_const && t0 < ntiles) ? min(S, nkt) : 0;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(full + i, bytes);
        load_a(t0 % m_tiles, i, i);
      }
      pdl_wait();
      if (!a.early_trigger) pdl_launch_dependents();
      for (int i = 0; i < pre; ++i) load_b(t0 / m_tiles, i, i);
      int g = pre;
      for (int tile = t0; ok && tile < ntiles; tile += gridDim.x) {
        const int mt = tile % m_tiles, nt = tile / m_tiles;
        for (int kt = (tile == t0 ? pre : 0); kt < nkt; ++kt, ++g) {
          const int s = g % S, u = g / S;
          if (u > 0 && !mbar_wait(empty + s, (uint32_t)((u - 1) & 1))) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, bytes);
          load_a(mt, kt, s);
          load_b(nt, kt, s);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4<128>();
      int g = 0, i = 0;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++i) {
        const int b = i & 1;
        if (i >= 2 && !mbar_wait(tempty + b, (uint32_t)(((i >> 1) - 1) & 1))) { ok = false; break; }
        tc_fence_after();
        for (int kt = 0; kt < nkt; ++kt, ++g) {
          const int s = g % S, u = g / S;
          if (!mbar_wait(full + s, (uint32_t)(u & 1)) || !mbar_wait(sready + s, (uint32_t)(u & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = tmem + 256 + 32 * s, sfb = sfa + 16;
          const uint64_t ad = desc_sw128(smem_u32(stA(s))), bd = desc_sw128(smem_u32(stB(s)));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_nvf4(tmem + b * 128, ad + 2 * j, bd + 2 * j, idesc, sfa + 4 * j, sfb + 4 * j, (kt | j) != 0);
          tc_commit(empty + s);
        }
        if (!ok) break;
        tc_commit(tfull + b);
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------ scales -> TMEM (warps 6..9)
    // Each warp writes its TMEM lane quarter with tcgen05.st: per 64-wide K
    // step the 16-byte scale row `lane` of the stage's atom, for both
    // operands (the layout tcgen05.cp.32x128b.warpx4 would give).
    const int q = warp & 3;
    int n_st = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) n_st += nkt;
    for (int g = 0; g < n_st; ++g) {
      const int s = g % S, u = g / S;
      // lane 0 waits and the warp follows it, so the collective TMEM stores
      // below always run with all 32 lanes (or none)
      const int got = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(full + s, (uint32_t)(u & 1)) : 0, 0);
      __syncwarp();
      if (!got) { ok = false; break; }
      uint32_t va[16], vb[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 x = *reinterpret_cast<const uint4 *>(stAtA(s) + j * kSFAtom + lane * 16);
        const uint4 y = *reinterpret_cast<const uint4 *>(stAtB(s) + j * kSFAtom + lane * 16);
        va[4 * j] = x.x; va[4 * j + 1] = x.y; va[4 * j + 2] = x.z; va[4 * j + 3] = x.w;
        vb[4 * j] = y.x; vb[4 * j + 1] = y.y; vb[4 * j + 2] = y.z; vb[4 * j + 3] = y.w;
      }
      const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + 256 + 32 * s;
      tmem_st16(base, va);
      tmem_st16(base + 16, vb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sready + s);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int t = threadIdx.x - 64;
    const bool vec = (a.ldc % 8) == 0 && (a.Ma % 8) == 0 && (reinterpret_cast<uintptr_t>(a.c) & 15u) == 0;
    uint16_t *tile_s = reinterpret_cast<uint16_t *>(staging);
    volatile uint32_t *eflag = tmem_holder + 1;
    int i = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
      const int b = i & 1;
      const int mt = tile % m_tiles, nt = tile / m_tiles;
      // one thread waits for the accumulator, so that all 128 leave the loop
      // together if the wait gives up (the named barriers below stay matched)
      if (t == 0) *eflag = mbar_wait(tfull + b, (uint32_t)((i >> 1) & 1)) ? 1u : 0u;
      asm volatile("bar.sync 1, 128;" ::: "memory");  // also: the previous tile's staging reads are done
      if (*eflag == 0) { ok = false; break; }
      tc_fence_after();
      const int m = mt * 128 + row;
      const float ts = (m < a.a_split ? a.ts_a0 : a.ts_a1) * a.ts_b;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + b * 128 + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c) tile_s[(c0 + c) * 128 + row] = f32_to_bf16_bits(__uint_as_float(r[c]) * ts);
      }
      tc_fence_before();
      mbar_arrive(tempty + b);  // the accumulator may take the tile after next
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the tile is staged; every thread has read the flag
      if (vec) {
        for (int idx = t; idx < 128 * 16; idx += 128) {
          const int cl = idx >> 4, ch = idx & 15;
          const int n = nt * 128 + cl, m0 = mt * 128 + ch * 8;
          if (n < a.Nb && m0 < a.Ma)
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.c) + (size_t)n * a.ldc + m0) =
                *reinterpret_cast<const uint4 *>(tile_s + cl * 128 + ch * 8);
        }
      } else if (m < a.Ma) {
        for (int c = 0; c < 128; ++c) {
          const int n = nt * 128 + c;
          if (n < a.Nb) static_cast<uint16_t *>(a.c)[(size_t)n * a.ldc + m] = tile_s[c * 128 + row];
        }
      }
    }
  }
  if (!ok && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

// ---------------------------------------------------------------- weight-stationary form
// K = 2048 (the in-projection): a 128-row weight tile is 128 KB of codes and
// 16 KB of scales, so it stays in shared memory while the CTA walks a run of
// token tiles. CTA c takes the output tiles [c U / G, (c + 1) U / G) of the U
// tiles in weight-tile-major order (G CTAs, one per SM), so it holds one or two
// weight tiles in turn; only the 128-token activation tiles stream through the
// S-stage ring. The weight scales go into TMEM once per weight tile (columns
// 0..127, four per 64-wide K step); accumulators at columns 128 and 256; the
// activation scales of ring stage s at 384 + 16 s. The activation scales are
// put into TMEM by four warps of their own with tcgen05.st (each writes its
// lane quarter: the 16-byte scale row of each 64-wide K step, the layout
// tcgen05.cp.32x128b.warpx4 would give), so the MMA thread issues only MMAs
// per ring stage. The MMA thread commits `afree` after the last MMA on a
// weight tile; the producer reloads the weights only after it fires. The
// epilogue stores straight from registers. Warps: 0 producer, 1 MMA, 2..5
// epilogue, 6..9 activation scales.
constexpr int kWK = 2048;
constexpr int kWKt = kWK / 256;                 // 256-wide K tiles
constexpr int kWCodes = kWKt * kATile;          // 128 KB
constexpr int kWScales = (kWK / 64) * kSFAtom;  // 16 KB
constexpr int kWStages = 4;

constexpr size_t wstat_smem_bytes() {
  return 1024 + (size_t)kWCodes + (size_t)kWStages * (128 * 128) + kWScales + (size_t)kWStages * 4 * kSFAtom +
         (3 * kWStages + 6) * 8 + 16;
}

__global__ void __launch_bounds__(kWThreads, 1)
    gemm_nvf4_wstat_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           TcArgs a) {
  constexpr int S = kWStages;
  static_assert(384 + 16 * S <= kPTmemCols, "scale columns exceed the allocation");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  unsigned char *sA = sm;                            // [kWKt][16 KB] swizzled weight codes
  unsigned char *sB0 = sA + kWCodes;                 // [S][16 KB] swizzled activation codes
  unsigned char *sSFA = sB0 + S * 128 * 128;         // [32][512 B] weight scale atoms
  unsigned char *sSFB0 = sSFA + kWScales;            // [S][4][512 B] activation scale atoms
  uint64_t *full = reinterpret_cast<uint64_t *>(sSFB0 + S * 4 * kSFAtom);
  uint64_t *empty = full + S;
  uint64_t *sready = empty + S;  // [S] the stage's activation scales are in TMEM (4 warp arrivals)
  uint64_t *tfull = sready + S;
  uint64_t *tempty = tfull + 2;
  uint64_t *afull = tempty + 2;
  uint64_t *afree = afull + 1;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(afree + 1);
  volatile uint32_t *eflag = tmem_holder + 1;  // [2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (a.Ma + 127) >> 7, n_tiles = (a.Nb + 127) >> 7;
  const long long U = (long long)m_tiles * n_tiles;
  const int u0 = (int)(U * blockIdx.x / gridDim.x), u1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
  constexpr int ksteps = kWK / 64;
  if (a.early_trigger) pdl_launch_dependents();
  if (a.K != kWK) {  // host-side contract broken: refuse, uniformly
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(a.status, GDN_E_SHAPE);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
      mbar_init(sready + s, 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, 128);
    }
    mbar_init(afull, 1);
    mbar_init(afree, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kPTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      auto load_w = [&](int mt) {
        mbar_arrive_expect_tx(afull, kWCodes + kWScales);
        for (int kt = 0; kt < kWKt; ++kt) {
          if (a.a_tiles)
            bulk_g2s(sA + kt * kATile, a.a_tiles + ((size_t)mt * kWKt + kt) * kATile, kATile, afull);
          else
            tma_load_2d(sA + kt * kATile, &tmA, kt * 128, mt * 128, afull);
        }
        bulk_g2s(sSFA, a.sfa_tiled + (size_t)mt * ksteps * kSFAtom, kWScales, afull);
      };
      int cur = -1, na = 0, g = 0;
      if (u0 < u1 && a.a_const) {  // the weights do not depend on the preceding kernel
        cur = u0 / n_tiles;
        load_w(cur);
        na = 1;
      }
      pdl_wait();
      if (!a.early_trigger) pdl_launch_dependents();
      for (int u = u0; ok && u < u1; ++u) {
        const int mt = u / n_tiles, nt = u % n_tiles;
        if (mt != cur) {
          if (na > 0 && !mbar_wait(afree, (uint32_t)((na - 1) & 1))) { ok = false; break; }
          load_w(mt);
          cur = mt;
          ++na;
        }
        for (int kt = 0; kt < kWKt; ++kt, ++g) {
          const int s = g % S, r = g / S;
          if (r > 0 && !mbar_wait(empty + s, (uint32_t)((r - 1) & 1))) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, 128 * 128 + 4 * kSFAtom);
          tma_load_2d(sB0 + s * 128 * 128, &tmB, kt * 128, nt * 128, full + s);
          bulk_g2s(sSFB0 + s * 4 * kSFAtom, a.sfb_tiled + ((size_t)nt * ksteps + (size_t)kt * 4) * kSFAtom,
                   4 * kSFAtom, full + s);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4<128>();
      int cur = -1, na = 0, g = 0, i = 0;
      for (int u = u0; ok && u < u1; ++u, ++i) {
        const int mt = u / n_tiles, b = i & 1;
        if (mt != cur) {
          if (na > 0) tc_commit(afree);  // every MMA on the previous weight tile
          if (!mbar_wait(afull, (uint32_t)(na & 1))) { ok = false; break; }
          tc_fence_after();
          for (int j = 0; j < ksteps; ++j) tc_cp_scales(tmem + 4 * j, desc_scales(smem_u32(sSFA) + j * kSFAtom));
          cur = mt;
          ++na;
        }
        if (i >= 2 && !mbar_wait(tempty + b, (uint32_t)(((i >> 1) - 1) & 1))) { ok = false; break; }
        tc_fence_after();
        for (int kt = 0; kt < kWKt; ++kt, ++g) {
          const int s = g % S, r = g / S;
          if (!mbar_wait(full + s, (uint32_t)(r & 1)) || !mbar_wait(sready + s, (uint32_t)(r & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfb = tmem + 384 + 16 * s;
          const uint64_t ad = desc_sw128(smem_u32(sA + kt * kATile)), bd = desc_sw128(smem_u32(sB0 + s * 128 * 128));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_nvf4(tmem + 128 + b * 128, ad + 2 * j, bd + 2 * j, idesc, tmem + 4 * (kt * 4 + j), sfb + 4 * j,
                        (kt | j) != 0);
          tc_commit(empty + s);
        }
        if (!ok) break;
        tc_commit(tfull + b);
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------ activation scales -> TMEM (warps 6..9)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int nst = (u1 - u0) * kWKt;
    for (int g = 0; g < nst; ++g) {
      const int s = g % S, r = g / S;
      // lane 0 waits and the warp follows it, so the collective TMEM store
      // below always runs with all 32 lanes (or none)
      const int got = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(full + s, (uint32_t)(r & 1)) : 0, 0);
      __syncwarp();
      if (!got) { ok = false; break; }
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // K step j: scale row `lane` of the stage's atom j
        const uint4 x = *reinterpret_cast<const uint4 *>(sSFB0 + s * 4 * kSFAtom + j * kSFAtom + lane * 16);
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
      }
      tmem_st16(tmem + ((uint32_t)(q * 32) << 16) + 384 + 16 * s, v);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sready + s);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int t = threadIdx.x - 64;
    uint16_t *C = static_cast<uint16_t *>(a.c);
    int i = 0;
    for (int u = u0; u < u1; ++u, ++i) {
      const int b = i & 1;
      const int mt = u / n_tiles, nt = u % n_tiles;
      // one thread waits, all 128 leave together if the wait gives up; the flag
      // alternates so that one barrier per tile keeps its reads and writes apart
      if (t == 0) eflag[b] = mbar_wait(tfull + b, (uint32_t)((i >> 1) & 1)) ? 1u : 0u;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (eflag[b] == 0) { ok = false; break; }
      tc_fence_after();
      const int m = mt * 128 + row;
      const float ts = (m < a.a_split ? a.ts_a0 : a.ts_a1) * a.ts_b;
      const int nlim = min(128, a.Nb - nt * 128);
      uint16_t *dst = C + (size_t)nt * 128 * a.ldc + m;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + 128 + b * 128 + c0, r);
        tmem_ld_wait();
        if (m < a.Ma) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (c0 + c < nlim) dst[(size_t)(c0 + c) * a.ldc] = f32_to_bf16_bits(__uint_as_float(r[c]) * ts);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty + b);  // the accumulator may take the tile after next
    }
  }
  if (!ok && lane == 0) flag_status(a.status, GDN_E_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

// ---------------------------------------------------------------- host side
template <int BN, int KS, int S>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)S * Layout<BN>::kStage + (KS > 1 ? (size_t)(KS - 1) * 128 * BN * 4 : 0) + (3 * S + 2) * 8 + 16;
}

template <int BN, int KS, int S>
cudaError_t launch_t(const TcGemm &g, const LaunchCtx &lc) {
  CUtensorMap mB = g.mapA, mSB = g.mapSA;  // decode form: never read
  if (!g.args.b_bf16 &&
      (!make_map(&mB, g.b_codes, (uint64_t)g.args.Nb, (uint64_t)g.args.K / 2, BN, 128, true) ||
       !make_map(&mSB, g.b_scales, (uint64_t)g.args.Nb, (uint64_t)g.args.K / 16, BN, 16, false)))
    return cudaErrorInvalidValue;
  size_t smem = smem_bytes<BN, KS, S>();
  if (smem < 80 * 1024) smem = 80 * 1024;  // at most two CTAs (2 x 256 TMEM columns) per SM
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_nvf4_kernel<BN, KS, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((g.args.Ma + 127) / 128) * KS, (g.args.Nb + BN - 1) / BN, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  ++na;
  if (KS > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = KS;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_nvf4_kernel<BN, KS, S>, g.mapA, mB, g.mapSA, mSB, g.args);
}

constexpr size_t kSmemCap = 227 * 1024;

constexpr int kPersistStages = 5;
static_assert(persist_smem_bytes<kPersistStages>() <= kSmemCap, "persistent GEMM shared memory");

static_assert(wstat_smem_bytes() <= kSmemCap, "weight-stationary GEMM shared memory");

cudaError_t launch_wstat(const TcGemm &g, const LaunchCtx &lc) {
  CUtensorMap mB;
  if (!make_map(&mB, g.b_codes, (uint64_t)g.args.Nb, (uint64_t)g.args.K / 2, 128, 128, true))
    return cudaErrorInvalidValue;
  constexpr size_t smem = wstat_smem_bytes();
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_nvf4_wstat_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int ntiles = ((g.args.Ma + 127) / 128) * ((g.args.Nb + 127) / 128);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(min(ntiles, lc.num_sms), 1, 1);
  cfg.blockDim = dim3(kWThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_nvf4_wstat_kernel, g.mapA, mB, g.args);
}

cudaError_t launch_persist(const TcGemm &g, const LaunchCtx &lc) {
  CUtensorMap mB;
  if (!make_map(&mB, g.b_codes, (uint64_t)g.args.Nb, (uint64_t)g.args.K / 2, 128, 128, true))
    return cudaErrorInvalidValue;
  constexpr size_t smem = persist_smem_bytes<kPersistStages>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_nvf4_persist_kernel<kPersistStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int ntiles = ((g.args.Ma + 127) / 128) * ((g.args.Nb + 127) / 128);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(min(ntiles, lc.num_sms), 1, 1);
  cfg.blockDim = dim3(kWThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_nvf4_persist_kernel<kPersistStages>, g.mapA, mB, g.args);
}

template <int BN>
cudaError_t launch_bn(const TcGemm &g, int ks, const LaunchCtx &lc) {
  // the largest split <= ks whose shared memory fits
  if (ks >= 8 && smem_bytes<BN, 8, 4>() <= kSmemCap) return launch_t<BN, 8, 4>(g, lc);
  if (ks >= 4 && smem_bytes<BN, 4, 4>() <= kSmemCap) return launch_t<BN, 4, 4>(g, lc);
  if (ks >= 2 && smem_bytes<BN, 2, 4>() <= kSmemCap) return launch_t<BN, 2, 4>(g, lc);
  return launch_t<BN, 1, 4>(g, lc);
}

}  // namespace

bool tc_make_weight_maps(TcGemm &g, const uint8_t *w_codes, const uint8_t *w_scales, int rows, int K) {
  return make_map(&g.mapA, w_codes, (uint64_t)rows, (uint64_t)K / 2, 128, 128, true) &&
         make_map(&g.mapSA, w_scales, (uint64_t)rows, (uint64_t)K / 16, 128, 16, false);
}

// Split-K so that the grid covers the GPU: tiles x KS >= SMs when K allows.
int tc_pick_split(int m_tiles, int n_tiles, int K, int num_sms) {
  const int kt = K / 256;
  int ks = 1;
  while (ks < 8 && m_tiles * n_tiles * ks * 2 <= num_sms && kt % (ks * 2) == 0) ks *= 2;
  return ks;
}

cudaError_t launch_tc_gemm(const TcGemm &g, const LaunchCtx &lc) {
  const TcArgs &a = g.args;
  if (a.Ma <= 0 || a.Nb <= 0) return cudaSuccess;
  if (a.K % 256) return cudaErrorInvalidValue;
  const int m_tiles = (a.Ma + 127) / 128;
  int bn = a.Nb <= 16 ? 16 : a.Nb <= 32 ? 32 : a.Nb <= 64 ? 64 : 128;
  const int n_tiles = (a.Nb + bn - 1) / bn;
  int ks = g.split_k > 0 ? g.split_k : tc_pick_split(m_tiles, n_tiles, a.K, lc.num_sms);
  while (ks > 1 && (a.K / 256) % ks) ks >>= 1;  // the split must divide the K tiles
  if (a.b_bf16) {  // decode form: at most 16 rows, every K tile of a CTA in its own stage
    if (bn != 16 || !a.a_const || !a.sfa_tiled) return cudaErrorInvalidValue;
    while (ks < 8 && (a.K / 256) / ks > 4) ks *= 2;
    if ((a.K / 256) % ks || (a.K / 256) / ks > 4) return cudaErrorInvalidValue;
  }
  // persistent forms: 128-token activation tiles, tiled scales, BF16 out.
  // Automatically the streaming form, from two output tiles per SM (measured
  // on GB300, prefill in-projection T = 16384: streaming 230 us, weight-
  // stationary 276 us, one tile per CTA 588 us; with 1.3 tiles per SM, batch
  // 256, the tile-per-CTA kernel was faster). Weight-stationary on request.
  if (!a.b_bf16 && a.sfa_tiled && a.sfb_tiled && a.c_is_bf16 && ks == 1 && bn == 128 && g.persist != 1) {
    if (g.persist == 3 && a.K == kWK && a.a_const) return launch_wstat(g, lc);
    if (g.persist >= 2 || m_tiles * n_tiles >= 2 * lc.num_sms) return launch_persist(g, lc);
  }
  switch (bn) {
    case 16: return launch_bn<16>(g, ks, lc);
    case 32: return launch_bn<32>(g, ks, lc);
    case 64: return launch_bn<64>(g, ks, lc);
    default: return launch_bn<128>(g, ks, lc);
  }
}

}  // namespace gdn
