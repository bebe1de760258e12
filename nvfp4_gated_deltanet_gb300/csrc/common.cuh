// Shared device helpers of the GDN kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn.h"

#define GDN_DEV __device__ __forceinline__

namespace gdn {

// ---------------------------------------------------------------- status word
// Sticky: the first non-zero code stays. Only error paths write it.
GDN_DEV void flag_status(int32_t *status, int code) {
  if (status) atomicCAS(reinterpret_cast<int *>(status), 0, code);
}

// ---------------------------------------------------------------- conversions
GDN_DEV float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

GDN_DEV uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&h);
}

// One element of a recurrent state stored as FP32 or as BF16 bits.
GDN_DEV float state_load(const void *S, int bf16, size_t i) {
  return bf16 ? bf16_bits_to_f32(static_cast<const uint16_t *>(S)[i]) : static_cast<const float *>(S)[i];
}
GDN_DEV void state_store(void *S, int bf16, size_t i, float v) {
  if (bf16)
    static_cast<uint16_t *>(S)[i] = f32_to_bf16_bits(v);
  else
    static_cast<float *>(S)[i] = v;
}

// E4M3 (OCP e4m3fn), round to nearest even, saturate finite values to 448.
// Returns the byte of `v` (v finite).
GDN_DEV uint32_t e4m3_from_f32(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// E4M3 byte -> float (exact).
GDN_DEV float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  uint16_t in = uint16_t(byte & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
}

// Two floats -> one byte of two E2M1 codes (lo in the low nibble), RNE, satfinite.
GDN_DEV uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u16.u8 %0, t;\n\t}"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// One byte of two E2M1 codes -> half2 (low nibble in .x), exact.
// Four E2M1 pairs (one 32-bit word: element 2i in the low nibble of byte i)
// to four FP16x2 values, exact. The word is split into its bytes by a vector
// move, so each pair costs one conversion and no shift or mask.
GDN_DEV void e2m1x8_to_h2x4(uint32_t w, __half2 (&h)[4]) {
  uint32_t r0, r1, r2, r3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
  h[0] = *reinterpret_cast<__half2 *>(&r0);
  h[1] = *reinterpret_cast<__half2 *>(&r1);
  h[2] = *reinterpret_cast<__half2 *>(&r2);
  h[3] = *reinterpret_cast<__half2 *>(&r3);
}

GDN_DEV __half2 e2m1x2_to_h2(uint32_t byte) {
  uint32_t h2;
  uint16_t in = uint16_t(byte & 0xFFu);
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.u8.u16 t, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2) : "h"(in));
  return *reinterpret_cast<__half2 *>(&h2);
}

// ---------------------------------------------------------------- NVFP4 block quantiser
// One 16-element block in FP32, in the fixed order of the library's NVFP4
// reading: amax, t = amax * inv6ts, s = E4M3(t), d = e4m3(s) * ts, r = 1/d,
// code = E2M1(x * r). inv6ts = 1 / (6 * ts), both FP32 roundings.
// Returns false (scale 0, codes 0) when the block holds NaN or infinity.
GDN_DEV bool quant_block16(const float (&v)[16], float ts, float inv6ts, uint32_t &codes_lo,
                           uint32_t &codes_hi, uint32_t &scale) {
  float amax = 0.0f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(v[i]);
    finite &= (a <= 3.402823466e38f);  // false for NaN and +inf
    amax = fmaxf(amax, a);
  }
  codes_lo = codes_hi = 0u;
  scale = 0u;
  if (!finite) return false;
  float t = __fmul_rn(amax, inv6ts);
  scale = e4m3_from_f32(t);
  float sv = e4m3_to_f32(scale);
  if (sv == 0.0f) return true;
  float r = __frcp_rn(__fmul_rn(sv, ts));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t b0 = e2m1x2_from_f32(__fmul_rn(v[2 * i], r), __fmul_rn(v[2 * i + 1], r));
    uint32_t b1 = e2m1x2_from_f32(__fmul_rn(v[8 + 2 * i], r), __fmul_rn(v[8 + 2 * i + 1], r));
    codes_lo |= b0 << (8 * i);
    codes_hi |= b1 << (8 * i);
  }
  return true;
}

GDN_DEV float inv6ts_of(float ts) { return __frcp_rn(__fmul_rn(6.0f, ts)); }

// Warp-level m16n8k16 MMA, FP16 inputs, FP32 accumulation starting from zero:
// d = A (16 x 16, row) * B (16 x 8, col). Lane (g = lane / 4, t = lane % 4)
// holds d[0], d[1] = rows g, columns 2t, 2t+1 and d[2], d[3] = row g + 8.
GDN_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// Four E4M3 bytes -> four floats (exact).
GDN_DEV void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
  uint32_t lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
  f[0] = __half2float(__ushort_as_half(uint16_t(lo & 0xFFFFu)));
  f[1] = __half2float(__ushort_as_half(uint16_t(lo >> 16)));
  f[2] = __half2float(__ushort_as_half(uint16_t(hi & 0xFFFFu)));
  f[3] = __half2float(__ushort_as_half(uint16_t(hi >> 16)));
}

// One NVFP4 block (codes lo/hi, scale byte) as x_hat = e2m1 * e4m3 in FP16,
// exact (|x_hat| <= 6 * 448 and >= 2^-10), written as 16 halves.
GDN_DEV void store_xhat_block(__half *dst, uint32_t lo, uint32_t hi, uint32_t s) {
  __half2 h[8];
  e2m1x8_to_h2x4(lo, *reinterpret_cast<__half2(*)[4]>(&h[0]));
  e2m1x8_to_h2x4(hi, *reinterpret_cast<__half2(*)[4]>(&h[4]));
  const __half2 sc = __float2half2_rn(e4m3_to_f32(s));
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = __hmul2(h[i], sc);
  reinterpret_cast<uint4 *>(dst)[0] = *reinterpret_cast<const uint4 *>(&h[0]);
  reinterpret_cast<uint4 *>(dst)[1] = *reinterpret_cast<const uint4 *>(&h[4]);
}

// 16 BF16 values (two 16-byte loads) -> FP32.
GDN_DEV void load_bf16x16(const uint16_t *p, float (&v)[16]) {
  const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 w4 = q[i];
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
      v[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

// Tiled scale layout read by tcgen05.cp .32x128b.warpx4 for one operand of the
// block-scaled MMA: the scales of 128 rows x one 64-wide K step form a 512-byte
// atom, row r at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + k-block; atoms are
// ordered [row tile][K step]. `blk` is the 16-element block index along K,
// `nblk` = K / 16 (a multiple of 4). Rows are padded to whole 128-row tiles.
__host__ __device__ __forceinline__ size_t sf_tiled_offset(int r, int blk, int nblk) {
  return ((size_t)(r >> 7) * (nblk >> 2) + (blk >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (blk & 3);
}
inline size_t sf_tiled_bytes(int rows, int K) { return (size_t)((rows + 127) / 128) * 128 * (K / 16); }

// ---------------------------------------------------------------- reductions
// xor butterfly: partners add the same two values in either order, so every
// lane ends with the bit-identical total.
GDN_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Reduce NV (power of two, 1..32) per-lane values over the warp with
// NV - 1 + log2(64/NV) shuffles instead of 5 * NV: each round halves the live
// values, a lane keeping one half and sending the other to its partner.
// Afterwards lane l holds the total of value reduce_index<NV>(l), and every
// lane holding the same value index holds the bit-identical total.
template <int NV>
GDN_DEV float warp_transpose_reduce(float (&v)[NV], int lane) {
  static_assert(NV >= 1 && NV <= 32 && (NV & (NV - 1)) == 0, "NV power of two <= 32");
  // Halve the live values each round; partner lanes differ in bit `b`.
  int live = NV;
#pragma unroll
  for (int b = 4; b >= 0; --b) {
    if (live > 1) {
      const int half = live >> 1;
      const bool upper = (lane >> b) & 1;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < half) {
          float send = upper ? v[i] : v[i + half];
          float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << b);
        }
      }
      live = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1 << b);
    }
  }
  return v[0];
}

// Which value's total lane `lane` holds after warp_transpose_reduce<NV>.
template <int NV>
GDN_DEV int reduce_index(int lane) {
  int idx = 0, live = NV;
#pragma unroll
  for (int b = 4; b >= 0; --b) {
    if (live > 1) {
      const int half = live >> 1;
      if ((lane >> b) & 1) idx += half;
      live = half;
    }
  }
  return idx;
}

// A lane that holds the total of value `idx` after warp_transpose_reduce<NV>.
template <int NV>
GDN_DEV int reduce_owner(int idx) {
  int lane = 0, live = NV;
#pragma unroll
  for (int b = 4; b >= 0; --b) {
    if (live > 1) {
      const int half = live >> 1;
      if (idx >= half) { lane |= 1 << b; idx -= half; }
      live = half;
    }
  }
  return lane;
}

// ---------------------------------------------------------------- async copies, mbarriers, PDL
GDN_DEV uint32_t smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

GDN_DEV void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async (TMA) proxy.
GDN_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
}
GDN_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
GDN_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Every wait is bounded: ~2^31 SM cycles (about one second at 2 GHz), then the
// caller records GDN_E_TIMEOUT and gives up instead of hanging the GPU.
constexpr long long kWaitCycles = 1LL << 31;
// The same test with a suspend-time hint: the thread sleeps until the phase
// completes or about `ns` nanoseconds pass, instead of spinning on the issue
// slots its neighbours need.
GDN_DEV bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
GDN_DEV bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 20000u))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}
// Bulk (non-tensor) copy global -> shared, completion counted on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
GDN_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Programmatic dependent launch: wait for the preceding grid (no-op when the
// launch did not ask for it); let the next grid start its prologue.
GDN_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
GDN_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

GDN_DEV float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
GDN_DEV float siluf_(float x) { return x / (1.0f + expf(-x)); }
GDN_DEV float softplusf_(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

}  // namespace gdn

// ---------------------------------------------------------------- launchers (internal)
namespace gdn {
struct LaunchCtx {
  cudaStream_t stream;
  int num_sms;
  bool pdl;  // launch with programmatic stream serialization (kernels read only
             // constants -- weights -- before griddepcontrol.wait)
};

// row_slot (optional): row r is quantised as zeros when row_slot[r] is not a
// valid slot (a padding row of a decode batch).
// sf_tiled: write the scales in the tiled layout (sf_tiled_offset) instead of
// row-major [rows][cols/16]; needs cols % 64 == 0.
cudaError_t launch_quantize(const void *x, int x_is_f32, int rows, int cols, float ts, uint8_t *codes,
                            uint8_t *scales, int32_t *status, cudaStream_t stream, const int32_t *row_slot = nullptr,
                            int num_slots = 0, bool pdl = false, bool sf_tiled = false);
// Repack row-major scales [rows][K/16] into the tiled layout (padding rows 0).
cudaError_t launch_tile_scales(const uint8_t *src, int rows, int K, uint8_t *dst, cudaStream_t stream);
// Repack row-major codes [rows][K/2] (K % 256 == 0) into pre-swizzled 16 KB
// MMA tiles (TcArgs::a_tiles); swizzled_tiles_bytes gives the size.
cudaError_t launch_swizzle_tiles(const uint8_t *src, int rows, int K, uint8_t *dst, cudaStream_t stream);
inline size_t swizzled_tiles_bytes(int rows, int K) { return (size_t)((rows + 127) / 128) * (K / 256) * 16384; }

// C[M][N] (ldc) = A_hat[M][K] * W_hat[N][K]^T. A is BF16 rows (quantised inside
// with ts_a; a_rows_valid may mark rows to treat as zero) or NVFP4. Rows of W
// below n_split use ts_w0, the rest ts_w1. M <= 16.
struct GemvArgs {
  const uint16_t *a_bf16;   // [M][K] or null
  const uint8_t *a_codes;   // [M][K/2] or null
  const uint8_t *a_scales;  // [M][K/16]
  float ts_a;
  const int32_t *row_slot;  // optional: row m is zero when row_slot[m] < 0 or >= num_slots
  int num_slots;
  const uint8_t *w_codes, *w_scales;
  float ts_w0, ts_w1;
  int n_split;
  void *c;
  int c_is_bf16;
  int ldc;
  int M, N, K;
  int32_t *status;
  int early_trigger;  // as TcArgs::early_trigger
  // Optional: the weights repacked for the warp-MMA kernel (launch_mma_tiles);
  // used for 1..8 rows when K % 512 == 0.
  const uint8_t *w_mma;
  // Warp-MMA tile: 1 (or 0) = two 16-row groups per CTA x four K slices, 2 = one
  // group x eight K slices, 3 = four groups x two K slices. mma_bulk: the
  // activation rows are bulk-copied into shared memory first.
  int mma_tile, mma_bulk;
};
cudaError_t launch_gemv(const GemvArgs &a, const LaunchCtx &lc);
// Warp-MMA one-row product (gemv_mma.cu) and its weight layout.
bool gemv_mma_ok(const GemvArgs &a);
cudaError_t launch_gemv_mma(const GemvArgs &a, const LaunchCtx &lc);
size_t mma_tiles_bytes(int rows, int K);
cudaError_t launch_mma_tiles(const uint8_t *codes, const uint8_t *scales, int rows, int K, uint8_t *dst,
                             cudaStream_t stream);

struct MixArgs {
  const uint16_t *qkvz;  // [B][ld_qkvz] BF16: q | k | v | z
  int ld_qkvz;
  const uint16_t *ba;    // [B][ld_ba] BF16: b | a
  int ld_ba;
  const int32_t *slot_ids;
  int B, num_slots;
  uint16_t *conv_state;       // [S][K-1][C]
  void *ssm_state;            // [S][Hv][dv][dk], FP32 or BF16 bits (state_bf16)
  const uint16_t *conv_w;     // [C][K]
  const float *A_log, *dt_bias, *norm_w;
  int Hk, Hv, D, C, Kc;
  float l2_eps, rms_eps, ts_out;
  uint8_t *y_codes;   // [B][Hv*dv/2] or null
  uint8_t *y_scales;  // [B][Hv*dv/16] row-major, or tiled when y_sf_tiled
  int y_sf_tiled;
  float *y_f32;       // [B][Hv*dv] or null
  int32_t *status;
  int slices;         // d_v slices per head (1, 2, 4), 0 = chosen from B
  int state_bf16;     // recurrent state stored as BF16 (loaded to FP32, stored rounded)
  // Verify passes (zero for a plain step): row b's q|k|v|z, b|a and y are row
  // b * io_mul + io_add of their buffers; its states are read from *_src
  // (row-indexed, element strides below) when set, else from its slot, and
  // written to *_dst when set, else back to its slot.
  int io_mul, io_add;
  const void *ssm_src;
  void *ssm_dst;
  const uint16_t *conv_src;
  uint16_t *conv_dst;
  size_t ssm_row_stride, conv_row_stride;
};
cudaError_t launch_mix(const MixArgs &a, const LaunchCtx &lc);

// In-projection + token mixing of a decode step in one cluster kernel
// (proj_mix.cu), B <= 8 rows; y goes out NVFP4 with row-major scales.
struct PmArgs {
  const uint16_t *x;                  // [B][H] BF16
  const int32_t *slot_ids;            // [B]
  int B, num_slots;
  const uint8_t *w_mma;               // [qkvz; ba] in the warp-MMA group layout (launch_mma_tiles)
  const uint8_t *w_codes, *w_scales;  // [qkvz; ba] row-major (the b and a rows are read from here)
  float ts_in, ts_qkvz, ts_ba;
  int H, Hk, Hv, Nqkvz, C, Kc;
  const uint16_t *conv_w;
  const float *A_log, *dt_bias, *norm_w;
  float l2_eps, rms_eps, ts_out;
  uint16_t *conv_state;               // [S][K-1][C]
  void *ssm_state;                    // [S][Hv][dv][dk], FP32 or BF16 bits
  int state_bf16;
  uint8_t *y_codes, *y_scales;        // [B][Hv*dv/2], [B][Hv*dv/16]
  int32_t *status;
};
bool proj_mix_ok(int H, int Hk, int Hv, int D, int Kc, int B);
cudaError_t launch_proj_mix(const PmArgs &a, const LaunchCtx &lc);

// Large-batch token mixing split in three kernels (batch.cu), bit-identical
// to launch_mix; the workspace holds the per-row intermediates.
struct BatchWs {
  float *qn, *kn;     // [B][Hk][D]: normalised q (times d^-1/2) and k
  float *v;           // [B][Hv][D]: conv output of the v channels
  float *beta, *gl;   // [B][Hv]
  float *o;           // [B][Hv][D]: delta-rule output
};
cudaError_t launch_batch_mix(const MixArgs &a, const BatchWs &w, const LaunchCtx &lc);

// Commit of a verify pass (verify.cu): row b with slot s >= 0 and accepted[b]
// = n in 1..r takes snapshot (b, n-1) as its slot's state; n = 0 keeps it.
struct VerifyCommitArgs {
  const int32_t *slot_ids, *accepted;  // [B] device
  int B, r, num_slots;
  const void *snap_ssm;                // [B][r] x ssm_bytes
  const uint16_t *snap_conv;           // [B][r] x conv_bytes
  void *ssm_state;                     // [S] x ssm_bytes
  uint16_t *conv_state;                // [S] x conv_bytes
  size_t ssm_bytes, conv_bytes;        // per slot, multiples of 16
  int32_t *status;
};
cudaError_t launch_verify_commit(const VerifyCommitArgs &a, cudaStream_t stream);

// KDA-style recurrent step (kda.cu): per-channel log-decays g.
struct KdaArgs {
  const float *q, *k, *g;  // [M][H][D]
  const float *v;          // [M][H][D]
  const float *beta;       // [M][H]
  void *state;             // [M][H][D][D] FP32, or BF16 bits (state_bf16)
  float *o;                // [M][H][D]
  int M, H, D, state_bf16;
};
cudaError_t launch_kda(const KdaArgs &a, cudaStream_t stream);

struct PrefillArgs {
  const uint16_t *proj;  // [T][ld] BF16: q | k | v | z | b | a
  int ld, T, Tp;         // Tp = T rounded up to whole 64-token chunks
  uint16_t *conv_state;  // this slot's [K-1][C]
  void *ssm;             // this slot's [Hv][D][D], FP32 or BF16 bits (state_bf16)
  int state_bf16;
  int scan_tc;           // chunk scan: 0 FP32 CUDA cores, 1 warp-level MMA, 2 tcgen05 (D = 128)
  const uint16_t *conv_w;
  const float *A_log, *dt_bias, *norm_w;
  int Hk, Hv, D, C, Kc;
  float l2_eps, rms_eps, ts_out;
  float *qn, *kn;        // [Hk][Tp][D]: normalised q (times d^-1/2) and k
  float *v;              // [Hv][Tp][D]
  float *beta, *gl;      // [Hv][Tp]: beta and the log-decay g
  float *W, *Ut;         // [Hv][nc][64][D]: per chunk T diag(beta e^Gamma) K and T diag(beta) V
  float *Am;             // [Hv][nc][64][64]: exp(Gamma_i - Gamma_j) q_i.k_j, j <= i
  float *Gam;            // [Hv][nc][64]: in-chunk cumulative log-decay
  // The tcgen05 chunk scan's operands in split FP16, x s = hi + lo with a
  // power-of-two scale s (the hi block first, the lo block after it), or null:
  uint16_t *Qs;          // [2][Hk][Tp][D]: q, s = 2^14 (written by prep; may alias qn)
  uint16_t *Ks;          // [2][Hk][Tp][D]: k, s = 2^14 (written by prep; may alias kn)
  uint16_t *Ws;          // [2][Hv][Tp][D]: W, s = Wsc of its chunk (may alias W)
  uint16_t *As;          // [2][Hv][Tp][64]: A, s = 2^14 (may alias Am)
  uint16_t *KTs;         // [2][Hk][nc][D][64]: per chunk K^T, s = 2^14
  float *Wsc;            // [Hv][nc]: power-of-two scale of each chunk's W
  float *Umax;           // [Hv][nc]: largest |Ut| of each chunk
  float *o;              // [T][Hv][D]
  uint8_t *y_codes;      // [T][Hv*D/2]
  uint8_t *y_scales;     // [T][Hv*D/16] row-major, or tiled when y_sf_tiled
  int y_sf_tiled;
  int32_t *status;
};
// The prefill chunk scan on tcgen05 (scan_tc.cu), d = 128; needs the split
// operands Qs, Ws, As, KTs and the per-chunk Wsc, Umax of chunk_prep_tc.
cudaError_t launch_chunk_scan_umma(const PrefillArgs &a, cudaStream_t stream);
// Block-scaled W4A4 GEMM on tcgen05: D[m][n] = W_hat[m][:] . X_hat[n][:],
// stored C[n][m] (ldc). W = weights (A operand, M = 128 rows per tile), X =
// activations (B operand). K % 256 == 0; row-major codes and scales.
struct TcArgs {
  int Ma, Nb, K;
  void *c;
  int ldc;
  int c_is_bf16;
  float ts_a0, ts_a1;  // weight tensor scale of rows < a_split, and of the rest
  int a_split;
  float ts_b;
  int a_const;         // weights written by no preceding kernel: stream them before griddepcontrol.wait
  // Optional: both operands' scales already in the tiled layout tcgen05.cp
  // reads (sf_tiled_offset); then they are bulk-copied straight into place.
  const uint8_t *sfa_tiled, *sfb_tiled;
  // Optional: the weight codes as pre-swizzled 16 KB tiles (launch_swizzle_tiles),
  // streamed with one contiguous bulk copy per K tile instead of a tensor-map
  // copy of 128 rows 1 KB apart.
  const uint8_t *a_tiles;
  int32_t *status;
  // Optional (decode rows, Nb <= 16): the B operand as BF16 rows [Nb][K],
  // quantised to NVFP4 (tensor scale ts_b) inside the kernel straight into the
  // MMA's shared-memory layout. Rows whose b_row_slot entry is not a valid slot
  // (-1 = padding) read as zero. Needs a_const and sfa_tiled, and every K tile
  // of a CTA resident at once (K / 256 / split <= the pipeline depth).
  const uint16_t *b_bf16;
  const int32_t *b_row_slot;
  int b_num_slots;
  // Signal dependents before waiting on the preceding kernel. Only for the last
  // kernel of a decode step: the next step's first kernel reads nothing but
  // weights until its own griddepcontrol.wait, which returns after this kernel
  // (and so everything before it) has completed.
  int early_trigger;
};
struct TcGemm {
  CUtensorMap mapA, mapSA;  // weights: codes [Ma][K/2] (128-byte swizzle), scales [Ma][K/16]
  const uint8_t *b_codes, *b_scales;
  TcArgs args;
  int split_k;  // 0 = automatic
  int persist;  // persistent forms: 0 = automatic, 1 = never, 2 = streaming (gemm_nvf4_persist_kernel) whenever
                // allowed, 3 = weight-stationary (gemm_nvf4_wstat_kernel, K = 2048) whenever allowed
};
bool tc_make_weight_maps(TcGemm &g, const uint8_t *w_codes, const uint8_t *w_scales, int rows, int K);
cudaError_t launch_tc_gemm(const TcGemm &g, const LaunchCtx &lc);

// The whole decode layer-step for one or two rows in one cooperative launch
// (fused.cu).
struct FusedArgs {
  const uint8_t *w_in_codes, *w_in_scales;    // [Nin][H/2], [Nin][H/16]: qkvz rows then ba rows
  const uint8_t *w_out_codes, *w_out_scales;  // [H][Vd/2], [H][Vd/16]
  float ts_qkvz, ts_ba, ts_wout;
  int Nqkvz, Nin;
  const uint16_t *conv_w;
  const float *A_log, *dt_bias, *norm_w;
  int H, Hk, Hv, D, C, Kc, Vd;
  float l2_eps, rms_eps, ts_in, ts_out;
  const uint16_t *x;
  const int32_t *slot_ids;
  int B, num_slots;
  uint16_t *out, *conv_state;
  float *ssm_state;
  uint16_t *proj;                 // scratch [B][Nin]
  uint8_t *y_codes, *y_scales;    // scratch [B][Vd/2], [B][Vd/16] row-major
  unsigned int *bar;              // grid barrier words (2), zeroed before every launch
  long long wait_cycles;          // budget of each grid-barrier wait, SM cycles
  int32_t *status;
  int rows_in, rows_out;          // weight rows per CTA (set by fused_plan)
};
bool fused_plan(FusedArgs &a, int num_sms);
cudaError_t launch_fused(const FusedArgs &a, const LaunchCtx &lc);

cudaError_t launch_prefill_mix(const PrefillArgs &a, uint16_t *tmp, const LaunchCtx &lc);

}  // namespace gdn
