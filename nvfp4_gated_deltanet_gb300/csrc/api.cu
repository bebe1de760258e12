// The C ABI of include/gdn.h: validation, the context, and the launch order of
// each call. Every step of the layer runs in the kernels of this directory.
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"

using namespace gdn;

struct gdn_ctx {
  gdn_config cfg;
  int Nqkvz, Nba, Nin, C, Vd, prow;
  int device, num_sms;
  uint8_t *w_in_codes, *w_in_scales;    // [Nin][H/2], [Nin][H/16]: qkvz rows then ba rows
  float ts_qkvz, ts_ba;
  uint8_t *w_out_codes, *w_out_scales;  // [H][Vd/2], [H][Vd/16]
  float ts_wout;
  uint16_t *conv_w;                     // [C][K]
  float *A_log, *dt_bias, *norm_w;
  uint16_t *proj;                       // [prow][Nin] BF16 projection outputs
  uint8_t *y_codes, *y_scales;          // [prow][Vd/2], [prow][Vd/16]
  float *qn, *kn, *v, *beta, *gl, *o;     // prefill intermediates (head-major, chunk-padded)
  BatchWs bws;                          // large-batch decode intermediates, max_batch rows
  float *W, *Ut, *Am, *Gam;               // per (value head, 64-token chunk) products
  uint16_t *KTs = nullptr;                // per (key head, chunk) K^T for the tcgen05 chunk scan, split FP16
  float *Wsc = nullptr;                   // per (value head, chunk) FP16 scale of W
  float *Umax = nullptr;                  // per (value head, chunk) largest |Ut|
  uint16_t *conv_tmp;                   // [K-1][C]
  uint8_t *xq_codes, *xq_scales;        // [prow][H/2] and tiled scales: x as NVFP4 for the tensor-core GEMM
  uint8_t *w_in_sf_t, *w_out_sf_t;      // the weights' scales in the tiled layout tcgen05.cp reads
  uint8_t *w_in_tiles, *w_out_tiles;    // the weights' codes as pre-swizzled 16 KB MMA tiles
  uint8_t *w_in_mma, *w_out_mma;        // the weights in the warp-MMA one-row layout
  TcGemm tc_in, tc_out;                 // weight tensor maps of the two projections
  bool tc_in_ok, tc_out_ok;             // K % 256 == 0: the tcgen05 path applies
  int32_t *status;
  unsigned int *grid_bar;               // the fused decode kernel's grid barrier words
  std::vector<void *> allocs;
};

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return GDN_OK;
  if (e == cudaErrorMemoryAllocation) return GDN_E_OOM;
  return GDN_E_CUDA;
}

// Process-wide tuning knobs (gdn_set_tuning).
struct Tuning {
  int decode_gemm = 0;  // 0 auto, 1 CUDA-core GEMV, 2 tcgen05
  int split_in = 0;     // split-K of the in-projection on tensor cores (0 = automatic)
  int split_out = 0;    // split-K of the out-projection
  int fused = 0;        // one- and two-row decode as one persistent kernel: 0 auto (off), 1 off, 2 on
  int in_quant_fused = 0;  // decode in-projection on tensor cores quantises x itself: 0 auto (on), 1 off, 2 on
  int early_trigger = 0;   // out-projection of a decode step signals the next kernel early: 0 auto (tensor-core
                           // out-projection only), 1 off, 2 on
  int swizzled_tiles = 0;  // tensor-core weights from the pre-swizzled tile copy: 0 auto (on), 1 off, 2 on
  int mix_slices = 0;      // d_v slices per head in the mixing kernel: 0 auto, 1, 2, 4
  int gemv_mma = 0;        // one-row projections with warp-level MMA block products: 0 auto (on), 1 off, 2 on
  int batch_split = 0;     // decode mixing as prep / delta / gated-norm kernels: 0 and 1 off, 2 on
  int scan_tc = 0;         // prefill chunk scan: 0 auto (tcgen05 for d = 128), 1 FP32 CUDA cores, 2 warp MMA, 3 tcgen05
  int persist_gemm = 0;    // tensor-core projections as one persistent CTA per SM: 0 auto, 1 off, 2 streaming
                           // form whenever allowed, 3 weight-stationary form whenever allowed
  long long barrier_wait = 0;  // grid-barrier wait budget in SM cycles (0 = kWaitCycles)
  int proj_mix = 0;        // decode of up to 8 rows with the in-projection inside the mixing kernel: 0 auto (off),
                           // 1 off, 2 on
  int tile_in = 0;         // warp-MMA tile of the in- / out-projection (GemvArgs::mma_tile): 0 auto
  int tile_out = 0;
  int act_bulk = 0;        // warp-MMA activation rows by one bulk copy: 0 auto, 1 off, 2 on
};
Tuning g_tune;

// Automatic choice, measured on GB300 (decode stack, us per layer-step): up
// to four rows on the warp-MMA kernel (c1 13.6 vs 18.3, c2 15.1 vs 18.8, c4
// 17.2 vs 19.2), from five rows on the tensor cores (c8 22.0 vs 27.2, c16
// 31.6 vs 97.9 on the CUDA-core GEMV).
bool use_tensor_cores(int rows) {
  if (g_tune.decode_gemm == 1) return false;
  if (g_tune.decode_gemm == 2) return true;
  return rows > 4;
}
// Warp-MMA tiles (GemvArgs::mma_tile), measured on GB300: the in-projection of
// one row as two 16-row groups per CTA x four K slices (c1 13.6 vs 14.0 with
// four groups x two slices), of 2..4 rows as four groups x two slices (c2 15.1
// vs 17.2); the out-projection with K slices of 512 (K = 4096: one group x
// eight slices, 128 CTAs, its post-wait MMA phase 1.5 -> 0.9 us; K = 2048: two
// groups x four, the two-way head slice's c1 12.1 -> 10.4 us).
int tile_in(int rows) { return g_tune.tile_in ? g_tune.tile_in : (rows == 1 ? 1 : 3); }
int tile_out(int K) { return g_tune.tile_out ? g_tune.tile_out : (K >= 4096 ? 2 : 1); }
// Activation rows by one bulk copy per CTA when there are several rows (c2
// 16.1 -> 14.5 us, c4 18.1 -> 17.3) or many CTAs read the same row (the
// full-width in-projection's 386: c1 15.6 -> 15.2 us); one row in a grid of a
// few hundred CTAs or fewer is faster with per-thread loads (two-way slice
// c1 10.4 -> 9.8).
int mma_ctas(int tile, int N) {
  const int gpc = tile == 2 ? 1 : (tile == 3 ? 4 : 2);
  return ((N + 15) / 16 + gpc - 1) / gpc;
}
bool act_bulk(int tile, int N, int rows) {
  if (g_tune.act_bulk) return g_tune.act_bulk == 2;
  return rows > 1 || mma_ctas(tile, N) >= 256;
}
// Split-K for few activation rows: spreads the K loop of the 97 (in) or 16
// (out) weight tiles over 2 or 4 CTAs of a cluster (measured best at B 1..16).
int split_for(int knob_value, int rows, int dflt) {
  if (knob_value > 0) return knob_value;
  return rows <= 64 ? dflt : 0;
}

template <typename T>
cudaError_t ctx_alloc(gdn_ctx *c, T **p, size_t count) {
  void *q = nullptr;
  cudaError_t e = cudaMalloc(&q, count ? count * sizeof(T) : 16);
  if (e != cudaSuccess) return e;
  c->allocs.push_back(q);
  *p = static_cast<T *>(q);
  return cudaSuccess;
}

void ctx_free(gdn_ctx *c) {
  for (void *p : c->allocs) cudaFree(p);
  c->allocs.clear();
}

// Sets *bad to 1 when a scale byte is an E4M3 NaN (0x7F or 0xFF).
__global__ void scan_nan_scales(const uint8_t *s, size_t n, int32_t *bad) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    if ((s[i] & 0x7F) == 0x7F) flag_status(bad, GDN_E_BAD_SCALE);
}

gdn_status check_nvfp4(const gdn_nvfp4 &m) {
  if (!m.codes || !m.scales) return GDN_E_NULL;
  if (!aligned16(m.codes) || !aligned16(m.scales)) return GDN_E_ALIGN;
  if (!std::isfinite(m.tensor_scale)) return GDN_E_NONFINITE;
  if (!(m.tensor_scale > 0.0f)) return GDN_E_BAD_SCALE;
  return GDN_OK;
}

// W4A4 product of M activation rows (BF16 quantised on the fly, or NVFP4)
// against the N weight rows, 16 activation rows per pass.
cudaError_t run_gemv(GemvArgs g, const LaunchCtx &lc, int M) {
  const int K = g.K;
  for (int r0 = 0; r0 < M; r0 += 16) {
    GemvArgs p = g;
    p.M = M - r0 < 16 ? M - r0 : 16;
    if (g.a_bf16) p.a_bf16 = g.a_bf16 + (size_t)r0 * K;
    if (g.a_codes) {
      p.a_codes = g.a_codes + (size_t)r0 * (K / 2);
      p.a_scales = g.a_scales + (size_t)r0 * (K / 16);
    }
    if (g.row_slot) p.row_slot = g.row_slot + r0;
    p.c = static_cast<char *>(g.c) + (size_t)r0 * g.ldc * (g.c_is_bf16 ? 2 : 4);
    cudaError_t e = launch_gemv(p, lc);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

gdn_status check_state_args(gdn_ctx *ctx, const void *x, const void *out, const uint16_t *conv_state,
                            const void *ssm_state, int num_slots) {
  if (!ctx || !x || !out || !conv_state || !ssm_state) return GDN_E_NULL;
  if (!aligned16(x) || !aligned16(out) || !aligned16(conv_state) || !aligned16(ssm_state)) return GDN_E_ALIGN;
  if (num_slots < 1) return GDN_E_SHAPE;
  const size_t per_slot = (size_t)ctx->cfg.n_v_heads * ctx->cfg.d_v * ctx->cfg.d_k;
  if ((size_t)num_slots > ((size_t)1 << 40) / per_slot) return GDN_E_OVERFLOW;
  return GDN_OK;
}

MixArgs mix_args(gdn_ctx *c) {
  MixArgs m{};
  m.conv_w = c->conv_w;
  m.A_log = c->A_log;
  m.dt_bias = c->dt_bias;
  m.norm_w = c->norm_w;
  m.Hk = c->cfg.n_k_heads;
  m.Hv = c->cfg.n_v_heads;
  m.D = c->cfg.d_k;
  m.C = c->C;
  m.Kc = c->cfg.conv_kernel;
  m.l2_eps = c->cfg.l2_eps;
  m.rms_eps = c->cfg.rms_eps;
  m.ts_out = c->cfg.act_scale_out;
  m.status = c->status;
  m.slices = g_tune.mix_slices;
  m.state_bf16 = c->cfg.state_bf16;
  return m;
}

// x (BF16 rows, padding rows masked by row_slot) -> the in-projection
// (q|k|v|z|b|a, BF16, ldc = Nin) on tensor cores, or on the CUDA cores.
cudaError_t run_in_proj(gdn_ctx *ctx, const uint16_t *x, int rows, const int32_t *row_slot, int num_slots,
                        const LaunchCtx &lc, bool allow_tc, uint16_t *dst = nullptr) {
  if (!dst) dst = ctx->proj;
  const gdn_config &c = ctx->cfg;
  if (allow_tc && ctx->tc_in_ok && use_tensor_cores(rows)) {
    TcGemm t = ctx->tc_in;
    // up to 16 rows: the GEMM quantises x itself; more: a quantisation kernel first
    const bool fused_q = rows <= 16 && g_tune.in_quant_fused != 1;
    if (!fused_q) {
      cudaError_t e = launch_quantize(x, 0, rows, c.hidden, c.act_scale_in, ctx->xq_codes, ctx->xq_scales, ctx->status,
                                      lc.stream, row_slot, num_slots, lc.pdl, true);
      if (e != cudaSuccess) return e;
    } else {
      t.args.b_bf16 = x;
      t.args.b_row_slot = row_slot;
      t.args.b_num_slots = num_slots;
    }
    t.b_codes = ctx->xq_codes;
    t.b_scales = ctx->xq_scales;
    t.args.Ma = ctx->Nin;
    t.args.Nb = rows;
    t.args.K = c.hidden;
    t.args.c = dst;
    t.args.ldc = ctx->Nin;
    t.args.c_is_bf16 = 1;
    t.args.ts_a0 = ctx->ts_qkvz;
    t.args.ts_a1 = ctx->ts_ba;
    t.args.a_split = ctx->Nqkvz;
    t.args.ts_b = c.act_scale_in;
    t.args.a_const = 1;
    t.args.sfa_tiled = ctx->w_in_sf_t;
    t.args.a_tiles = g_tune.swizzled_tiles != 1 ? ctx->w_in_tiles : nullptr;
    t.args.sfb_tiled = ctx->xq_scales;
    t.args.status = ctx->status;
    t.split_k = split_for(g_tune.split_in, rows, 2);
    t.persist = g_tune.persist_gemm;
    return launch_tc_gemm(t, lc);
  }
  GemvArgs g{};
  g.a_bf16 = x;
  g.ts_a = c.act_scale_in;
  g.row_slot = row_slot;
  g.num_slots = num_slots;
  g.w_codes = ctx->w_in_codes;
  g.w_scales = ctx->w_in_scales;
  g.ts_w0 = ctx->ts_qkvz;
  g.ts_w1 = ctx->ts_ba;
  g.n_split = ctx->Nqkvz;
  g.c = dst;
  g.c_is_bf16 = 1;
  g.ldc = ctx->Nin;
  g.N = ctx->Nin;
  g.K = c.hidden;
  g.status = ctx->status;
  g.w_mma = g_tune.gemv_mma != 1 ? ctx->w_in_mma : nullptr;
  g.mma_tile = tile_in(rows);
  g.mma_bulk = act_bulk(g.mma_tile, g.N, rows);
  return run_gemv(g, lc, rows);
}

// Whether the out-projection of `rows` rows runs on tensor cores, so the
// mixing stage must write y's scales in the tiled layout.
bool out_proj_tiled(const gdn_ctx *ctx, int rows) { return ctx->tc_out_ok && use_tensor_cores(rows); }

// y (NVFP4 in the context's workspace) -> out (BF16 [rows][H]).
// early: the out-projection is the last kernel of a decode step and lets the
// next kernel in the stream launch before it waits (TcArgs::early_trigger).
cudaError_t run_out_proj(gdn_ctx *ctx, uint16_t *out, int rows, const LaunchCtx &lc, bool allow_tc,
                         bool early = false) {
  const gdn_config &c = ctx->cfg;
  if (allow_tc && ctx->tc_out_ok && use_tensor_cores(rows)) {
    TcGemm t = ctx->tc_out;
    t.b_codes = ctx->y_codes;
    t.b_scales = ctx->y_scales;
    t.args.Ma = c.hidden;
    t.args.Nb = rows;
    t.args.K = ctx->Vd;
    t.args.c = out;
    t.args.ldc = c.hidden;
    t.args.c_is_bf16 = 1;
    t.args.ts_a0 = t.args.ts_a1 = ctx->ts_wout;
    t.args.a_split = c.hidden;
    t.args.ts_b = c.act_scale_out;
    t.args.a_const = 1;
    t.args.sfa_tiled = ctx->w_out_sf_t;
    t.args.a_tiles = g_tune.swizzled_tiles != 1 ? ctx->w_out_tiles : nullptr;
    t.args.sfb_tiled = ctx->y_scales;  // written tiled by the mixing stage (out_proj_tiled)
    t.args.status = ctx->status;
    t.split_k = split_for(g_tune.split_out, rows, 4);
    t.persist = g_tune.persist_gemm;
    t.args.early_trigger = early && g_tune.early_trigger != 1;
    return launch_tc_gemm(t, lc);
  }
  GemvArgs o{};
  o.a_codes = ctx->y_codes;
  o.a_scales = ctx->y_scales;
  o.ts_a = c.act_scale_out;
  o.w_codes = ctx->w_out_codes;
  o.w_scales = ctx->w_out_scales;
  o.ts_w0 = o.ts_w1 = ctx->ts_wout;
  o.n_split = c.hidden;
  o.c = out;
  o.c_is_bf16 = 1;
  o.ldc = c.hidden;
  o.N = c.hidden;
  o.K = ctx->Vd;
  o.status = ctx->status;
  o.w_mma = g_tune.gemv_mma != 1 ? ctx->w_out_mma : nullptr;
  o.mma_tile = tile_out(ctx->Vd);
  o.mma_bulk = act_bulk(o.mma_tile, c.hidden, rows);
  // measured slower for the one-row GEMV chain (its weight prefetch then
  // competes with the mixing kernel), so only on request
  o.early_trigger = early && g_tune.early_trigger == 2 && rows <= 16;  // one launch, the step's last
  return run_gemv(o, lc, rows);
}

// The fused in-projection + mixing kernel's arguments (y row-major NVFP4).
PmArgs pm_args(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, uint16_t *conv_state, void *ssm_state,
               int num_slots, uint8_t *y_codes, uint8_t *y_scales) {
  const gdn_config &c = ctx->cfg;
  PmArgs p{};
  p.x = x;
  p.slot_ids = slot_ids;
  p.B = B;
  p.num_slots = num_slots;
  p.w_mma = ctx->w_in_mma;
  p.w_codes = ctx->w_in_codes;
  p.w_scales = ctx->w_in_scales;
  p.ts_in = c.act_scale_in;
  p.ts_qkvz = ctx->ts_qkvz;
  p.ts_ba = ctx->ts_ba;
  p.H = c.hidden;
  p.Hk = c.n_k_heads;
  p.Hv = c.n_v_heads;
  p.Nqkvz = ctx->Nqkvz;
  p.C = ctx->C;
  p.Kc = c.conv_kernel;
  p.conv_w = ctx->conv_w;
  p.A_log = ctx->A_log;
  p.dt_bias = ctx->dt_bias;
  p.norm_w = ctx->norm_w;
  p.l2_eps = c.l2_eps;
  p.rms_eps = c.rms_eps;
  p.ts_out = c.act_scale_out;
  p.conv_state = conv_state;
  p.ssm_state = ssm_state;
  p.state_bf16 = c.state_bf16;
  p.y_codes = y_codes;
  p.y_scales = y_scales;
  p.status = ctx->status;
  return p;
}

// The warp-MMA out-projection of B <= 8 NVFP4 rows (row-major scales).
GemvArgs out_gemv_args(gdn_ctx *ctx, const uint8_t *y_codes, const uint8_t *y_scales, int B, uint16_t *out,
                       bool early) {
  const gdn_config &c = ctx->cfg;
  GemvArgs o{};
  o.a_codes = y_codes;
  o.a_scales = y_scales;
  o.ts_a = c.act_scale_out;
  o.w_codes = ctx->w_out_codes;
  o.w_scales = ctx->w_out_scales;
  o.ts_w0 = o.ts_w1 = ctx->ts_wout;
  o.n_split = c.hidden;
  o.c = out;
  o.c_is_bf16 = 1;
  o.ldc = c.hidden;
  o.M = B;
  o.N = c.hidden;
  o.K = ctx->Vd;
  o.status = ctx->status;
  o.w_mma = ctx->w_out_mma;
  o.mma_tile = tile_out(ctx->Vd);
  o.mma_bulk = act_bulk(o.mma_tile, c.hidden, B);
  o.early_trigger = early ? 1 : 0;
  return o;
}

bool pm_path(const gdn_ctx *ctx, int B) {
  const gdn_config &c = ctx->cfg;
  return ctx->w_in_mma && ctx->w_out_mma && proj_mix_ok(c.hidden, c.n_k_heads, c.n_v_heads, c.d_k, c.conv_kernel, B);
}

FusedArgs fused_args(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, uint16_t *out,
                     uint16_t *conv_state, float *ssm_state, int num_slots) {
  const gdn_config &c = ctx->cfg;
  FusedArgs f{};
  f.w_in_codes = ctx->w_in_codes;
  f.w_in_scales = ctx->w_in_scales;
  f.w_out_codes = ctx->w_out_codes;
  f.w_out_scales = ctx->w_out_scales;
  f.ts_qkvz = ctx->ts_qkvz;
  f.ts_ba = ctx->ts_ba;
  f.ts_wout = ctx->ts_wout;
  f.Nqkvz = ctx->Nqkvz;
  f.Nin = ctx->Nin;
  f.conv_w = ctx->conv_w;
  f.A_log = ctx->A_log;
  f.dt_bias = ctx->dt_bias;
  f.norm_w = ctx->norm_w;
  f.H = c.hidden;
  f.Hk = c.n_k_heads;
  f.Hv = c.n_v_heads;
  f.D = c.d_k;
  f.C = ctx->C;
  f.Kc = c.conv_kernel;
  f.Vd = ctx->Vd;
  f.l2_eps = c.l2_eps;
  f.rms_eps = c.rms_eps;
  f.ts_in = c.act_scale_in;
  f.ts_out = c.act_scale_out;
  f.x = x;
  f.slot_ids = slot_ids;
  f.B = B;
  f.num_slots = num_slots;
  f.out = out;
  f.conv_state = conv_state;
  f.ssm_state = ssm_state;
  f.proj = ctx->proj;
  f.y_codes = ctx->y_codes;
  f.y_scales = ctx->y_scales;
  f.bar = ctx->grid_bar;
  f.wait_cycles = g_tune.barrier_wait > 0 ? g_tune.barrier_wait : kWaitCycles;
  f.status = ctx->status;
  return f;
}

}  // namespace

extern "C" {

gdn_status gdn_set_tuning(int knob, int value) {
  switch (knob) {
    case 0:
      if (value < 0 || value > 2) return GDN_E_RANGE;
      g_tune.decode_gemm = value;
      return GDN_OK;
    case 1:
    case 2:
      if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return GDN_E_RANGE;
      (knob == 1 ? g_tune.split_in : g_tune.split_out) = value;
      return GDN_OK;
    case 3:
      if (value < 0 || value > 2) return GDN_E_RANGE;
      g_tune.fused = value;
      return GDN_OK;
    case 4:
    case 5:
    case 6:
      if (value < 0 || value > 2) return GDN_E_RANGE;
      (knob == 4 ? g_tune.in_quant_fused : knob == 5 ? g_tune.early_trigger : g_tune.swizzled_tiles) = value;
      return GDN_OK;
    case 7:
      if (value != 0 && value != 1 && value != 2 && value != 4) return GDN_E_RANGE;
      g_tune.mix_slices = value;
      return GDN_OK;
    case 8:
      if (value < 0 || value > 2) return GDN_E_RANGE;
      g_tune.gemv_mma = value;
      return GDN_OK;
    case 9:
      if (value < 0 || value > 2) return GDN_E_RANGE;
      g_tune.batch_split = value;
      return GDN_OK;
    case 10:
      if (value < 0 || value > 3) return GDN_E_RANGE;
      g_tune.scan_tc = value;
      return GDN_OK;
    case 11:
      if (value < 0 || value > 3) return GDN_E_RANGE;
      g_tune.persist_gemm = value;
      return GDN_OK;
    case 12:
      if (value < 0) return GDN_E_RANGE;
      g_tune.barrier_wait = value;
      return GDN_OK;
    case 13:
      if (value < 0 || value > 2) return GDN_E_RANGE;
      g_tune.proj_mix = value;
      return GDN_OK;
    case 14:
    case 15:
      if (value < 0 || value > 3) return GDN_E_RANGE;
      (knob == 14 ? g_tune.tile_in : g_tune.tile_out) = value;
      return GDN_OK;
    case 16:
      if (value < 0 || value > 2) return GDN_E_RANGE;
      g_tune.act_bulk = value;
      return GDN_OK;
    default:
      return GDN_E_RANGE;
  }
}

const char *gdn_status_string(int s) {
  static const char *names[] = {"GDN_OK",          "GDN_E_NULL",     "GDN_E_SHAPE",   "GDN_E_ALIGN",
                                "GDN_E_NONFINITE", "GDN_E_BAD_SCALE", "GDN_E_RANGE",   "GDN_E_OVERFLOW",
                                "GDN_E_CUDA",      "GDN_E_OOM",      "GDN_E_TIMEOUT", "GDN_E_STATE"};
  if (s < 0 || s > 11) return "GDN_E_UNKNOWN";
  return names[s];
}

gdn_status gdn_create(const gdn_config *cfg, const gdn_weights *w, void *stream, gdn_ctx **out) {
  if (!out) return GDN_E_NULL;
  *out = nullptr;
  if (!cfg || !w) return GDN_E_NULL;
  const gdn_config c = *cfg;
  if (c.hidden <= 0 || c.n_k_heads <= 0 || c.n_v_heads <= 0 || c.max_batch < 1 || c.max_batch > 256 ||
      c.max_prefill_tokens < 0)
    return GDN_E_SHAPE;
  if (c.hidden % 64 || c.n_v_heads % c.n_k_heads || c.n_v_heads / c.n_k_heads > 8) return GDN_E_SHAPE;
  if (c.d_k != c.d_v || (c.d_k != 32 && c.d_k != 64 && c.d_k != 128)) return GDN_E_SHAPE;
  if (c.conv_kernel < 2 || c.conv_kernel > 4) return GDN_E_SHAPE;
  if (c.state_bf16 != 0 && c.state_bf16 != 1) return GDN_E_SHAPE;
  if ((c.n_v_heads * c.d_v) % 64) return GDN_E_SHAPE;
  if (!std::isfinite(c.rms_eps) || !std::isfinite(c.l2_eps) || !std::isfinite(c.act_scale_in) ||
      !std::isfinite(c.act_scale_out))
    return GDN_E_NONFINITE;
  if (c.rms_eps < 0 || c.l2_eps < 0 || !(c.act_scale_in > 0) || !(c.act_scale_out > 0)) return GDN_E_BAD_SCALE;
  gdn_status st;
  if ((st = check_nvfp4(w->qkvz)) != GDN_OK || (st = check_nvfp4(w->ba)) != GDN_OK ||
      (st = check_nvfp4(w->out)) != GDN_OK)
    return st;
  if (!w->conv_w || !w->A_log || !w->dt_bias || !w->norm_w) return GDN_E_NULL;
  if (!aligned16(w->conv_w) || !aligned16(w->A_log) || !aligned16(w->dt_bias) || !aligned16(w->norm_w))
    return GDN_E_ALIGN;
  const long long H = c.hidden, Hk = c.n_k_heads, Hv = c.n_v_heads, D = c.d_k;
  const long long Nqkvz = 2 * Hk * D + 2 * Hv * D, Nba = 2 * Hv, Nin = Nqkvz + Nba;
  const long long Cc = 2 * Hk * D + Hv * D, Vd = Hv * D;
  const long long prow = c.max_batch > c.max_prefill_tokens ? c.max_batch : c.max_prefill_tokens;
  if (Nin * H > (1LL << 31) || H * Vd > (1LL << 31) || prow * Nin > (1LL << 34) || Vd > 16384 || H > 16384)
    return GDN_E_OVERFLOW;

  gdn_ctx *ctx = new (std::nothrow) gdn_ctx();
  if (!ctx) return GDN_E_OOM;
  ctx->cfg = c;
  ctx->Nqkvz = (int)Nqkvz;
  ctx->Nba = (int)Nba;
  ctx->Nin = (int)Nin;
  ctx->C = (int)Cc;
  ctx->Vd = (int)Vd;
  ctx->prow = (int)prow;
  ctx->ts_qkvz = w->qkvz.tensor_scale;
  ctx->ts_ba = w->ba.tensor_scale;
  ctx->ts_wout = w->out.tensor_scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  const long long T = c.max_prefill_tokens;
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->w_in_codes, Nin * H / 2);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->w_in_scales, Nin * H / 16);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->w_out_codes, H * Vd / 2);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->w_out_scales, H * Vd / 16);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->conv_w, Cc * c.conv_kernel);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->A_log, Hv);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->dt_bias, Hv);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->norm_w, D);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->proj, prow * Nin);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->y_codes, prow * Vd / 2);
  {
    const size_t mb = (size_t)c.max_batch;
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->bws.qn, mb * Hk * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->bws.kn, mb * Hk * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->bws.v, mb * Hv * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->bws.beta, mb * Hv);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->bws.gl, mb * Hv);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->bws.o, mb * Hv * D);
  }
  // scales sized for both layouts: row-major, or tiled (rows padded to 128)
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->y_scales, sf_tiled_bytes((int)prow, (int)Vd));
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->w_in_sf_t, sf_tiled_bytes((int)Nin, (int)H));
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->w_out_sf_t, sf_tiled_bytes((int)H, (int)Vd));
  if (e == cudaSuccess && H % 256 == 0) e = ctx_alloc(ctx, &ctx->w_in_tiles, swizzled_tiles_bytes((int)Nin, (int)H));
  if (e == cudaSuccess && Vd % 256 == 0) e = ctx_alloc(ctx, &ctx->w_out_tiles, swizzled_tiles_bytes((int)H, (int)Vd));
  if (e == cudaSuccess && H % 256 == 0) e = ctx_alloc(ctx, &ctx->w_in_mma, mma_tiles_bytes((int)Nin, (int)H));
  if (e == cudaSuccess && Vd % 256 == 0) e = ctx_alloc(ctx, &ctx->w_out_mma, mma_tiles_bytes((int)H, (int)Vd));
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->status, 1);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->grid_bar, 4);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->conv_tmp, (c.conv_kernel - 1) * Cc);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->xq_codes, prow * H / 2);
  if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->xq_scales, sf_tiled_bytes((int)prow, (int)H));
  if (T > 0) {
    const long long Tp = (T + 63) / 64 * 64;
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->qn, Tp * Hk * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->kn, Tp * Hk * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->v, Tp * Hv * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->o, T * Hv * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->beta, Tp * Hv);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->gl, Tp * Hv);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->W, Tp * Hv * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->Ut, Tp * Hv * D);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->Am, Tp * Hv * 64);
    if (e == cudaSuccess) e = ctx_alloc(ctx, &ctx->Gam, Tp * Hv);
    if (e == cudaSuccess && D == 128) e = ctx_alloc(ctx, &ctx->KTs, 2 * Tp * Hk * D);
    if (e == cudaSuccess && D == 128) e = ctx_alloc(ctx, &ctx->Wsc, Tp / 64 * Hv);
    if (e == cudaSuccess && D == 128) e = ctx_alloc(ctx, &ctx->Umax, Tp / 64 * Hv);
  }
  // weights into the kernels' layout: [qkvz; ba] as one matrix for one pass over x
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->w_in_codes, w->qkvz.codes, Nqkvz * H / 2, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ctx->w_in_codes + Nqkvz * H / 2, w->ba.codes, Nba * H / 2, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->w_in_scales, w->qkvz.scales, Nqkvz * H / 16, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ctx->w_in_scales + Nqkvz * H / 16, w->ba.scales, Nba * H / 16, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->w_out_codes, w->out.codes, H * Vd / 2, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->w_out_scales, w->out.scales, H * Vd / 16, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ctx->conv_w, w->conv_w, Cc * c.conv_kernel * 2, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->A_log, w->A_log, Hv * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->dt_bias, w->dt_bias, Hv * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->norm_w, w->norm_w, D * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && H % 64 == 0) e = launch_tile_scales(ctx->w_in_scales, (int)Nin, (int)H, ctx->w_in_sf_t, s);
  if (e == cudaSuccess && Vd % 64 == 0) e = launch_tile_scales(ctx->w_out_scales, (int)H, (int)Vd, ctx->w_out_sf_t, s);
  if (e == cudaSuccess && H % 256 == 0) e = launch_swizzle_tiles(ctx->w_in_codes, (int)Nin, (int)H, ctx->w_in_tiles, s);
  if (e == cudaSuccess && Vd % 256 == 0) e = launch_swizzle_tiles(ctx->w_out_codes, (int)H, (int)Vd, ctx->w_out_tiles, s);
  if (e == cudaSuccess && H % 256 == 0)
    e = launch_mma_tiles(ctx->w_in_codes, ctx->w_in_scales, (int)Nin, (int)H, ctx->w_in_mma, s);
  if (e == cudaSuccess && Vd % 256 == 0)
    e = launch_mma_tiles(ctx->w_out_codes, ctx->w_out_scales, (int)H, (int)Vd, ctx->w_out_mma, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->status, 0, 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->grid_bar, 0, 16, s);
  if (e == cudaSuccess) {
    scan_nan_scales<<<256, 256, 0, s>>>(ctx->w_in_scales, (size_t)(Nin * H / 16), ctx->status);
    scan_nan_scales<<<256, 256, 0, s>>>(ctx->w_out_scales, (size_t)(H * Vd / 16), ctx->status);
    e = cudaGetLastError();
  }
  int32_t flag = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&flag, ctx->status, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess || flag != 0) {
    gdn_status r = e != cudaSuccess ? cuda_status(e) : (gdn_status)flag;
    ctx_free(ctx);
    delete ctx;
    return r;
  }
  ctx->tc_in_ok = H % 256 == 0 && tc_make_weight_maps(ctx->tc_in, ctx->w_in_codes, ctx->w_in_scales, (int)Nin, (int)H);
  ctx->tc_out_ok = Vd % 256 == 0 && tc_make_weight_maps(ctx->tc_out, ctx->w_out_codes, ctx->w_out_scales, (int)H, (int)Vd);
  *out = ctx;
  return GDN_OK;
}

gdn_status gdn_destroy(gdn_ctx *ctx) {
  if (!ctx) return GDN_OK;
  ctx_free(ctx);
  delete ctx;
  return GDN_OK;
}

gdn_status nvfp4_quantize(const void *x, int x_is_f32, int rows, int cols, float tensor_scale, uint8_t *codes,
                          uint8_t *scales, int32_t *dev_status, void *stream) {
  if (rows < 0 || cols <= 0 || cols % 16) return GDN_E_SHAPE;
  if (rows == 0) return GDN_OK;
  if (!x || !codes || !scales) return GDN_E_NULL;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return GDN_E_ALIGN;
  if (!std::isfinite(tensor_scale)) return GDN_E_NONFINITE;
  if (!(tensor_scale > 0)) return GDN_E_BAD_SCALE;
  if ((long long)rows * cols > (1LL << 40)) return GDN_E_OVERFLOW;
  return cuda_status(launch_quantize(x, x_is_f32, rows, cols, tensor_scale, codes, scales, dev_status,
                                     static_cast<cudaStream_t>(stream)));
}

gdn_status nvfp4_gemm(const gdn_nvfp4 *A, int M, const gdn_nvfp4 *B, int N, int K, void *C, int c_is_bf16,
                      void *stream) {
  if (!A || !B) return GDN_E_NULL;
  if (M < 0 || N < 0 || K <= 0 || K % 64) return GDN_E_SHAPE;
  if (M == 0 || N == 0) return GDN_OK;
  gdn_status st;
  if ((st = check_nvfp4(*A)) != GDN_OK || (st = check_nvfp4(*B)) != GDN_OK) return st;
  if (!C) return GDN_E_NULL;
  if (!aligned16(C)) return GDN_E_ALIGN;
  if ((long long)N * K > (1LL << 31) || (long long)M * K > (1LL << 40) || K > 32768) return GDN_E_OVERFLOW;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_status(e);
  LaunchCtx lc{static_cast<cudaStream_t>(stream), sms, false};  // B may come from a preceding kernel
  if (K % 256 == 0 && !(g_tune.decode_gemm == 1 && M <= 16)) {
    // tensor cores: B (N rows) is the MMA's A operand, A (M rows) its B operand
    TcGemm t{};
    if (!tc_make_weight_maps(t, B->codes, B->scales, N, K)) return GDN_E_CUDA;
    t.b_codes = A->codes;
    t.b_scales = A->scales;
    t.args.Ma = N;
    t.args.Nb = M;
    t.args.K = K;
    t.args.c = C;
    t.args.ldc = N;
    t.args.c_is_bf16 = c_is_bf16 ? 1 : 0;
    t.args.ts_a0 = t.args.ts_a1 = B->tensor_scale;
    t.args.a_split = N;
    t.args.ts_b = A->tensor_scale;
    t.args.a_const = 0;
    return cuda_status(launch_tc_gemm(t, lc));
  }
  if ((size_t)16 * (K >> 6) * (4 * 2 * 16 + 16) > 200 * 1024) return GDN_E_SHAPE;
  GemvArgs g{};
  g.a_codes = A->codes;
  g.a_scales = A->scales;
  g.ts_a = A->tensor_scale;
  g.w_codes = B->codes;
  g.w_scales = B->scales;
  g.ts_w0 = g.ts_w1 = B->tensor_scale;
  g.n_split = N;
  g.c = C;
  g.c_is_bf16 = c_is_bf16 ? 1 : 0;
  g.ldc = N;
  g.N = N;
  g.K = K;
  return cuda_status(run_gemv(g, lc, M));
}

gdn_status gdn_decode_step(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, uint16_t *out,
                           uint16_t *conv_state, void *ssm_state, int num_slots, void *stream) {
  gdn_status st = check_state_args(ctx, x, out, conv_state, ssm_state, num_slots);
  if (st != GDN_OK) return st;
  if (!slot_ids) return GDN_E_NULL;
  if (!aligned16(slot_ids)) return GDN_E_ALIGN;
  if (B < 1 || B > ctx->cfg.max_batch) return GDN_E_SHAPE;
  LaunchCtx lc{static_cast<cudaStream_t>(stream), ctx->num_sms, true};
  // The persistent single-kernel step (fused.cu) is correct but measured slower
  // on GB300 (c1 20.8 vs 14.6 us per layer-step: each grid barrier costs
  // ~2.5 us, more than a PDL kernel boundary), so it runs only on request.
  if (g_tune.fused == 2 && g_tune.decode_gemm != 2 && B <= 2 && !ctx->cfg.state_bf16) {
    FusedArgs f = fused_args(ctx, x, slot_ids, B, out, conv_state, static_cast<float *>(ssm_state), num_slots);
    if (fused_plan(f, ctx->num_sms)) {
      // fresh barrier words for every launch: a launch whose barrier gave up
      // leaves nothing behind for the next one
      cudaError_t e = cudaMemsetAsync(ctx->grid_bar, 0, 16, lc.stream);
      if (e != cudaSuccess) return cuda_status(e);
      return cuda_status(launch_fused(f, lc));
    }
  }
  if (g_tune.proj_mix == 2 && g_tune.decode_gemm != 2 && pm_path(ctx, B)) {
    // projections + mixing as one cluster kernel, then the warp-MMA out-projection
    cudaError_t e = launch_proj_mix(pm_args(ctx, x, slot_ids, B, conv_state, ssm_state, num_slots, ctx->y_codes,
                                            ctx->y_scales), lc);
    if (e != cudaSuccess) return cuda_status(e);
    // the step's last kernel lets the next one start at once: every kernel of
    // this library that can follow reads only weights (and slot ids) before
    // its own dependency wait
    return cuda_status(launch_gemv_mma(out_gemv_args(ctx, ctx->y_codes, ctx->y_scales, B, out,
                                                     g_tune.early_trigger != 1), lc));
  }
  cudaError_t e = run_in_proj(ctx, x, B, slot_ids, num_slots, lc, true);
  if (e != cudaSuccess) return cuda_status(e);
  MixArgs m = mix_args(ctx);
  m.qkvz = ctx->proj;
  m.ld_qkvz = ctx->Nin;
  m.ba = ctx->proj + ctx->Nqkvz;
  m.ld_ba = ctx->Nin;
  m.slot_ids = slot_ids;
  m.B = B;
  m.num_slots = num_slots;
  m.conv_state = conv_state;
  m.ssm_state = ssm_state;
  m.y_codes = ctx->y_codes;
  m.y_scales = ctx->y_scales;
  m.y_sf_tiled = out_proj_tiled(ctx, B) ? 1 : 0;
  m.y_f32 = nullptr;
  // the mixing as three kernels (bit-identical) only on request: the fused
  // kernel's streaming form measured faster at every batch (96: 91.4 against
  // 100.6 us per layer-step, 128: 109.3 against 119.9, 256: 194.8 against 209.1)
  const bool split = g_tune.batch_split == 2;
  e = split ? launch_batch_mix(m, ctx->bws, lc) : launch_mix(m, lc);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(run_out_proj(ctx, out, B, lc, true, true));
}

gdn_status gdn_verify(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, int r, uint16_t *out,
                      const uint16_t *conv_state, const void *ssm_state, int num_slots, uint16_t *snap_conv,
                      void *snap_ssm, void *stream) {
  gdn_status st = check_state_args(ctx, x, out, conv_state, ssm_state, num_slots);
  if (st != GDN_OK) return st;
  if (!slot_ids || !snap_conv || !snap_ssm) return GDN_E_NULL;
  if (!aligned16(slot_ids) || !aligned16(snap_conv) || !aligned16(snap_ssm)) return GDN_E_ALIGN;
  if (B < 1 || r < 1 || (long long)B * r > ctx->cfg.max_batch) return GDN_E_SHAPE;
  const gdn_config &c = ctx->cfg;
  const int rows = B * r;
  LaunchCtx lc{static_cast<cudaStream_t>(stream), ctx->num_sms, true};
  // every candidate token's projections at once: they do not depend on the state
  cudaError_t e = run_in_proj(ctx, x, rows, nullptr, 0, lc, true);
  if (e != cudaSuccess) return cuda_status(e);
  const size_t conv_elems = (size_t)(c.conv_kernel - 1) * ctx->C;
  const size_t ssm_elems = (size_t)c.n_v_heads * c.d_v * c.d_k;
  const size_t esz = c.state_bf16 ? 2 : 4;
  for (int t = 0; t < r; ++t) {  // the recurrence, token by token
    MixArgs m = mix_args(ctx);
    m.qkvz = ctx->proj;
    m.ld_qkvz = ctx->Nin;
    m.ba = ctx->proj + ctx->Nqkvz;
    m.ld_ba = ctx->Nin;
    m.slot_ids = slot_ids;
    m.B = B;
    m.num_slots = num_slots;
    m.conv_state = const_cast<uint16_t *>(conv_state);  // read only: writes go to the snapshots
    m.ssm_state = const_cast<void *>(ssm_state);
    m.io_mul = r;
    m.io_add = t;
    m.conv_src = t ? snap_conv + (size_t)(t - 1) * conv_elems : nullptr;
    m.conv_dst = snap_conv + (size_t)t * conv_elems;
    m.conv_row_stride = (size_t)r * conv_elems;
    m.ssm_src = t ? static_cast<const char *>(snap_ssm) + (size_t)(t - 1) * ssm_elems * esz : nullptr;
    m.ssm_dst = static_cast<char *>(snap_ssm) + (size_t)t * ssm_elems * esz;
    m.ssm_row_stride = (size_t)r * ssm_elems;
    m.y_codes = ctx->y_codes;
    m.y_scales = ctx->y_scales;
    m.y_sf_tiled = out_proj_tiled(ctx, rows) ? 1 : 0;
    m.y_f32 = nullptr;
    // token t > 0 reads the snapshot token t-1 wrote: no early start
    LaunchCtx lm = lc;
    if (t > 0) lm.pdl = false;
    e = launch_mix(m, lm);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return cuda_status(run_out_proj(ctx, out, rows, lc, true));
}

gdn_status gdn_verify_commit(gdn_ctx *ctx, const int32_t *slot_ids, int B, int r, const int32_t *accepted,
                             const uint16_t *snap_conv, const void *snap_ssm, uint16_t *conv_state, void *ssm_state,
                             int num_slots, void *stream) {
  if (!ctx || !slot_ids || !accepted || !snap_conv || !snap_ssm || !conv_state || !ssm_state) return GDN_E_NULL;
  if (!aligned16(snap_conv) || !aligned16(snap_ssm) || !aligned16(conv_state) || !aligned16(ssm_state))
    return GDN_E_ALIGN;
  if (B < 1 || r < 1 || (long long)B * r > ctx->cfg.max_batch || num_slots < 1) return GDN_E_SHAPE;
  const gdn_config &c = ctx->cfg;
  VerifyCommitArgs v{};
  v.slot_ids = slot_ids;
  v.accepted = accepted;
  v.B = B;
  v.r = r;
  v.num_slots = num_slots;
  v.snap_ssm = snap_ssm;
  v.snap_conv = snap_conv;
  v.ssm_state = ssm_state;
  v.conv_state = conv_state;
  v.ssm_bytes = (size_t)c.n_v_heads * c.d_v * c.d_k * (c.state_bf16 ? 2 : 4);
  v.conv_bytes = (size_t)(c.conv_kernel - 1) * ctx->C * 2;
  v.status = ctx->status;
  return cuda_status(launch_verify_commit(v, static_cast<cudaStream_t>(stream)));
}

gdn_status kda_step(const float *q, const float *k, const float *v, const float *g, const float *beta, void *state,
                    int state_bf16, int M, int H, int d, float *o, void *stream) {
  if (!q || !k || !v || !g || !beta || !state || !o) return GDN_E_NULL;
  if (M < 1 || H < 1 || (d != 32 && d != 64 && d != 128) || (state_bf16 != 0 && state_bf16 != 1)) return GDN_E_SHAPE;
  if ((long long)M * H > (1LL << 24)) return GDN_E_OVERFLOW;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) || !aligned16(state) ||
      !aligned16(o))
    return GDN_E_ALIGN;
  KdaArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.state = state;
  a.o = o;
  a.M = M;
  a.H = H;
  a.D = d;
  a.state_bf16 = state_bf16;
  return cuda_status(launch_kda(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_in_proj(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, uint16_t *proj,
                       void *stream) {
  if (!ctx || !x || !proj) return GDN_E_NULL;
  if (!aligned16(x) || !aligned16(proj) || (slot_ids && !aligned16(slot_ids))) return GDN_E_ALIGN;
  if (B < 1 || B > ctx->prow) return GDN_E_SHAPE;  // up to max(max_batch, max_prefill_tokens) rows
  LaunchCtx lc{static_cast<cudaStream_t>(stream), ctx->num_sms, false};
  // a row is zero when its slot id is negative (no slot range to check here)
  return cuda_status(run_in_proj(ctx, x, B, slot_ids, 0x7fffffff, lc, true, proj));
}

gdn_status gdn_mix_step(gdn_ctx *ctx, const uint16_t *qkvz, const uint16_t *ba, const int32_t *slot_ids, int B,
                        float *y, uint16_t *conv_state, void *ssm_state, int num_slots, void *stream) {
  gdn_status st = check_state_args(ctx, qkvz, y, conv_state, ssm_state, num_slots);
  if (st != GDN_OK) return st;
  if (!ba || !slot_ids) return GDN_E_NULL;
  if (!aligned16(ba) || !aligned16(slot_ids)) return GDN_E_ALIGN;
  if (B < 1 || B > ctx->cfg.max_batch) return GDN_E_SHAPE;
  // no programmatic launch: the mixing kernel reads the state before its
  // griddepcontrol.wait, so it must not overlap a preceding decode step
  LaunchCtx lc{static_cast<cudaStream_t>(stream), ctx->num_sms, false};
  MixArgs m = mix_args(ctx);
  m.qkvz = qkvz;
  m.ld_qkvz = ctx->Nqkvz;
  m.ba = ba;
  m.ld_ba = ctx->Nba;
  m.slot_ids = slot_ids;
  m.B = B;
  m.num_slots = num_slots;
  m.conv_state = conv_state;
  m.ssm_state = ssm_state;
  m.y_codes = nullptr;
  m.y_scales = nullptr;
  m.y_f32 = y;
  return cuda_status(launch_mix(m, lc));
}

gdn_status gdn_prefill(gdn_ctx *ctx, const uint16_t *x, int T, int slot, int init_zero, uint16_t *out,
                       uint16_t *conv_state, void *ssm_state, int num_slots, void *stream) {
  gdn_status st = check_state_args(ctx, x, out, conv_state, ssm_state, num_slots);
  if (st != GDN_OK) return st;
  if (T < 1 || T > ctx->cfg.max_prefill_tokens) return GDN_E_SHAPE;
  if (slot < 0 || slot >= num_slots) return GDN_E_RANGE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchCtx lc{s, ctx->num_sms, true};
  const gdn_config &c = ctx->cfg;
  const int D = c.d_k;
  uint16_t *cst = conv_state + (size_t)slot * (c.conv_kernel - 1) * ctx->C;
  const size_t s_elem = c.state_bf16 ? 2 : 4;
  void *S = static_cast<char *>(ssm_state) + (size_t)slot * c.n_v_heads * D * D * s_elem;
  cudaError_t e = cudaSuccess;
  if (init_zero) {
    e = cudaMemsetAsync(cst, 0, (size_t)(c.conv_kernel - 1) * ctx->C * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(S, 0, (size_t)c.n_v_heads * D * D * s_elem, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  e = run_in_proj(ctx, x, T, nullptr, 0, lc, true);
  if (e != cudaSuccess) return cuda_status(e);
  PrefillArgs p{};
  p.proj = ctx->proj;
  p.ld = ctx->Nin;
  p.T = T;
  p.conv_state = cst;
  p.ssm = S;
  p.state_bf16 = c.state_bf16;
  p.scan_tc = g_tune.scan_tc == 1 ? 0 : (g_tune.scan_tc == 2 || D != 128) ? 1 : 2;
  p.conv_w = ctx->conv_w;
  p.A_log = ctx->A_log;
  p.dt_bias = ctx->dt_bias;
  p.norm_w = ctx->norm_w;
  p.Hk = c.n_k_heads;
  p.Hv = c.n_v_heads;
  p.D = D;
  p.C = ctx->C;
  p.Kc = c.conv_kernel;
  p.l2_eps = c.l2_eps;
  p.rms_eps = c.rms_eps;
  p.ts_out = c.act_scale_out;
  p.Tp = (T + 63) / 64 * 64;
  p.qn = ctx->qn;
  p.kn = ctx->kn;
  p.v = ctx->v;
  p.beta = ctx->beta;
  p.gl = ctx->gl;
  p.W = ctx->W;
  p.Ut = ctx->Ut;
  p.Am = ctx->Am;
  p.Gam = ctx->Gam;
  // the tcgen05 path writes its split q, k, W and A over the FP32 ones (same bytes)
  p.Qs = p.scan_tc == 2 ? reinterpret_cast<uint16_t *>(ctx->qn) : nullptr;
  p.Ks = p.scan_tc == 2 ? reinterpret_cast<uint16_t *>(ctx->kn) : nullptr;
  p.Ws = p.scan_tc == 2 ? reinterpret_cast<uint16_t *>(ctx->W) : nullptr;
  p.As = p.scan_tc == 2 ? reinterpret_cast<uint16_t *>(ctx->Am) : nullptr;
  p.KTs = p.scan_tc == 2 ? ctx->KTs : nullptr;
  p.Wsc = p.scan_tc == 2 ? ctx->Wsc : nullptr;
  p.Umax = p.scan_tc == 2 ? ctx->Umax : nullptr;
  p.o = ctx->o;
  p.y_codes = ctx->y_codes;
  p.y_scales = ctx->y_scales;
  p.y_sf_tiled = out_proj_tiled(ctx, T) ? 1 : 0;
  p.status = ctx->status;
  e = launch_prefill_mix(p, ctx->conv_tmp, lc);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(run_out_proj(ctx, out, T, lc, true));
}

gdn_status gdn_in_mix(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, uint8_t *y_codes,
                      uint8_t *y_scales, uint16_t *conv_state, void *ssm_state, int num_slots, void *stream) {
  gdn_status st = check_state_args(ctx, x, y_codes, conv_state, ssm_state, num_slots);
  if (st != GDN_OK) return st;
  if (!slot_ids || !y_scales) return GDN_E_NULL;
  if (!aligned16(slot_ids) || !aligned16(y_scales)) return GDN_E_ALIGN;
  if (B < 1 || B > ctx->cfg.max_batch || !pm_path(ctx, B)) return GDN_E_SHAPE;
  // no programmatic launch: the state must not be read before a preceding
  // kernel that writes it has finished
  LaunchCtx lc{static_cast<cudaStream_t>(stream), ctx->num_sms, false};
  return cuda_status(
      launch_proj_mix(pm_args(ctx, x, slot_ids, B, conv_state, ssm_state, num_slots, y_codes, y_scales), lc));
}

gdn_status gdn_out_proj(gdn_ctx *ctx, const uint8_t *y_codes, const uint8_t *y_scales, int B, uint16_t *out,
                        void *stream) {
  if (!ctx || !y_codes || !y_scales || !out) return GDN_E_NULL;
  if (!aligned16(y_codes) || !aligned16(y_scales) || !aligned16(out)) return GDN_E_ALIGN;
  if (B < 1 || B > 8 || !ctx->w_out_mma || ctx->Vd % 256) return GDN_E_SHAPE;
  LaunchCtx lc{static_cast<cudaStream_t>(stream), ctx->num_sms, false};
  return cuda_status(launch_gemv_mma(out_gemv_args(ctx, y_codes, y_scales, B, out, false), lc));
}

gdn_status gdn_check(gdn_ctx *ctx, int clear, void *stream) {
  if (!ctx) return GDN_E_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t flag = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&flag, ctx->status, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(ctx->status, 0, 4);
  if (e != cudaSuccess) return GDN_E_CUDA;
  return (gdn_status)flag;
}

}  // extern "C"
