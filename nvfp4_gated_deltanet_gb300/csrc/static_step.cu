// gdn_decode_step_static: the decode step without a context and without any
// device allocation.
//
// Who needs it: callers that may not allocate device memory once they are
// running -- serving runtimes that plan every byte of device memory at start-up
// and forbid cudaMalloc afterwards, code that issues work while a CUDA graph is
// being captured (allocation is not allowed there), and plug-in style hosts
// that hand over tensors but cannot keep a gdn_ctx alive between calls. The
// caller passes the weights (as for gdn_create), the inputs and the outputs;
// the intermediates of the step (NVFP4 copy of x, the projections, the NVFP4
// gated-norm output) live in one file-scope device array of fixed size, below.
//
// Set-up: the first call on a device looks up that array's device address with
// cudaGetSymbolAddress (with the device current) and caches it per device.
// Make that first call before any stream capture.
//
// Sharing: every call on a device uses the same array. Calls whose kernels
// overlap on the GPU (two streams, or two host threads) race on it; serialise
// them. Nothing in the array needs to start at zero: every byte a call reads
// was written earlier in the same call.
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace gdn {
namespace {

// Limits of the static scratch (bytes in brackets):
constexpr int kMaxRows = 16;          // decode rows per call (c1..c16)
constexpr int kMaxHidden = 2048;      // H
constexpr int kMaxProj = 12352;       // 2*Hk*dk + 2*Hv*dv + 2*Hv (the q|k|v|z|b|a row)
constexpr int kMaxValue = 4096;       // Hv*dv
constexpr size_t kProjBytes = (size_t)kMaxRows * kMaxProj * 2;          // [395,264]
constexpr size_t kXqCodeBytes = (size_t)kMaxRows * kMaxHidden / 2;      // [16,384]
constexpr size_t kXqScaleBytes = (size_t)kMaxRows * kMaxHidden / 16;    // [2,048]
constexpr size_t kYCodeBytes = (size_t)kMaxRows * kMaxValue / 2;        // [32,768]
constexpr size_t kYScaleBytes = (size_t)kMaxRows * kMaxValue / 16;      // [4,096]
constexpr size_t kOffXqCode = kProjBytes;
constexpr size_t kOffXqScale = kOffXqCode + kXqCodeBytes;
constexpr size_t kOffYCode = kOffXqScale + kXqScaleBytes;
constexpr size_t kOffYScale = kOffYCode + kYCodeBytes;
constexpr size_t kScratchBytes = kOffYScale + kYScaleBytes;              // 450,560 bytes
static_assert(kOffXqCode % 256 == 0 && kOffXqScale % 256 == 0 && kOffYCode % 256 == 0 && kOffYScale % 256 == 0,
              "every scratch region starts 256-byte aligned");

// The scratch itself. In host code this name is only a stand-in for the
// device array: kernels get the address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_step_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char *g_scratch_ptr[kMaxDevices] = {};

// The device address of the scratch on the current device (set up once).
cudaError_t scratch_for_current_device(unsigned char **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_step_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status to_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_E_CUDA; }

// One projection of `rows` activation rows (NVFP4 codes/scales in the scratch,
// or BF16 x quantised on the fly) onto the n rows of weight matrix w, written
// to the first n columns of c, a [rows][ldc] BF16 output.
cudaError_t project(const gdn_nvfp4 &w, int n, int K, int rows, const uint16_t *x_bf16, const int32_t *row_slot,
                    int num_slots, const uint8_t *a_codes, const uint8_t *a_scales, float ts_a, uint16_t *c, int ldc,
                    bool tensor_cores, int32_t *status, const LaunchCtx &lc) {
  if (tensor_cores) {
    TcGemm t{};
    if (!tc_make_weight_maps(t, w.codes, w.scales, n, K)) return cudaErrorInvalidValue;
    t.b_codes = a_codes;
    t.b_scales = a_scales;
    t.args.Ma = n;
    t.args.Nb = rows;
    t.args.K = K;
    t.args.c = c;
    t.args.ldc = ldc;
    t.args.c_is_bf16 = 1;
    t.args.ts_a0 = t.args.ts_a1 = w.tensor_scale;
    t.args.a_split = n;
    t.args.ts_b = ts_a;
    t.args.a_const = 0;
    t.args.status = status;
    return launch_tc_gemm(t, lc);
  }
  GemvArgs g{};
  g.a_bf16 = x_bf16;
  g.a_codes = x_bf16 ? nullptr : a_codes;
  g.a_scales = x_bf16 ? nullptr : a_scales;
  g.ts_a = ts_a;
  g.row_slot = row_slot;
  g.num_slots = num_slots;
  g.w_codes = w.codes;
  g.w_scales = w.scales;
  g.ts_w0 = g.ts_w1 = w.tensor_scale;
  g.n_split = n;
  g.c = c;
  g.c_is_bf16 = 1;
  g.ldc = ldc;
  g.M = rows;
  g.N = n;
  g.K = K;
  g.status = status;
  return launch_gemv(g, lc);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_decode_step_static(const gdn_config *cfg, const gdn_weights *w, const uint16_t *x,
                                             const int32_t *slot_ids, int B, uint16_t *out, uint16_t *conv_state,
                                             void *ssm_state, int num_slots, int32_t *dev_status, void *stream) {
  if (!cfg || !w || !x || !slot_ids || !out || !conv_state || !ssm_state) return GDN_E_NULL;
  const gdn_config &c = *cfg;
  if (c.n_k_heads <= 0 || c.n_v_heads <= 0 || c.n_v_heads % c.n_k_heads || c.n_v_heads / c.n_k_heads > 8 ||
      c.d_k != c.d_v || (c.d_k != 32 && c.d_k != 64 && c.d_k != 128) || c.conv_kernel < 2 || c.conv_kernel > 4 ||
      c.hidden <= 0 || c.hidden % 64 || (c.n_v_heads * c.d_v) % 64 || (c.state_bf16 != 0 && c.state_bf16 != 1))
    return GDN_E_SHAPE;
  const int H = c.hidden, Hk = c.n_k_heads, Hv = c.n_v_heads, D = c.d_k;
  const int Nqkvz = 2 * Hk * D + 2 * Hv * D, Nba = 2 * Hv, Nin = Nqkvz + Nba, Vd = Hv * D;
  // the fixed scratch bounds the shape
  if (B < 1 || B > kMaxRows || H > kMaxHidden || Nin > kMaxProj || Vd > kMaxValue || num_slots < 1)
    return GDN_E_SHAPE;
  if (!std::isfinite(c.rms_eps) || !std::isfinite(c.l2_eps) || !std::isfinite(c.act_scale_in) ||
      !std::isfinite(c.act_scale_out))
    return GDN_E_NONFINITE;
  if (c.rms_eps < 0 || c.l2_eps < 0 || !(c.act_scale_in > 0) || !(c.act_scale_out > 0)) return GDN_E_BAD_SCALE;
  const gdn_nvfp4 *mats[3] = {&w->qkvz, &w->ba, &w->out};
  for (const gdn_nvfp4 *m : mats) {
    if (!m->codes || !m->scales) return GDN_E_NULL;
    if (!aligned16(m->codes) || !aligned16(m->scales)) return GDN_E_ALIGN;
    if (!std::isfinite(m->tensor_scale)) return GDN_E_NONFINITE;
    if (!(m->tensor_scale > 0)) return GDN_E_BAD_SCALE;
  }
  if (!w->conv_w || !w->A_log || !w->dt_bias || !w->norm_w) return GDN_E_NULL;
  if (!aligned16(x) || !aligned16(slot_ids) || !aligned16(out) || !aligned16(conv_state) || !aligned16(ssm_state) ||
      !aligned16(w->conv_w) || !aligned16(w->A_log) || !aligned16(w->dt_bias) || !aligned16(w->norm_w))
    return GDN_E_ALIGN;

  unsigned char *scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) return GDN_E_CUDA;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return GDN_E_CUDA;
  const LaunchCtx lc{static_cast<cudaStream_t>(stream), sms, false};
  uint16_t *proj = reinterpret_cast<uint16_t *>(scratch);
  uint8_t *xq_codes = scratch + kOffXqCode, *xq_scales = scratch + kOffXqScale;
  uint8_t *y_codes = scratch + kOffYCode, *y_scales = scratch + kOffYScale;

  // x -> q|k|v|z and b|a (one row: CUDA cores; more: tensor cores, as in decode)
  const bool tc_in = B > 1 && H % 256 == 0;
  if (tc_in) {
    e = launch_quantize(x, 0, B, H, c.act_scale_in, xq_codes, xq_scales, dev_status, lc.stream, slot_ids, num_slots,
                        false);
    if (e != cudaSuccess) return GDN_E_CUDA;
  }
  e = project(w->qkvz, Nqkvz, H, B, tc_in ? nullptr : x, slot_ids, num_slots, xq_codes, xq_scales, c.act_scale_in,
              proj, Nin, tc_in, dev_status, lc);
  if (e == cudaSuccess)
    e = project(w->ba, Nba, H, B, tc_in ? nullptr : x, slot_ids, num_slots, xq_codes, xq_scales, c.act_scale_in,
                proj + Nqkvz, Nin, tc_in, dev_status, lc);
  if (e != cudaSuccess) return to_status(e);

  MixArgs m{};
  m.qkvz = proj;
  m.ld_qkvz = Nin;
  m.ba = proj + Nqkvz;
  m.ld_ba = Nin;
  m.slot_ids = slot_ids;
  m.B = B;
  m.num_slots = num_slots;
  m.conv_state = conv_state;
  m.ssm_state = ssm_state;
  m.state_bf16 = c.state_bf16;
  m.conv_w = w->conv_w;
  m.A_log = w->A_log;
  m.dt_bias = w->dt_bias;
  m.norm_w = w->norm_w;
  m.Hk = Hk;
  m.Hv = Hv;
  m.D = D;
  m.C = 2 * Hk * D + Hv * D;
  m.Kc = c.conv_kernel;
  m.l2_eps = c.l2_eps;
  m.rms_eps = c.rms_eps;
  m.ts_out = c.act_scale_out;
  m.y_codes = y_codes;
  m.y_scales = y_scales;
  m.y_f32 = nullptr;
  m.status = dev_status;
  e = launch_mix(m, lc);
  if (e != cudaSuccess) return GDN_E_CUDA;

  const bool tc_out = B > 1 && Vd % 256 == 0;
  return to_status(project(w->out, H, Vd, B, nullptr, nullptr, 0, y_codes, y_scales, c.act_scale_out, out, H, tc_out,
                           dev_status, lc));
}
