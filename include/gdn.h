/*
 * gdn.h -- C ABI of one NVFP4 W4A4 Gated DeltaNet (GDN) layer step on one GPU.
 *
 * The operation (Rocket blog, "A reduction barrier makes Qwen GDN graph replay
 * bit exact", setup table; "the Rocket GDN entry" below): one GDN
 * linear-attention layer as it is served from
 * an NVFP4 checkpoint -- W4A4 QKVZ/BA projections, a BF16 causal convolution,
 * an FP32 recurrent state updated by the gated delta rule (state laid out
 * [v][k], the "pretranspose" decode layout), a z-gated RMSNorm and a W4A4
 * output projection. NVFP4 (bloomery issue #565, §4, #489/#687): packed
 * E2M1 pairs, one E4M3 scale per 16 values, one FP32 scale per tensor; W4A4
 * quantises the activations to NVFP4 as well.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument that names a tensor is a DEVICE pointer, 16-byte
 *   aligned, to row-major storage. The caller owns it; no call frees it.
 * - BF16 tensors are passed as uint16_t bit patterns, E2M1 codes as bytes
 *   holding two codes (element 2i in the low nibble of byte i), E4M3 scales as
 *   one byte per 16 elements of a row.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call
 *   except gdn_create and gdn_check is asynchronous on it, allocates nothing,
 *   never synchronises and never reads device memory on the host, so it may be
 *   captured into a CUDA graph.
 * - Host-detectable errors (NULL pointers, sizes, alignment, non-finite scales)
 *   return a status before anything is launched. Errors only the device can see
 *   (non-finite activations, slot ids out of range or repeated) are written to a
 *   sticky device status word and read back by gdn_check. Device code never
 *   traps.
 * - Numerics: every reduction has a fixed order and no atomics are used, so
 *   repeated calls on the same inputs give bit-identical results.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_E_NULL = 1,       /* a required pointer is NULL */
  GDN_E_SHAPE = 2,      /* a size is outside what the call or the context supports */
  GDN_E_ALIGN = 3,      /* a tensor pointer is not 16-byte aligned */
  GDN_E_NONFINITE = 4,  /* a scale, epsilon or activation is NaN or infinite */
  GDN_E_BAD_SCALE = 5,  /* a scale is <= 0, or an E4M3 weight scale byte is NaN */
  GDN_E_RANGE = 6,      /* a slot id is out of range or repeated within one call */
  GDN_E_OVERFLOW = 7,   /* a size product overflows the index types */
  GDN_E_CUDA = 8,       /* a CUDA runtime call failed */
  GDN_E_OOM = 9,        /* gdn_create could not allocate its device memory */
  GDN_E_TIMEOUT = 10,   /* a bounded device wait gave up */
  GDN_E_STATE = 11      /* the context is unusable (creation failed part way) */
} gdn_status;

/* Short, static, human-readable name of a status ("GDN_E_SHAPE", ...). */
const char *gdn_status_string(int status);

/* Layer shape and the static quantiser settings of one layer. */
typedef struct {
  int hidden;             /* H: model width, multiple of 64 */
  int n_k_heads;          /* Hk: key/query heads */
  int n_v_heads;          /* Hv: value heads, a multiple of Hk; value head h reads key head h / (Hv/Hk) */
  int d_k, d_v;           /* head sizes; d_k == d_v in {32, 64, 128} */
  int conv_kernel;        /* depthwise causal conv taps; 4 */
  int max_batch;          /* largest B gdn_decode_step accepts (1..256) */
  int max_prefill_tokens; /* largest T gdn_prefill accepts (0 = no prefill) */
  float rms_eps;          /* gated RMSNorm epsilon (inside the square root) */
  float l2_eps;           /* q/k L2-norm epsilon (inside the square root) */
  float act_scale_in;     /* FP32 tensor scale of the x quantiser, > 0 */
  float act_scale_out;    /* FP32 tensor scale of the gated-norm output quantiser, > 0 */
  int state_bf16;         /* recurrent state storage: 0 = FP32; 1 = BF16 (same layout, 2-byte
                             elements). The arithmetic stays FP32: a decode step loads the
                             BF16 state, updates it in FP32 and stores it rounded to nearest
                             even; a prefill call carries it in FP32 from its first token to
                             its last and rounds once at the end. Halves the dominant
                             per-sequence bytes (Rocket blog, "KDA state tile": BF16 state
                             storage measured beside FP32). */
} gdn_config;

/* One NVFP4 matrix W[rows][cols]: codes [rows][cols/2], scales [rows][cols/16]
 * (device pointers), value = e2m1(code) * e4m3(scale) * tensor_scale. */
typedef struct {
  const uint8_t *codes;
  const uint8_t *scales;
  float tensor_scale;
} gdn_nvfp4;

/* Layer weights (device pointers). Read once by gdn_create; the caller may
 * free them after it returns.
 *   qkvz: [2*Hk*d_k + 2*Hv*d_v][H], rows ordered q | k | v | z, heads contiguous
 *   ba:   [2*Hv][H], rows ordered b | a
 *   out:  [H][Hv*d_v]
 *   conv_w: BF16 [C][conv_kernel], C = 2*Hk*d_k + Hv*d_v channels ordered q | k | v,
 *           taps oldest to newest
 *   A_log, dt_bias: FP32 [Hv];  norm_w: FP32 [d_v] */
typedef struct {
  gdn_nvfp4 qkvz, ba, out;
  const uint16_t *conv_w;
  const float *A_log, *dt_bias, *norm_w;
} gdn_weights;

typedef struct gdn_ctx gdn_ctx;

/* Validate the config and weights, copy the weights into the kernels' layouts
 * and allocate the context's workspace on the current device. The pages define
 * no such call (an interface choice of this library): it holds what the Rocket
 * GDN entry's setup table fixes for a served layer -- the W4A4 NVFP4 QKVZ/BA
 * and output projection weights, the BF16 causal-convolution taps and the
 * gate parameters -- in the layouts the kernels stream. Synchronises
 * `stream` once (the only call that does besides gdn_check). On failure *out is
 * NULL and nothing stays allocated. Errors: GDN_E_NULL, GDN_E_SHAPE,
 * GDN_E_NONFINITE (eps/scales), GDN_E_BAD_SCALE (scale <= 0 or an E4M3 weight
 * scale byte 0x7F/0xFF), GDN_E_OVERFLOW, GDN_E_OOM, GDN_E_CUDA. */
gdn_status gdn_create(const gdn_config *cfg, const gdn_weights *w, void *stream, gdn_ctx **out);

/* Free everything the context owns. NULL is accepted. Synchronises the device
 * work of the context's own allocations (cudaFree). No counterpart on the
 * pages: an interface choice of this library, the inverse of gdn_create. */
gdn_status gdn_destroy(gdn_ctx *ctx);

/* NVFP4 quantisation of x[rows][cols] (bloomery issue #565, §4, #687:
 * "4-bit activations"). x is BF16 bits (x_is_f32 = 0) or FP32 (x_is_f32 = 1);
 * cols % 16 == 0. For every 16-block, in FP32 with round-to-nearest-even:
 *   inv6ts = 1 / (6 * tensor_scale); amax = max |x|; s = E4M3_satfinite(amax * inv6ts);
 *   if e4m3(s) == 0 the 16 codes are 0, else r = 1 / (e4m3(s) * tensor_scale) and
 *   code = E2M1_satfinite(x * r), sign kept (-0 is code 8).
 * Writes codes [rows][cols/2] and scales [rows][cols/16]. A block holding NaN or
 * infinity gets scale 0 and codes 0 and sets GDN_E_NONFINITE in *dev_status
 * (a device int32, may be NULL). Errors: GDN_E_NULL, GDN_E_SHAPE (rows < 0,
 * cols % 16), GDN_E_ALIGN, GDN_E_NONFINITE / GDN_E_BAD_SCALE (tensor_scale). */
gdn_status nvfp4_quantize(const void *x, int x_is_f32, int rows, int cols, float tensor_scale,
                          uint8_t *codes, uint8_t *scales, int32_t *dev_status, void *stream);

/* Block-scaled W4A4 product C[M][N] = sum_k A_hat[m][k] * B_hat[n][k], FP32
 * accumulation, written as BF16 (c_is_bf16 = 1, round to nearest even) or FP32
 * (bloomery issue #565, §4, #687: W4A4 means both the 4-bit weights and the
 * activations enter the product as NVFP4; the Rocket GDN entry's setup table
 * runs the QKVZ/BA and output projections of the layer this way).
 * A is [M][K], B is [N][K], both NVFP4 (struct fields are device pointers,
 * the struct itself is host memory). K % 64 == 0, M, N >= 0 (0 is a no-op).
 * Errors: GDN_E_NULL, GDN_E_SHAPE, GDN_E_ALIGN, GDN_E_BAD_SCALE (tensor
 * scale <= 0 or non-finite), GDN_E_OVERFLOW. */
gdn_status nvfp4_gemm(const gdn_nvfp4 *A, int M, const gdn_nvfp4 *B, int N, int K,
                      void *C, int c_is_bf16, void *stream);

/* One decode step of B sequences (c1..c16 buckets and larger batches): the
 * layer step of the Rocket GDN entry (setup table and decode table: W4A4 QKVZ/BA projections, a
 * BF16 causal convolution, the FP32 recurrent state in the pretranspose [v][k]
 * layout, the output projection; buckets c1, c2, c4, c8, c16).
 *   x:          BF16 [B][H]
 *   slot_ids:   int32 [B] (device), the state slot of each row; -1 marks a padding
 *               row, whose output row is written as zeros and which touches no state.
 *               Ids must be distinct; an id >= num_slots or < -1, or a repeated id,
 *               sets GDN_E_RANGE in the status word and that row is treated as padding.
 *   out:        BF16 [B][H]
 *   conv_state: BF16 [num_slots][conv_kernel-1][C], the last conv_kernel-1 raw
 *               inputs of every channel, oldest first; updated in place
 *   ssm_state:  FP32 [num_slots][Hv][d_v][d_k], or BF16 bits of the same shape when
 *               the config's state_bf16 is set; updated in place
 * Per active row: x -> NVFP4(act_scale_in) -> W4A4 qkvz/ba -> BF16; conv + SiLU;
 * q,k L2-normalised (q also scaled by d_k^-1/2); beta = sigmoid(b),
 * g = -exp(A_log) * softplus(a + dt_bias); per value head S <- exp(g) S,
 * u = beta (v - S k), S <- S + u k^T, o = S q; y = o * rsqrt(mean(o^2) + rms_eps)
 * * norm_w * SiLU(z); y -> NVFP4(act_scale_out) -> W4A4 out_proj -> BF16.
 * Errors: GDN_E_NULL, GDN_E_SHAPE (B < 1 or > max_batch, num_slots < 1),
 * GDN_E_ALIGN, GDN_E_OVERFLOW, GDN_E_CUDA. */
gdn_status gdn_decode_step(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B,
                           uint16_t *out, uint16_t *conv_state, void *ssm_state, int num_slots,
                           void *stream);

/* The in-projection stage of gdn_decode_step (B <= max_batch) or gdn_prefill
 * (B tokens) alone, for stage-wise checks and timing: x BF16 [B][H] -> proj
 * BF16 [B][2*Hk*d_k + 2*Hv*d_v + 2*Hv], each row q | k | v | z | b | a; rows
 * whose slot_ids entry is negative are zero (slot_ids: device int32 [B], or
 * NULL for none). Same kernels and results as inside those calls for the same
 * row count. Errors: GDN_E_NULL, GDN_E_ALIGN, GDN_E_SHAPE (B < 1 or more than
 * max(max_batch, max_prefill_tokens)), GDN_E_CUDA. */
gdn_status gdn_in_proj(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, uint16_t *proj,
                       void *stream);

/* The token-mixing stage of gdn_decode_step alone, for stage-wise checks and
 * for callers that run the projections themselves: takes the BF16 projection
 * outputs qkvz [B][2*Hk*d_k + 2*Hv*d_v] and ba [B][2*Hv] and writes the FP32
 * gated-norm output y [B][Hv*d_v] (zeros for padding rows); conv_state and
 * ssm_state as in gdn_decode_step, updated in place. Same errors. */
gdn_status gdn_mix_step(gdn_ctx *ctx, const uint16_t *qkvz, const uint16_t *ba,
                        const int32_t *slot_ids, int B, float *y, uint16_t *conv_state,
                        void *ssm_state, int num_slots, void *stream);

/* The in-projection and token-mixing stages of gdn_decode_step as the one
 * kernel that step runs for up to 8 rows (tuning knob 13), for stage-wise
 * checks and timing: x BF16 [B][H] -> y, the gated-norm output as NVFP4 with
 * tensor scale act_scale_out: codes [B][Hv*d_v/2] and row-major scales
 * [B][Hv*d_v/16] (zeros for padding rows); conv_state and ssm_state as in
 * gdn_decode_step, updated in place. Not launched early: it starts after the
 * preceding work in the stream has finished. Errors: as gdn_decode_step,
 * GDN_E_SHAPE when B > 8 or the shape is outside what the kernel covers
 * (d_k = 128, Hv / Hk of 1 or 2, H a multiple of 256 up to 2048). */
gdn_status gdn_in_mix(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, uint8_t *y_codes,
                      uint8_t *y_scales, uint16_t *conv_state, void *ssm_state, int num_slots, void *stream);

/* The out-projection stage alone on the warp-MMA kernel gdn_decode_step runs
 * for up to 8 rows: y NVFP4 (codes [B][Hv*d_v/2], row-major scales
 * [B][Hv*d_v/16], tensor scale act_scale_out) -> out BF16 [B][H]. Errors:
 * GDN_E_NULL, GDN_E_ALIGN, GDN_E_SHAPE (B outside 1..8, or Hv*d_v not a
 * multiple of 256), GDN_E_CUDA. */
gdn_status gdn_out_proj(gdn_ctx *ctx, const uint8_t *y_codes, const uint8_t *y_scales, int B, uint16_t *out,
                        void *stream);

/* Prefill of T tokens of one sequence held in slot `slot` (host int): the same
 * arithmetic as T successive decode steps of that sequence (bloomery issue #565,
 * §4, #812: the delta rule of a prompt runs on tensor cores in chunks).
 * x BF16 [T][H] -> out BF16 [T][H]; init_zero != 0 starts from zero conv and
 * recurrent state (the slot's state is overwritten), else from the slot's
 * state. The slot's state is left as after the last token. Errors: GDN_E_NULL,
 * GDN_E_SHAPE (T < 1 or > max_prefill_tokens), GDN_E_RANGE (slot), GDN_E_ALIGN. */
gdn_status gdn_prefill(gdn_ctx *ctx, const uint16_t *x, int T, int slot, int init_zero,
                       uint16_t *out, uint16_t *conv_state, void *ssm_state, int num_slots,
                       void *stream);

/* Multi-token verify (speculative decoding's check of r candidate tokens per
 * sequence) and its commit, the pair of passes the pages run beside prompt and
 * decode on a GDN layer's delta state (bloomery issue #565, §10, PR #1127).
 *
 * gdn_verify runs r tokens of each of B sequences through the layer, token by
 * token, exactly as r successive gdn_decode_step calls would, but leaves the
 * slots' states untouched: the state after each token goes to the caller's
 * snapshot buffers instead.
 *   x:         BF16 [B][r][H], row b's candidate tokens in order
 *   slot_ids:  int32 [B] (device), as for gdn_decode_step (-1 = padding: zero
 *              output rows, no snapshot written; its x rows must be finite)
 *   out:       BF16 [B][r][H]
 *   conv_state, ssm_state: the slots' states as for gdn_decode_step (read only)
 *   snap_conv: BF16 [B][r][conv_kernel-1][C]; snap_ssm: [B][r][Hv][d_v][d_k] in
 *              the state's storage type (FP32, or BF16 bits with state_bf16):
 *              snapshot (b, t) is row b's state after its token t.
 * B * r must not exceed max_batch. Errors: as gdn_decode_step, GDN_E_SHAPE for
 * r < 1 or B * r > max_batch.
 *
 * gdn_verify_commit then makes row b's slot take snapshot (b, n-1), where
 * n = accepted[b] (device int32 [B], read by the kernel so the commit can be
 * captured in a graph after the acceptance decision): n = 0 keeps the slot's
 * state, n in 1..r commits the state after the n-th token, n > r sets
 * GDN_E_RANGE in the status word and leaves that slot untouched. Padding rows
 * are skipped. Slot ids must be distinct. Errors: GDN_E_NULL, GDN_E_ALIGN,
 * GDN_E_SHAPE, GDN_E_CUDA. */
gdn_status gdn_verify(gdn_ctx *ctx, const uint16_t *x, const int32_t *slot_ids, int B, int r, uint16_t *out,
                      const uint16_t *conv_state, const void *ssm_state, int num_slots, uint16_t *snap_conv,
                      void *snap_ssm, void *stream);
gdn_status gdn_verify_commit(gdn_ctx *ctx, const int32_t *slot_ids, int B, int r, const int32_t *accepted,
                             const uint16_t *snap_conv, const void *snap_ssm, uint16_t *conv_state,
                             void *ssm_state, int num_slots, void *stream);

/* KDA-style recurrent step: the gated delta rule with one decay per key
 * channel, for M streams x H heads of size d (Rocket blog, "Moving the KDA
 * state tile out of shared memory is 4.6x at M=8": a 64 x 128 x 128 state per
 * stream read and written every step). Per (stream, head), with S [d][d] laid
 * out [d_v][d_k]:
 *   S <- S diag(exp(g));  u = beta (v - S k);  S <- S + u k^T;  o = S q
 * q, k, g (per-channel log-decay), v, o: FP32 [M][H][d]; beta: FP32 [M][H];
 * state: [M][H][d][d], FP32, or BF16 bits when state_bf16 = 1 (loaded to FP32,
 * stored rounded to nearest even), updated in place. All device pointers,
 * 16-byte aligned. No normalisation of q or k inside the step. Asynchronous on
 * `stream`, allocates nothing. Errors: GDN_E_NULL, GDN_E_SHAPE (M, H < 1,
 * d not 32/64/128, state_bf16 not 0/1), GDN_E_ALIGN, GDN_E_OVERFLOW, GDN_E_CUDA. */
gdn_status kda_step(const float *q, const float *k, const float *v, const float *g, const float *beta,
                    void *state, int state_bf16, int M, int H, int d, float *o, void *stream);

/* The decode step of gdn_decode_step for callers that cannot allocate device
 * memory or keep a context: runtimes that fix all device memory at start-up,
 * work issued while a CUDA graph is captured, hosts that pass only tensors.
 * (It has no counterpart on the pages the library follows: it is an interface
 * choice of this library.) The caller passes the config and the weights
 * exactly as for gdn_create (device pointers, read on every call), and x,
 * slot_ids, out, conv_state, ssm_state as for gdn_decode_step. The call
 * allocates nothing: its intermediates live in one fixed device array of
 * 450,560 bytes inside the library, which bounds the shape: B <= 16,
 * hidden <= 2048, 2*Hk*d_k + 2*Hv*d_v + 2*Hv <= 12352, Hv*d_v <= 4096
 * (else GDN_E_SHAPE). The first call on a device looks up that array's
 * address (make it before any stream capture). All calls on a device share the
 * array: calls that overlap on the GPU race, so serialise them. Weight scale
 * bytes are not scanned for NaN (gdn_create does that). Device-detected errors
 * go to *dev_status (device int32, may be NULL) as in nvfp4_quantize.
 * Errors: as gdn_create's checks and gdn_decode_step's, plus GDN_E_CUDA. */
gdn_status gdn_decode_step_static(const gdn_config *cfg, const gdn_weights *w, const uint16_t *x,
                                  const int32_t *slot_ids, int B, uint16_t *out, uint16_t *conv_state,
                                  void *ssm_state, int num_slots, int32_t *dev_status, void *stream);

/* Process-wide tuning knobs (they change speed, never results beyond FP32
 * summation order). knob 0: projection kernel of decode and prefill:
 * 0 = automatic (more than 4 activation rows and a reduction length that is a
 * multiple of 256: tcgen05 block-scaled MMA; else the CUDA-core kernels, the
 * warp-MMA one for up to 8 rows),
 * 1 = CUDA-core kernel (also for nvfp4_gemm with M <= 16), 2 = tensor cores
 * where the reduction length allows. knob 1 / knob 2: split-K of the in- /
 * out-projection on tensor cores, 0 = automatic, or 1, 2, 4, 8 (reduced to
 * the largest power of two that divides the 256-wide K tiles). knob 3: decode
 * of one or two rows as one persistent cooperative kernel (weights and state
 * prefetched into shared memory, grid barriers between the stages): 0 and 1 =
 * never (the default: it measured slower than the three-kernel step on
 * GB300), 2 = when the shape allows (d_k = 128, B <= 2, knob 0 is not 2).
 * knob 4: a decode in-projection on tensor cores with at most 16 rows
 * quantises x inside the GEMM (0 and 2 = yes, the default; 1 = a separate
 * quantisation kernel first). knob 5: the out-projection of gdn_decode_step
 * lets the next kernel in the stream launch before it waits on the mixing
 * kernel (0 = on the tensor-core out-projection only, the default; 1 = never;
 * 2 = also on the CUDA-core one); every kernel of this library that may follow
 * it reads only weights until its own dependency wait.
 * knob 6: tensor-core projections of a context stream the weight codes from a
 * pre-swizzled copy made at gdn_create, one contiguous 16 KB bulk copy per
 * 128 x 256 tile (0 and 2 = yes, the default; 1 = tensor-map copies from the
 * row-major codes). knob 7: d_v slices per head in the decode mixing kernel
 * (0 = chosen from the batch and the value-head count, the default: 4 while
 * Hv * B <= 16, else 2 up to 4 rows, else 1; or 1, 2 or 4, reduced while the
 * cluster of a key head would exceed 8 CTAs). knob 8: one-row projections
 * of a context on the CUDA cores take the block dot products with warp-level
 * MMA (mma.sync, FP16 in, FP32 out; weights repacked at create) instead of
 * FP16x2 chains (0 and 2 = yes, the default; 1 = no). knob 9: the decode
 * token mixing as three kernels -- conv/norms/gates, the delta rule alone,
 * gated norm + quantisation -- with bit-identical results (0 and 1 = never,
 * the default: the one mixing kernel, whose state streams through registers
 * when its grid exceeds two CTAs per SM, measured faster at every batch size;
 * 2 = always). knob 10: the prefill chunk stages' products -- K K^T and
 * Q K^T per chunk, then the scan's W S^T, Q S^T, A U and state update -- in
 * split precision: 0 = automatic (tcgen05 MMAs with TMEM accumulators for
 * d = 128, else FP32 on the CUDA cores), 1 = the scan in FP32 on the CUDA
 * cores, 2 = warp-level MMA in split TF32 (d = 128), 3 = tcgen05 (d = 128:
 * K K^T, Q K^T and the scan's products in split FP16 with power-of-two
 * block scales); the forms agree to FP32 rounding. knob 11: tensor-core projections with
 * 128-token activation tiles, tiled scales and BF16 output as one persistent
 * CTA per SM with two TMEM accumulators, so that the epilogue of one output
 * tile overlaps the MMAs of the next. Two forms: streaming (both operands
 * through one shared-memory ring that runs across tiles) and, for a reduction
 * length of 2048, weight-stationary (a CTA keeps a 128-row weight tile and its
 * scales resident and streams only activation tiles; measured slower than
 * streaming on GB300). 0 = automatic, the default: streaming from two output
 * tiles per SM, else one tile per CTA; 1 = one tile per CTA; 2 = streaming
 * whenever the form allows; 3 = weight-stationary whenever the form allows
 * (else as 2). knob 12: the budget, in SM cycles, of each grid-barrier wait of
 * the persistent single-kernel step (knob 3): 0 = the default, 2^31 (about
 * one second); any positive value sets it. A wait that runs out records
 * GDN_E_TIMEOUT in the status word and the kernel finishes without it (that
 * step's results are then meaningless); the barrier words are cleared before
 * every launch, so the next call starts clean. A short budget exists to test
 * that path: these waits guard no copy in flight.
 * knob 13: decode of up to 8 rows (d_k = 128, Hv / Hk of 1 or 2, H <= 2048)
 * as two kernels: the in-projection rows of each key head computed inside the
 * cluster that mixes that head (conv, norms, gates, delta rule, gated norm,
 * quantisation), then the warp-MMA out-projection, which lets the next kernel
 * start at once (0 and 1 = off, the default: measured slower on GB300, only
 * 15 of its 16 eight-CTA clusters fit at once; 2 = on where the shape allows
 * and knob 0 is not 2). Bit-identical to the three-kernel step on the warp-MMA
 * projections with four K slices (knob 0 = 1, knob 14 = 1).
 * knob 14 / knob 15: tile of the warp-MMA in- / out-projection: 0 = automatic
 * (in: one row 1, 2..4 rows 3; out: 2 when Hv*d_v >= 4096, else 1), 1 = two
 * 16-row groups per CTA x four K slices, 2 = one group x eight K slices
 * (reduction length a multiple of 512, else as 1), 3 = four groups x two K
 * slices. knob 16: the warp-MMA kernels bring their activation rows into
 * shared memory with one bulk copy per CTA (0 = automatic: for two or more
 * rows, or one row in a launch of at least 256 CTAs; 1 = never, per-thread
 * loads; 2 = always).
 * Returns GDN_E_RANGE for an unknown knob or value. Not thread-safe; set it
 * before launching work. */
gdn_status gdn_set_tuning(int knob, int value);

/* Synchronise `stream`, read the context's sticky device status word, clear it
 * if `clear`, and return it (GDN_OK when nothing was flagged). A CUDA error seen
 * while synchronising returns GDN_E_CUDA. */
gdn_status gdn_check(gdn_ctx *ctx, int clear, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
