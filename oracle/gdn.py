"""Gated DeltaNet layer step, written out stage by stage in float64.

The pages name the serving path of one GDN layer (Rocket blog, "A reduction
barrier makes Qwen GDN graph replay bit exact", setup table): W4A4 QKVZ/BA and
output projections, a BF16 causal convolution, an FP32 recurrent state whose
update follows vLLM's fused_recurrent gated delta rule, with the decode state
laid out [v][k] as in FlashInfer's pretranspose decode. They do not print the
equations. The readings taken here:

* projections: x -> NVFP4 (static tensor scale s_in) -> W4A4 GEMM -> FP32 ->
  BF16 (bloomery issue #565, #1039: the q, k, v projections are stored in
  BF16). Output order [q | k | v | z] and [b | a], heads contiguous.
* convolution: depthwise over the [q | k | v] channels, kernel K, no bias,
  taps oldest to newest; the state keeps the last K-1 raw BF16 inputs of each
  channel, oldest first; output SiLU(pre).
* q and k are L2-normalised per key head: k_hat = k / sqrt(sum k^2 + eps),
  q_hat = q / sqrt(sum q^2 + eps) * d_k^-1/2.
* gates: beta = sigmoid(b); g = -exp(A_log) * softplus(a + dt_bias) with
  softplus(x) = x for x > 20; alpha = exp(g).
* value head h reads key head h // (Hv / Hk).
* delta rule on S[d_v][d_k]: S <- alpha S; u = beta (v - S k_hat);
  S <- S + u k_hat^T; o = S q_hat. The state is stored in FP32 after each step,
  or, for a layer whose state is kept in BF16 (Rocket blog, "KDA state tile":
  the state stored in BF16 beside FP32), rounded FP32 -> BF16 (nearest even)
  after each decode step; a prefill call then carries the state in FP32 from
  its first token to its last and rounds once at the end.
* gated RMSNorm per value head: y = o * (mean(o^2) + eps)^-1/2 * w * SiLU(z).
* y -> FP32 -> NVFP4 (static s_out) -> W4A4 out_proj -> FP32 -> BF16.
* a padding row (slot id -1) writes a zero output row and touches no state.
"""
from __future__ import annotations

import math

import numpy as np

from . import codecs, nvfp4


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sigmoid(x)


def softplus(x):
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 20.0, x, np.log1p(np.exp(np.minimum(x, 20.0))))


# ------------------------------------------------------------------ stages

def project(x_bf16_bits: np.ndarray, w_op, act_scale: float) -> np.ndarray:
    """BF16 rows -> NVFP4 -> W4A4 GEMM with the NVFP4 weight operand w_op
    (``nvfp4.Operand``) -> FP32 -> BF16 values (float64)."""
    xf = codecs.bf16_to_f32(x_bf16_bits)
    xc, xs = nvfp4.quantize(xf, act_scale)
    y32 = nvfp4.gemm_op(nvfp4.Operand(xc, xs, act_scale), w_op)
    return codecs.round_bf16(y32)


def conv_step(win_state: np.ndarray, x_new: np.ndarray, conv_w: np.ndarray):
    """One causal depthwise-conv step for every channel.

    win_state: float64 [K-1][C] (oldest first), x_new: float64 [C],
    conv_w: float64 [C][K]. Returns (SiLU(pre) [C], new state [K-1][C])."""
    window = np.concatenate([win_state, x_new[None, :]], axis=0)        # [K][C], oldest first
    pre = np.zeros(x_new.shape, dtype=np.float64)
    for j in range(window.shape[0]):
        pre += conv_w[:, j] * window[j]
    return silu(pre), window[1:].copy()


def l2norm(x: np.ndarray, eps: float) -> np.ndarray:
    """Normalise the last axis: x / sqrt(sum x^2 + eps)."""
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + eps)


def gates(b: np.ndarray, a: np.ndarray, A_log: np.ndarray, dt_bias: np.ndarray):
    """beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias)."""
    beta = sigmoid(np.asarray(b, dtype=np.float64))
    g = -np.exp(np.asarray(A_log, dtype=np.float64)) * softplus(np.asarray(a, dtype=np.float64)
                                                                + np.asarray(dt_bias, dtype=np.float64))
    return beta, g


def delta_step(S: np.ndarray, q_hat: np.ndarray, k_hat: np.ndarray, v: np.ndarray,
               beta: np.ndarray, g: np.ndarray):
    """One gated delta-rule step for every value head.

    S: float64 [Hv][dv][dk]; q_hat, k_hat: [Hk][dk]; v: [Hv][dv]; beta, g: [Hv].
    Returns (o [Hv][dv], new S [Hv][dv][dk]) in float64 (not rounded)."""
    Hv = S.shape[0]
    Hk = k_hat.shape[0]
    group = Hv // Hk
    S_new = np.empty_like(S)
    o = np.empty(v.shape, dtype=np.float64)
    for h in range(Hv):
        kh = k_hat[h // group]
        qh = q_hat[h // group]
        Sh = math.exp(g[h]) * S[h]
        u = beta[h] * (v[h] - Sh @ kh)
        Sh = Sh + np.outer(u, kh)
        S_new[h] = Sh
        o[h] = Sh @ qh
    return o, S_new


def gated_rmsnorm(o: np.ndarray, z: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """o, z: [Hv][dv]; w: [dv]. y = o * (mean(o^2) + eps)^-1/2 * w * SiLU(z)."""
    r = 1.0 / np.sqrt((o * o).mean(axis=-1, keepdims=True) + eps)
    return o * r * w[None, :] * silu(z)


# ------------------------------------------------------------------ layer

class Layer:
    """One GDN layer: weights from ``synth.LayerWeights``."""

    def __init__(self, weights, state_bf16: bool = False):
        self.w = weights
        self.state_bf16 = bool(state_bf16)
        sh = weights.shape
        self.sh = sh
        self.conv_w = codecs.bf16_to_f32(weights.conv_w).astype(np.float64)
        self.A_log = weights.A_log.astype(np.float64)
        self.dt_bias = weights.dt_bias.astype(np.float64)
        self.norm_w = weights.norm_w.astype(np.float64)
        self.op_qkvz = nvfp4.Operand(weights.qkvz.codes, weights.qkvz.scales, weights.qkvz.tensor_scale)
        self.op_ba = nvfp4.Operand(weights.ba.codes, weights.ba.scales, weights.ba.tensor_scale)
        self.op_out = nvfp4.Operand(weights.out.codes, weights.out.scales, weights.out.tensor_scale)

    # -- the parts of one token's step, exposed for stage-wise comparisons
    def projections(self, x_bits: np.ndarray):
        """x BF16 bits [B][H] -> (qkvz [B][Nqkvz], ba [B][2Hv]) BF16 values."""
        return (project(x_bits, self.op_qkvz, self.w.act_scale_in),
                project(x_bits, self.op_ba, self.w.act_scale_in))

    def mix(self, qkvz_row: np.ndarray, ba_row: np.ndarray, conv_st: np.ndarray, S: np.ndarray,
            state_store: str | None = None):
        """Conv, norms, gates, delta rule and gated norm for one sequence.

        qkvz_row, ba_row: BF16 values (float64); conv_st: BF16 bits [K-1][C];
        S: [Hv][dv][dk] float32 values. Returns (y float64 [Hv*dv], conv_st',
        S', extras) where extras holds the intermediates and S' is the updated
        state rounded to its storage type: "f32", or "bf16" (FP32 then BF16,
        held in float32); by default the layer's own."""
        sh = self.sh
        nq = sh.n_k_heads * sh.d_k
        nv = sh.n_v_heads * sh.d_v
        qkv_in = qkvz_row[: 2 * nq + nv]
        z = qkvz_row[2 * nq + nv:].reshape(sh.n_v_heads, sh.d_v)
        b = ba_row[: sh.n_v_heads]
        a = ba_row[sh.n_v_heads:]
        win = codecs.bf16_to_f32(conv_st).astype(np.float64)
        conv_out, win_new = conv_step(win, qkv_in, self.conv_w)
        q = conv_out[:nq].reshape(sh.n_k_heads, sh.d_k)
        k = conv_out[nq:2 * nq].reshape(sh.n_k_heads, sh.d_k)
        v = conv_out[2 * nq:].reshape(sh.n_v_heads, sh.d_v)
        k_hat = l2norm(k, self.w.l2_eps)
        q_hat = l2norm(q, self.w.l2_eps) / math.sqrt(sh.d_k)
        beta, g = gates(b, a, self.A_log, self.dt_bias)
        o, S64 = delta_step(S.astype(np.float64), q_hat, k_hat, v, beta, g)
        y = gated_rmsnorm(o, z, self.norm_w, self.w.rms_eps)
        new_conv = codecs.f32_to_bf16(win_new.astype(np.float32))       # raw BF16 inputs: exact
        extras = dict(conv_out=conv_out, q_hat=q_hat, k_hat=k_hat, v=v, beta=beta, g=g, o=o)
        store = state_store or ("bf16" if self.state_bf16 else "f32")
        S_new = S64.astype(np.float32)
        if store == "bf16":
            S_new = codecs.bf16_to_f32(codecs.f32_to_bf16(S_new))
        return y.reshape(-1), new_conv, S_new, extras

    def out_proj(self, y: np.ndarray) -> np.ndarray:
        """y float64 [B][Hv*dv] -> FP32 -> NVFP4 (s_out) -> GEMM -> BF16 bits [B][H]."""
        y32 = np.asarray(y, dtype=np.float64).astype(np.float32)
        yc, ys = nvfp4.quantize(y32, self.w.act_scale_out)
        o32 = nvfp4.gemm_op(nvfp4.Operand(yc, ys, self.w.act_scale_out), self.op_out)
        return codecs.f32_to_bf16(o32)

    # -- whole steps
    def decode_step(self, x_bits: np.ndarray, slot_ids, conv_state: np.ndarray, ssm_state: np.ndarray):
        """One decode step for B rows.

        x_bits: BF16 [B][H]; slot_ids: [B] ints, -1 = padding row;
        conv_state: BF16 bits [S][K-1][C] and ssm_state: FP32 [S][Hv][dv][dk],
        both updated in place. Returns out BF16 bits [B][H]."""
        x_bits = np.asarray(x_bits, dtype=np.uint16).reshape(len(slot_ids), self.sh.hidden)
        qkvz, ba = self.projections(x_bits)
        B = len(slot_ids)
        y = np.zeros((B, self.sh.value_dim), dtype=np.float64)
        for r, slot in enumerate(slot_ids):
            if slot < 0:
                continue
            y[r], conv_state[slot], ssm_state[slot], _ = self.mix(qkvz[r], ba[r], conv_state[slot],
                                                                  ssm_state[slot])
        out = self.out_proj(y)
        for r, slot in enumerate(slot_ids):
            if slot < 0:
                out[r] = 0
        return out

    def verify(self, x_bits: np.ndarray, slot_ids, conv_state: np.ndarray, ssm_state: np.ndarray):
        """Speculative verify of r candidate tokens per row: x_bits BF16 [B][r][H].
        Each live row runs its tokens in order from its slot's state, as r
        decode steps would; the slots are not modified. Returns (out BF16 bits
        [B][r][H], snapshots) where snapshots[b][t] = (conv, ssm) after token t
        (None for padding rows)."""
        x_bits = np.asarray(x_bits, dtype=np.uint16)
        B, r = x_bits.shape[0], x_bits.shape[1]
        qkvz, ba = self.projections(x_bits.reshape(B * r, self.sh.hidden))
        y = np.zeros((B * r, self.sh.value_dim), dtype=np.float64)
        snaps = []
        for b, slot in enumerate(slot_ids):
            if slot < 0:
                snaps.append(None)
                continue
            c, s = conv_state[slot].copy(), ssm_state[slot].copy()
            row = []
            for t in range(r):
                y[b * r + t], c, s, _ = self.mix(qkvz[b * r + t], ba[b * r + t], c, s)
                row.append((c.copy(), s.copy()))
            snaps.append(row)
        out = self.out_proj(y).reshape(B, r, self.sh.hidden)
        for b, slot in enumerate(slot_ids):
            if slot < 0:
                out[b] = 0
        return out, snaps

    @staticmethod
    def verify_commit(slot_ids, accepted, snaps, conv_state: np.ndarray, ssm_state: np.ndarray):
        """Slot of live row b takes its state after token accepted[b] (0 = unchanged)."""
        for b, slot in enumerate(slot_ids):
            n = int(accepted[b])
            if slot < 0 or n <= 0:
                continue
            conv_state[slot], ssm_state[slot] = snaps[b][n - 1]

    def prefill(self, x_bits: np.ndarray, conv_state: np.ndarray, ssm_state: np.ndarray,
                init_zero: bool):
        """Token-by-token prefill of one sequence: x_bits BF16 [T][H]; conv_state
        [K-1][C] and ssm_state [Hv][dv][dk] of that sequence, updated in place.
        Returns out BF16 bits [T][H]."""
        if init_zero:
            conv_state[...] = 0
            ssm_state[...] = 0
        qkvz, ba = self.projections(np.asarray(x_bits, dtype=np.uint16))
        T = qkvz.shape[0]
        y = np.empty((T, self.sh.value_dim), dtype=np.float64)
        for t in range(T):   # the state in FP32 within the call
            y[t], conv_state[...], ssm_state[...], _ = self.mix(qkvz[t], ba[t], conv_state, ssm_state, "f32")
        if self.state_bf16:  # stored once, at the end of the call
            ssm_state[...] = codecs.bf16_to_f32(codecs.f32_to_bf16(ssm_state.astype(np.float32)))
        return self.out_proj(y)


# ------------------------------------------------------------------ chunked form

def chunked_delta(q_hat, k_hat, v, beta, g, S0, chunk: int = 64):
    """The delta rule of ``delta_step`` over T tokens of one value head, in the
    chunked (WY / UT) form, float64. A self-test of the algebra a chunked GPU
    kernel uses, not a second definition.

    q_hat, k_hat: [T][dk]; v: [T][dv]; beta, g: [T]; S0: [dv][dk].
    Within a chunk with start state S0 and rows i = 1..C:
      Gamma_i = sum_{j<=i} g_j,  D_ij = exp(Gamma_i - Gamma_j) for j <= i,
      L_ij = beta_i D_ij (k_i . k_j) for j < i,
      (I + L) U = diag(beta) V - diag(beta exp(Gamma)) K S0^T,
      O_i = exp(Gamma_i) S0 q_i + sum_{j<=i} D_ij (q_i . k_j) u_j,
      S_C = exp(Gamma_C) S0 + sum_j D_Cj u_j k_j^T.
    Returns (O [T][dv], S_T [dv][dk])."""
    T = q_hat.shape[0]
    S = np.array(S0, dtype=np.float64)
    O = np.empty((T, v.shape[1]), dtype=np.float64)
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        Q, K, V, bt, gg = q_hat[sl], k_hat[sl], v[sl], beta[sl], g[sl]
        C = Q.shape[0]
        Gam = np.cumsum(gg)
        D = np.exp(np.tril(Gam[:, None] - Gam[None, :]))
        D = np.tril(D)
        KK = K @ K.T
        L = np.tril(bt[:, None] * D * KK, -1)
        rhs = bt[:, None] * V - (bt * np.exp(Gam))[:, None] * (K @ S.T)
        U = np.linalg.solve(np.eye(C) + L, rhs)
        QK = Q @ K.T
        O[sl] = np.exp(Gam)[:, None] * (Q @ S.T) + (D * QK) @ U
        S = np.exp(Gam[-1]) * S + (D[-1][:, None] * U).T @ K
    return O, S
