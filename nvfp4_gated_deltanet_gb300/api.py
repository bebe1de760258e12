"""Python names of the C entry points (argument marshalling only).

Tensors are PyTorch CUDA tensors, contiguous; BF16 tensors may be passed as
torch.bfloat16 or as int16/uint16 bit patterns. Outputs are allocated with
torch when not given.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import GdnConfig, GdnNVFP4, GdnWeights, _check, _ptr, _stream, lib

__all__ = ["nvfp4_quantize", "nvfp4_gemm", "kda_step", "GatedDeltaNetLayer", "layer_from_synth", "status_name"]


def status_name(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def _dev(t: torch.Tensor) -> torch.Tensor:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t


def nvfp4_quantize(x: torch.Tensor, tensor_scale: float, codes=None, scales=None, dev_status=None, stream=None):
    """x [rows][cols] BF16 (or its bits) or FP32 -> (codes uint8 [rows][cols/2], scales uint8 [rows][cols/16])."""
    _dev(x)
    rows, cols = x.shape
    if codes is None:
        codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(rows, cols // 16, dtype=torch.uint8, device=x.device)
    st = lib().nvfp4_quantize(_ptr(x), int(x.dtype == torch.float32), rows, cols, float(tensor_scale),
                              _ptr(codes), _ptr(scales), _ptr(dev_status), _stream(stream))
    _check(st, "nvfp4_quantize")
    return codes, scales


def _nv(codes, scales, ts) -> GdnNVFP4:
    return GdnNVFP4(_ptr(_dev(codes)), _ptr(_dev(scales)), float(ts))


def nvfp4_gemm(a_codes, a_scales, a_ts, b_codes, b_scales, b_ts, out_dtype=torch.bfloat16, c=None, stream=None):
    """C[M][N] = A_hat[M][K] B_hat[N][K]^T (FP32 accumulation) as BF16 or FP32."""
    M, N, K = a_codes.shape[0], b_codes.shape[0], a_codes.shape[1] * 2
    if c is None:
        c = torch.empty(M, N, dtype=out_dtype, device=a_codes.device)
    A, B = _nv(a_codes, a_scales, a_ts), _nv(b_codes, b_scales, b_ts)
    st = lib().nvfp4_gemm(ctypes.byref(A), M, ctypes.byref(B), N, K, _ptr(c), int(c.dtype != torch.float32),
                          _stream(stream))
    _check(st, "nvfp4_gemm")
    return c


def kda_step(q, k, v, g, beta, state, o=None, stream=None):
    """KDA-style recurrent step in place on `state` [M][H][d][d] (FP32, or BF16
    bits as int16/bfloat16); q, k, g, v [M][H][d] and beta [M][H] FP32.
    Returns o [M][H][d] FP32."""
    M, H, d = q.shape
    for t in (q, k, v, g, beta):
        if t.dtype != torch.float32:
            raise ValueError("q, k, v, g, beta must be float32")
    bf16 = state.dtype in (torch.int16, torch.bfloat16)
    if not bf16 and state.dtype != torch.float32:
        raise ValueError("state must be float32 or BF16 bits")
    if o is None:
        o = torch.empty(M, H, d, dtype=torch.float32, device=q.device)
    st = lib().kda_step(_ptr(_dev(q)), _ptr(_dev(k)), _ptr(_dev(v)), _ptr(_dev(g)), _ptr(_dev(beta)),
                        _ptr(_dev(state)), int(bf16), M, H, d, _ptr(_dev(o)), _stream(stream))
    _check(st, "kda_step")
    return o


class GatedDeltaNetLayer:
    """One GDN layer context (gdn_create / gdn_destroy) and its calls."""

    def __init__(self, hidden, n_k_heads, n_v_heads, d_k, d_v, conv_kernel, weights: dict, max_batch=16,
                 max_prefill_tokens=0, rms_eps=1e-6, l2_eps=1e-6, act_scale_in=2.0 ** -8, act_scale_out=2.0 ** -4,
                 stream=None, state_bf16=False):
        self.cfg = GdnConfig(hidden, n_k_heads, n_v_heads, d_k, d_v, conv_kernel, max_batch, max_prefill_tokens,
                             rms_eps, l2_eps, act_scale_in, act_scale_out, int(bool(state_bf16)))
        self.state_bf16 = bool(state_bf16)
        w = weights
        self._w = GdnWeights(_nv(*w["qkvz"]), _nv(*w["ba"]), _nv(*w["out"]), _ptr(_dev(w["conv_w"])),
                             _ptr(_dev(w["A_log"])), _ptr(_dev(w["dt_bias"])), _ptr(_dev(w["norm_w"])))
        self._ctx = ctypes.c_void_p()
        st = lib().gdn_create(ctypes.byref(self.cfg), ctypes.byref(self._w), _stream(stream), ctypes.byref(self._ctx))
        _check(st, "gdn_create")
        self.H, self.Hk, self.Hv, self.D, self.Kc = hidden, n_k_heads, n_v_heads, d_k, conv_kernel
        self.C = 2 * n_k_heads * d_k + n_v_heads * d_v

    def close(self):
        if self._ctx:
            lib().gdn_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> int:
        return self._ctx.value

    def new_states(self, num_slots: int, device="cuda"):
        """Zeroed conv state BF16 bits [S][K-1][C] and recurrent state [S][Hv][dv][dk]:
        FP32, or BF16 bits (int16) for a layer created with state_bf16."""
        conv = torch.zeros(num_slots, self.Kc - 1, self.C, dtype=torch.int16, device=device)
        ssm = torch.zeros(num_slots, self.Hv, self.D, self.D,
                          dtype=torch.int16 if self.state_bf16 else torch.float32, device=device)
        return conv, ssm

    def _state(self, ssm_state):
        want = (torch.int16, torch.bfloat16) if self.state_bf16 else (torch.float32,)
        if ssm_state.dtype not in want:
            raise ValueError(f"recurrent state must be {want[0]} for this layer, got {ssm_state.dtype}")
        return _dev(ssm_state)

    def decode_step(self, x, slot_ids, conv_state, ssm_state, out=None, stream=None):
        B = x.shape[0]
        if out is None:
            out = torch.empty(B, self.H, dtype=torch.int16, device=x.device)
        st = lib().gdn_decode_step(self._ctx, _ptr(_dev(x)), _ptr(_dev(slot_ids)), B, _ptr(out),
                                   _ptr(_dev(conv_state)), _ptr(self._state(ssm_state)), conv_state.shape[0],
                                   _stream(stream))
        _check(st, "gdn_decode_step")
        return out

    def mix_step(self, qkvz, ba, slot_ids, conv_state, ssm_state, y=None, stream=None):
        B = qkvz.shape[0]
        if y is None:
            y = torch.empty(B, self.Hv * self.D, dtype=torch.float32, device=qkvz.device)
        st = lib().gdn_mix_step(self._ctx, _ptr(_dev(qkvz)), _ptr(_dev(ba)), _ptr(_dev(slot_ids)), B, _ptr(y),
                                _ptr(_dev(conv_state)), _ptr(self._state(ssm_state)), conv_state.shape[0], _stream(stream))
        _check(st, "gdn_mix_step")
        return y

    def in_proj(self, x, slot_ids=None, out=None, stream=None):
        """x [B][H] -> the in-projection rows [B][Nin] BF16 bits (q|k|v|z|b|a)."""
        B = x.shape[0]
        nin = 2 * self.Hk * self.D + 2 * self.Hv * self.D + 2 * self.Hv
        if out is None:
            out = torch.empty(B, nin, dtype=torch.int16, device=x.device)
        st = lib().gdn_in_proj(self._ctx, _ptr(_dev(x)), _ptr(slot_ids), B, _ptr(_dev(out)), _stream(stream))
        _check(st, "gdn_in_proj")
        return out

    def in_mix(self, x, slot_ids, conv_state, ssm_state, y_codes=None, y_scales=None, stream=None):
        """In-projection + mixing of B <= 8 rows as one kernel: x [B][H] -> y as
        NVFP4 (codes uint8 [B][Hv*D/2], row-major scales uint8 [B][Hv*D/16])."""
        B = x.shape[0]
        vd = self.Hv * self.D
        if y_codes is None:
            y_codes = torch.empty(B, vd // 2, dtype=torch.uint8, device=x.device)
        if y_scales is None:
            y_scales = torch.empty(B, vd // 16, dtype=torch.uint8, device=x.device)
        st = lib().gdn_in_mix(self._ctx, _ptr(_dev(x)), _ptr(_dev(slot_ids)), B, _ptr(_dev(y_codes)),
                              _ptr(_dev(y_scales)), _ptr(_dev(conv_state)), _ptr(self._state(ssm_state)),
                              conv_state.shape[0], _stream(stream))
        _check(st, "gdn_in_mix")
        return y_codes, y_scales

    def out_proj(self, y_codes, y_scales, out=None, stream=None):
        """The out-projection of B <= 8 NVFP4 rows -> out [B][H] BF16 bits."""
        B = y_codes.shape[0]
        if out is None:
            out = torch.empty(B, self.H, dtype=torch.int16, device=y_codes.device)
        st = lib().gdn_out_proj(self._ctx, _ptr(_dev(y_codes)), _ptr(_dev(y_scales)), B, _ptr(_dev(out)),
                                _stream(stream))
        _check(st, "gdn_out_proj")
        return out

    def new_snapshots(self, B: int, r: int, device="cuda"):
        """Snapshot buffers of a verify pass: conv [B][r][K-1][C] BF16 bits and
        recurrent [B][r][Hv][dv][dk] in the layer's state type."""
        conv = torch.empty(B, r, self.Kc - 1, self.C, dtype=torch.int16, device=device)
        ssm = torch.empty(B, r, self.Hv, self.D, self.D,
                          dtype=torch.int16 if self.state_bf16 else torch.float32, device=device)
        return conv, ssm

    def verify(self, x, slot_ids, conv_state, ssm_state, snap_conv, snap_ssm, out=None, stream=None):
        """x [B][r][H] candidate tokens -> out [B][r][H]; snapshots of the state
        after every token; the slots' states are not modified."""
        B, r = x.shape[0], x.shape[1]
        if out is None:
            out = torch.empty(B, r, self.H, dtype=torch.int16, device=x.device)
        st = lib().gdn_verify(self._ctx, _ptr(_dev(x)), _ptr(_dev(slot_ids)), B, r, _ptr(out),
                              _ptr(_dev(conv_state)), _ptr(self._state(ssm_state)), conv_state.shape[0],
                              _ptr(_dev(snap_conv)), _ptr(self._state(snap_ssm)), _stream(stream))
        _check(st, "gdn_verify")
        return out

    def verify_commit(self, slot_ids, accepted, snap_conv, snap_ssm, conv_state, ssm_state, stream=None):
        """Slot of row b takes the state after its accepted[b]-th token (device int32 [B]; 0 = keep)."""
        B, r = snap_conv.shape[0], snap_conv.shape[1]
        st = lib().gdn_verify_commit(self._ctx, _ptr(_dev(slot_ids)), B, r, _ptr(_dev(accepted)),
                                     _ptr(_dev(snap_conv)), _ptr(self._state(snap_ssm)), _ptr(_dev(conv_state)),
                                     _ptr(self._state(ssm_state)), conv_state.shape[0], _stream(stream))
        _check(st, "gdn_verify_commit")

    def prefill(self, x, slot, init_zero, conv_state, ssm_state, out=None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.int16, device=x.device)
        st = lib().gdn_prefill(self._ctx, _ptr(_dev(x)), T, int(slot), int(bool(init_zero)), _ptr(out),
                               _ptr(_dev(conv_state)), _ptr(self._state(ssm_state)), conv_state.shape[0], _stream(stream))
        _check(st, "gdn_prefill")
        return out

    def check(self, clear=True, stream=None) -> int:
        """Synchronise and return (and optionally clear) the sticky device status."""
        return int(lib().gdn_check(self._ctx, int(bool(clear)), _stream(stream)))


def _t(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def layer_from_synth(w, max_batch=16, max_prefill_tokens=0, device="cuda", stream=None,
                     state_bf16=False) -> GatedDeltaNetLayer:
    """Upload ``synth.LayerWeights`` and create the layer context."""
    sh = w.shape
    dw = {
        "qkvz": (_t(w.qkvz.codes, device), _t(w.qkvz.scales, device), w.qkvz.tensor_scale),
        "ba": (_t(w.ba.codes, device), _t(w.ba.scales, device), w.ba.tensor_scale),
        "out": (_t(w.out.codes, device), _t(w.out.scales, device), w.out.tensor_scale),
        "conv_w": _t(w.conv_w, device), "A_log": _t(w.A_log, device), "dt_bias": _t(w.dt_bias, device),
        "norm_w": _t(w.norm_w, device),
    }
    layer = GatedDeltaNetLayer(sh.hidden, sh.n_k_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.conv_kernel, dw,
                               max_batch=max_batch, max_prefill_tokens=max_prefill_tokens, rms_eps=w.rms_eps,
                               l2_eps=w.l2_eps, act_scale_in=w.act_scale_in, act_scale_out=w.act_scale_out,
                               stream=stream, state_bf16=state_bf16)
    torch.cuda.synchronize()
    return layer
