"""Seeded synthetic inputs for the NVFP4 Gated DeltaNet layer step.

This module draws random numbers and stores them in the layer's storage
types. It holds none of the layer's arithmetic: no quantisation, no GEMM, no
convolution or recurrence. Rounding a drawn float to a storage type (BF16,
E4M3) is done by PyTorch's own dtype conversion (round-to-nearest-even), a
library primitive, so the CPU oracle and the CUDA path receive byte-identical
inputs without sharing any codec.

Distributions (the workload recipe of the layer's published configurations):

* NVFP4 weights: every E2M1 nibble uniform over the 16 codes (so -0 appears);
  E4M3 block scales uniform in [2^-4, 2^2] in linear value, then rounded to
  E4M3; FP32 tensor scale 2^-6.
* x: BF16 of N(0, 1).
* A_log ~ U(0, ln 16), dt_bias ~ U(-1, 1), FP32.
* depthwise conv taps ~ U(-0.5, 0.5) in BF16 (the usual 1/sqrt(fan_in) bound
  with fan_in = 4); gated-norm weight ~ U(0.5, 1.5) FP32.
* conv state BF16 of N(0, 1); recurrent state FP32 N(0, 0.1^2) (std 0.1).

Each tensor has its own stream: numpy PCG64 seeded by SeedSequence([seed,
stream id]). numpy's PCG64 and its ziggurat normal sampler give the same
numbers on x86_64 and aarch64.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

# Stream ids: one per drawn tensor, fixed forever so stored fixtures stay valid.
_STREAM = {
    "qkvz.codes": 1, "qkvz.scales": 2,
    "ba.codes": 3, "ba.scales": 4,
    "out.codes": 5, "out.scales": 6,
    "conv_w": 7, "A_log": 8, "dt_bias": 9, "norm_w": 10,
    "x": 11, "conv_state": 12, "ssm_state": 13,
    "mat.codes": 14, "mat.scales": 15, "mat.values": 16,
    "kda": 17,
}

WEIGHT_TENSOR_SCALE = 2.0 ** -6
ACT_SCALE_IN = 2.0 ** -8   # static tensor scale of the x quantiser
ACT_SCALE_OUT = 2.0 ** -4  # static tensor scale of the gated-norm output quantiser
RMS_EPS = 1e-6
L2_EPS = 1e-6


@dataclasses.dataclass(frozen=True)
class LayerShape:
    hidden: int
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    conv_kernel: int = 4

    @property
    def qkvz_out(self) -> int:
        return 2 * self.n_k_heads * self.d_k + 2 * self.n_v_heads * self.d_v

    @property
    def ba_out(self) -> int:
        return 2 * self.n_v_heads

    @property
    def conv_channels(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    @property
    def value_dim(self) -> int:
        return self.n_v_heads * self.d_v


TINY = LayerShape(hidden=256, n_k_heads=2, n_v_heads=4, d_k=32, d_v=32)
FULL = LayerShape(hidden=2048, n_k_heads=16, n_v_heads=32, d_k=128, d_v=128)
# One rank's slice of the full layer under two-way head-parallel serving
# (half the key and value heads; hidden unchanged, out_proj keeps half its
# input columns): the shape the pages' GB10 decode table was measured on.
TP2 = LayerShape(hidden=2048, n_k_heads=8, n_v_heads=16, d_k=128, d_v=128)


def rng(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), _STREAM[name]])))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 BF16 bit patterns (PyTorch RNE conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    """float32 array (finite, < 464) -> uint8 E4M3 bit patterns (PyTorch RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


@dataclasses.dataclass
class NVFP4Matrix:
    """Row-major NVFP4 matrix [rows][cols]: packed E2M1 codes (element 2i in the
    low nibble of byte i), one E4M3 scale byte per 16 elements, FP32 tensor scale."""
    codes: np.ndarray   # uint8 [rows][cols/2]
    scales: np.ndarray  # uint8 [rows][cols/16]
    tensor_scale: float

    @property
    def shape(self):
        return self.codes.shape[0], self.codes.shape[1] * 2


def nvfp4_random(rows: int, cols: int, seed: int, prefix: str = "mat",
                 tensor_scale: float = WEIGHT_TENSOR_SCALE) -> NVFP4Matrix:
    assert cols % 16 == 0
    codes = rng(seed, prefix + ".codes").integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    u = rng(seed, prefix + ".scales").uniform(2.0 ** -4, 2.0 ** 2, size=(rows, cols // 16))
    return NVFP4Matrix(codes, to_e4m3_bits(u.astype(np.float32)), float(tensor_scale))


@dataclasses.dataclass
class LayerWeights:
    shape: LayerShape
    qkvz: NVFP4Matrix
    ba: NVFP4Matrix
    out: NVFP4Matrix
    conv_w: np.ndarray   # uint16 BF16 [C][K_conv]
    A_log: np.ndarray    # float32 [Hv]
    dt_bias: np.ndarray  # float32 [Hv]
    norm_w: np.ndarray   # float32 [d_v]
    act_scale_in: float = ACT_SCALE_IN
    act_scale_out: float = ACT_SCALE_OUT
    rms_eps: float = RMS_EPS
    l2_eps: float = L2_EPS


def layer_weights(shape: LayerShape, seed: int) -> LayerWeights:
    H = shape.hidden
    qkvz = nvfp4_random(shape.qkvz_out, H, seed, "qkvz")
    ba = nvfp4_random(shape.ba_out, H, seed, "ba")
    out = nvfp4_random(H, shape.value_dim, seed, "out")
    C = shape.conv_channels
    conv_w = to_bf16_bits(rng(seed, "conv_w").uniform(-0.5, 0.5, size=(C, shape.conv_kernel)).astype(np.float32))
    A_log = rng(seed, "A_log").uniform(0.0, math.log(16.0), size=shape.n_v_heads).astype(np.float32)
    dt_bias = rng(seed, "dt_bias").uniform(-1.0, 1.0, size=shape.n_v_heads).astype(np.float32)
    norm_w = rng(seed, "norm_w").uniform(0.5, 1.5, size=shape.d_v).astype(np.float32)
    return LayerWeights(shape, qkvz, ba, out, conv_w, A_log, dt_bias, norm_w)


def x_tokens(shape: LayerShape, seed: int, steps: int) -> np.ndarray:
    """BF16 bits [steps][hidden] for one sequence."""
    return to_bf16_bits(rng(seed, "x").standard_normal(size=(steps, shape.hidden)).astype(np.float32))


def conv_state(shape: LayerShape, seed: int, zero: bool = False) -> np.ndarray:
    """BF16 bits [K_conv-1][C] (oldest tap first) for one sequence."""
    n = (shape.conv_kernel - 1, shape.conv_channels)
    if zero:
        return np.zeros(n, dtype=np.uint16)
    return to_bf16_bits(rng(seed, "conv_state").standard_normal(size=n).astype(np.float32))


def ssm_state(shape: LayerShape, seed: int, zero: bool = False) -> np.ndarray:
    """FP32 [Hv][d_v][d_k] for one sequence."""
    n = (shape.n_v_heads, shape.d_v, shape.d_k)
    if zero:
        return np.zeros(n, dtype=np.float32)
    return (0.1 * rng(seed, "ssm_state").standard_normal(size=n)).astype(np.float32)


def bf16_normal(rows: int, cols: int, seed: int, std: float = 1.0) -> np.ndarray:
    """BF16 bits of N(0, std^2), for quantiser and GEMM cases."""
    return to_bf16_bits((std * rng(seed, "mat.values").standard_normal(size=(rows, cols))).astype(np.float32))


def slot_seed(slot: int) -> int:
    """Per-sequence seed of the multi-sequence decode workloads."""
    return 100 + int(slot)


def kda_inputs(M: int, H: int, D: int, seed: int):
    """Inputs of a KDA-style recurrent step for M streams x H heads, head size D:
    q, k ~ N(0, 1/D) (norm about 1), v ~ N(0, 1), per-channel log-decay
    g = -0.5 U(0, 1), beta ~ U(0, 1), all FP32; state N(0, 0.1^2) FP32
    [M][H][D][D]."""
    r = rng(seed, "kda")
    s = 1.0 / np.sqrt(D)
    q = (s * r.standard_normal(size=(M, H, D))).astype(np.float32)
    k = (s * r.standard_normal(size=(M, H, D))).astype(np.float32)
    v = r.standard_normal(size=(M, H, D)).astype(np.float32)
    g = (-0.5 * r.uniform(0.0, 1.0, size=(M, H, D))).astype(np.float32)
    beta = r.uniform(0.0, 1.0, size=(M, H)).astype(np.float32)
    S = (0.1 * r.standard_normal(size=(M, H, D, D))).astype(np.float32)
    return q, k, v, g, beta, S
