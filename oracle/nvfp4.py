"""NVFP4 quantisation and the block-scaled W4A4 product.

Format (bloomery issue #565, §4, #489 and #687; Rocket blog, "FP8 and
NVFP4 serving maps": ModelOpt block-16 packing): a value is
    x_hat = e2m1(code) * e4m3(block scale) * tensor_scale,
one unsigned E4M3 scale per 16 consecutive elements of a row, one FP32 scale
per tensor.

The pages do not print the quantiser's arithmetic. This oracle takes the
plainest reading that makes every block's largest magnitude land on the top
E2M1 value 6, and fixes the order of operations so that "bit-exact" has one
meaning. All decisions are taken in IEEE binary32 (numpy float32 arithmetic is
correctly rounded), the precision the kernel decides in:

  1. inv6ts = 1 / (6 * ts)                  two FP32 roundings, computed once
  2. amax   = max |x| over the 16-block     exact
  3. t      = amax * inv6ts                 FP32
  4. s      = E4M3(t)                       RNE, satfinite (448)
  5. if e4m3(s) == 0: the block's 16 codes are 0
  6. else d = e4m3(s) * ts (FP32), r = 1 / d (FP32), code = E2M1(x * r)
     (x * r in FP32, E2M1 RNE, satfinite at 6, sign kept).
"""
from __future__ import annotations

import numpy as np

from . import codecs


def quantize(x: np.ndarray, tensor_scale: float):
    """x: float32 [rows][cols] (cols % 16 == 0), finite. Returns (codes uint8
    [rows][cols/2] packed, scales uint8 [rows][cols/16])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % 16:
        raise ValueError("quantize: need [rows][cols] with cols % 16 == 0")
    if not np.isfinite(x).all():
        raise ValueError("quantize: non-finite input")
    ts = np.float32(tensor_scale)
    if not (np.isfinite(ts) and ts > 0):
        raise ValueError("quantize: tensor scale must be finite and > 0")
    rows, cols = x.shape
    blocks = x.reshape(rows, cols // 16, 16)
    inv6ts = np.float32(1.0) / (np.float32(6.0) * ts)
    amax = np.abs(blocks).max(axis=2)                                  # float32, exact
    t = (amax * inv6ts).astype(np.float32)
    s = codecs.e4m3_encode(t)
    sval = codecs.e4m3_decode(s).astype(np.float32)                    # exact in float32
    d = (sval * ts).astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(sval > 0, np.float32(1.0) / np.where(d > 0, d, np.float32(1.0)), np.float32(0.0))
    r = r.astype(np.float32)
    scaled = (blocks * r[:, :, None]).astype(np.float32)
    codes = codecs.e2m1_encode(scaled)
    codes = np.where((sval > 0)[:, :, None], codes, 0).astype(np.uint8)
    return codecs.pack_nibbles(codes.reshape(rows, cols)), s


def dequantize(codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    """Packed codes [rows][cols/2], scales [rows][cols/16] -> float64 [rows][cols]."""
    c = codecs.e2m1_decode(codecs.unpack_nibbles(codes))
    rows, cols = c.shape
    s = codecs.e4m3_decode(scales).repeat(16, axis=1)
    return c * s * float(np.float32(tensor_scale))


class Operand:
    """Integer forms of an NVFP4 matrix for the exact product: 2*e2m1 (exact
    integers in -12..12) as float64 [nb][rows][16], and e4m3 * 2^9 (exact
    integers up to 229376) as int64 [nb][rows]."""

    def __init__(self, codes: np.ndarray, scales: np.ndarray, tensor_scale: float):
        c2 = 2.0 * codecs.e2m1_decode(codecs.unpack_nibbles(codes))
        rows, cols = c2.shape
        self.rows, self.nb = rows, cols // 16
        self.c2 = np.ascontiguousarray(c2.reshape(rows, self.nb, 16).transpose(1, 0, 2))
        self.s512 = np.ascontiguousarray(np.rint(codecs.e4m3_decode(scales) * 512.0).astype(np.int64).T)
        self.ts = float(np.float32(tensor_scale))


def gemm_op(a: Operand, b: Operand) -> np.ndarray:
    """C[m][n] = sum_k a_hat[m,k] * b_hat[n,k], exact, then rounded once to FP32.

    Each 16-block contributes (sum of 4*e2m1*e2m1, an integer of at most 2304
    in magnitude) * (512*sa) * (512*sb), an integer of at most 2^47; with at
    most 2^8 blocks (K <= 4096) the int64 sum is exact. The result is that
    integer times 2^-20 * ts_a * ts_b: converted in float64 (relative error
    2^-53, far below the FP32 rounding that follows) and rounded to FP32.
    """
    if a.nb != b.nb:
        raise ValueError("gemm: K mismatch")
    if a.nb > 256:
        raise ValueError("gemm: K > 4096 would leave the exact int64 range")
    acc = np.zeros((a.rows, b.rows), dtype=np.int64)
    for blk in range(a.nb):
        q = np.rint(a.c2[blk] @ b.c2[blk].T).astype(np.int64)          # 4*sum e2m1*e2m1, exact
        acc += q * (a.s512[blk][:, None] * b.s512[blk][None, :])
    scale = 2.0 ** -20 * a.ts * b.ts
    return (acc.astype(np.float64) * scale).astype(np.float32)


def gemm(a_codes, a_scales, a_ts, b_codes, b_scales, b_ts) -> np.ndarray:
    """gemm_op on raw packed operands."""
    return gemm_op(Operand(a_codes, a_scales, a_ts), Operand(b_codes, b_scales, b_ts))
