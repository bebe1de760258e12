"""Pins of the oracle's NVFP4 quantiser and W4A4 product: a hand-worked golden
fixture, closed forms and exact rational brute force."""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codecs, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_blocks():
    out = []
    with open(os.path.join(GOLDEN, "nvfp4_blocks.txt")) as f:
        for ln in f:
            if not ln.strip() or ln.startswith("#"):
                continue
            vals, scale, codes = ln.split("|")
            x = np.array([float(v) for v in vals.split()], dtype=np.float32)
            out.append((x, int(scale, 16), [int(c, 16) for c in codes.split()]))
    return out


def test_quantize_hand_worked_blocks():
    blocks = _golden_blocks()
    assert len(blocks) == 5
    x = np.stack([b[0] for b in blocks])          # one block per row
    codes, scales = nvfp4.quantize(x, 2.0 ** -8)
    for i, (_, s, c) in enumerate(blocks):
        assert scales[i, 0] == s, i
        assert codes[i].tolist() == c, i


def test_quantize_inv6ts_is_two_fp32_roundings():
    # 6 * 2^-8 is exact, 1/0.0234375 rounds to 0x422AAAAB
    assert np.float32(1.0) / (np.float32(6.0) * np.float32(2.0 ** -8)) == np.uint32(0x422AAAAB).view(np.float32)


@pytest.mark.parametrize("k", [-6, -2, 0, 3, 6])
def test_quantize_power_of_two_amax_hits_code7(k):
    # amax = 6 * ts * 2^k -> scale exactly 2^k and the amax element -> code 7
    ts = 2.0 ** -6
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, 5] = 6 * ts * 2.0 ** k
    x[0, 9] = -6 * ts * 2.0 ** k
    codes, scales = nvfp4.quantize(x, ts)
    assert codecs.e4m3_decode(scales)[0, 0] == 2.0 ** k
    c = codecs.unpack_nibbles(codes)[0]
    assert c[5] == 7 and c[9] == 15 and (np.delete(c, [5, 9]) == 0).all()


def test_quantize_refuses_nan_and_bad_scale():
    with pytest.raises(ValueError):
        nvfp4.quantize(np.full((1, 16), np.nan, np.float32), 1.0)
    with pytest.raises(ValueError):
        nvfp4.quantize(np.ones((1, 16), np.float32), 0.0)
    with pytest.raises(ValueError):
        nvfp4.quantize(np.ones((1, 15), np.float32), 1.0)


def test_quantize_error_bound():
    # |x - x_hat| <= half an E2M1 step at |x*r| times d, when nothing saturates
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    ts = 2.0 ** -8
    codes, scales = nvfp4.quantize(x, ts)
    xh = nvfp4.dequantize(codes, scales, ts)
    d = (codecs.e4m3_decode(scales) * np.float32(ts)).repeat(16, axis=1)
    a = np.abs(x) / d
    half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    assert (np.abs(x - xh) <= half_step * d * (1 + 1e-6)).all()


def _frac_value(code, scale_byte, ts):
    return Fraction(float(codecs.e2m1_decode(code))) * Fraction(float(codecs.e4m3_decode(scale_byte))) \
        * Fraction(float(np.float32(ts)))


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (3, 4, 32), (2, 5, 64)])
def test_gemm_exact_rational_brute_force(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a_codes = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b_codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    a_sc = rng.integers(0, 127, (M, K // 16), dtype=np.uint8)      # any finite E4M3 incl. subnormals
    b_sc = rng.integers(0, 127, (N, K // 16), dtype=np.uint8)
    ta, tb = 2.0 ** -7, 0.3
    got = nvfp4.gemm(a_codes, a_sc, ta, b_codes, b_sc, tb)
    ac, bc = codecs.unpack_nibbles(a_codes), codecs.unpack_nibbles(b_codes)
    for m in range(M):
        for n in range(N):
            exact = sum(_frac_value(ac[m, k], a_sc[m, k // 16], ta) * _frac_value(bc[n, k], b_sc[n, k // 16], tb)
                        for k in range(K))
            g = Fraction(float(got[m, n]))
            ulp = Fraction(float(np.spacing(np.float32(abs(float(exact))) if exact != 0 else np.float32(0))))
            assert abs(g - exact) <= ulp / 2 + Fraction(1, 10 ** 40), (m, n)


def test_gemm_one_hot_selects_one_weight():
    rng = np.random.default_rng(2)
    N, K = 6, 64
    b_codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    b_sc = rng.integers(8, 120, (N, K // 16), dtype=np.uint8)
    tb = 2.0 ** -6
    for k in [0, 17, 63]:
        a = np.zeros((1, K), dtype=np.uint8)
        a[0, k] = 2                                   # E2M1 code 2 = 1.0
        a_codes = codecs.pack_nibbles(a)
        a_sc = np.zeros((1, K // 16), dtype=np.uint8)
        a_sc[0, k // 16] = 0x38                       # E4M3 1.0
        got = nvfp4.gemm(a_codes, a_sc, 1.0, b_codes, b_sc, tb)
        want = nvfp4.dequantize(b_codes, b_sc, tb)[:, k]
        np.testing.assert_array_equal(got[0], want.astype(np.float32))


def test_gemm_zero_block_contributes_nothing():
    rng = np.random.default_rng(4)
    a_codes = rng.integers(0, 256, (2, 16), dtype=np.uint8)
    a_sc = rng.integers(8, 100, (2, 2), dtype=np.uint8)
    b_codes = rng.integers(0, 256, (3, 16), dtype=np.uint8)
    b_sc = rng.integers(8, 100, (3, 2), dtype=np.uint8)
    a_sc0 = a_sc.copy()
    a_sc0[:, 1] = 0
    full = nvfp4.gemm(a_codes, a_sc0, 1.0, b_codes, b_sc, 1.0)
    first = nvfp4.gemm(a_codes[:, :8], a_sc0[:, :1], 1.0, b_codes[:, :8], b_sc[:, :1], 1.0)
    np.testing.assert_array_equal(full, first)
