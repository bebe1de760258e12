"""Pins of the oracle's number formats against things other than itself:
the published code tables, brute-force nearest search, PyTorch's own float8 /
bfloat16 conversions (library routines), and the FNV-1a published vectors."""
import os

import numpy as np
import pytest
import torch

from oracle import codecs, fnv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_table_is_the_published_one():
    # E2M1 magnitudes of codes 0..7 as the OCP MX spec lists them.
    assert codecs.E2M1_GRID.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_round_trip_all_16_codes():
    codes = np.arange(16, dtype=np.uint8)
    vals = codecs.e2m1_decode(codes)
    back = codecs.e2m1_encode(vals)
    assert back.tolist() == codes.tolist()          # includes -0 -> code 8
    assert np.signbit(vals[8]) and vals[8] == 0.0


def _brute_nearest(mags, grid):
    """Nearest grid index by exhaustive distance, ties to the even index, clamp at top."""
    d = np.abs(mags[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    idx = np.where(cand.sum(axis=1) > 1,
                   np.argmax(cand & (np.arange(len(grid)) % 2 == 0)[None, :], axis=1),
                   np.argmax(cand, axis=1))
    return np.where(mags >= grid[-1], len(grid) - 1, idx)


def _midpoint_probes(grid):
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    pts = np.concatenate([grid.astype(np.float32), mids,
                          np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    return pts


def test_e2m1_encode_matches_brute_force():
    rng = np.random.default_rng(5)
    v = np.concatenate([_midpoint_probes(codecs.E2M1_GRID),
                        rng.uniform(0, 8, 200000).astype(np.float32),
                        np.float32([6.0, 6.5, 7.0, 1e30, 1e-30, 0.0])])
    got = codecs.e2m1_encode(v).astype(np.int64)
    want = _brute_nearest(v.astype(np.float64), codecs.E2M1_GRID)
    np.testing.assert_array_equal(got, want)
    neg = codecs.e2m1_encode(-v).astype(np.int64)
    np.testing.assert_array_equal(neg, want + 8)    # sign kept, incl. -0 -> 8


def test_e4m3_table_matches_torch():
    codes = np.arange(127, dtype=np.uint8)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(codecs.E4M3_GRID, t.astype(np.float64))
    assert codecs.E4M3_GRID[-1] == 448.0 and codecs.E4M3_GRID[1] == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(7)
    # every float32 with its low 13 bits zero below 464, plus the exact midpoints
    # of adjacent E4M3 values and their float32 neighbours, plus random values
    top = np.float32(464.0).view(np.uint32)
    lattice = (np.arange(0, int(top) >> 13, dtype=np.uint32) << 13).view(np.float32)
    v = np.concatenate([lattice, _midpoint_probes(codecs.E4M3_GRID),
                        rng.uniform(0, 463.9, 300000).astype(np.float32),
                        np.exp2(rng.uniform(-14, 8.8, 300000)).astype(np.float32)])
    v = v[v < 464.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codecs.e4m3_encode(v)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_satfinite():
    assert codecs.e4m3_encode(np.float32([464.0, 500.0, 1e30])).tolist() == [0x7E] * 3
    assert codecs.e4m3_encode(np.float32([2.0 ** -10])).tolist() == [0]       # tie to even (0)
    assert codecs.e4m3_encode(np.float32([2.0 ** -10 * 1.0001])).tolist() == [1]


def test_bf16_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(500000).astype(np.float32) * np.float32(1e3),
                        np.exp2(rng.uniform(-140, 120, 200000)).astype(np.float32),
                        np.float32([0.0, -0.0, 1.0, 3.3895314e38, 1e-45, -1e-45])])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(codecs.f32_to_bf16(v), ref)
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert codecs.f32_to_bf16(np.float32([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert codecs.f32_to_bf16(np.float32([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82


def test_nibble_packing_order():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    packed = codecs.pack_nibbles(codes)
    assert packed.tolist() == [[0x21, 0x43]]
    np.testing.assert_array_equal(codecs.unpack_nibbles(packed), codes)


def test_fnv1a64_published_vectors():
    with open(os.path.join(GOLDEN, "fnv1a64_vectors.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for s, h in rows:
        data = b"" if s == "<empty>" else s.encode()
        assert fnv.fnv1a64(data) == int(h, 16), s
