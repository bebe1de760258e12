"""The three forms of the prefill chunk stages (tuning knob 10) compute the
same chunk recurrence: tcgen05 MMAs with TMEM accumulators (the default for
d = 128; every product in split FP16 with power-of-two block scales), warp-level
MMA in split TF32, and FP32 on the CUDA cores. They must agree to FP32
rounding on ragged prompts from a non-zero state, and the tcgen05 form must
match the oracle's token recurrence on its own."""
import numpy as np
import pytest

from conftest import rel_l2
from helpers import oracle_layer, to_dev, to_host, weights
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    import nvfp4_gated_deltanet_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return pkg


def _bf(bits):
    from oracle import codecs
    return codecs.bf16_to_f32(bits)


def _prefill(api, shape_name, T, form):
    shape = getattr(synth, shape_name)
    L = api.lib()
    assert L.gdn_set_tuning(10, form) == 0
    try:
        layer = api.layer_from_synth(weights(shape_name, 1), max_batch=1, max_prefill_tokens=T)
        x = synth.x_tokens(shape, 7, T)
        conv_d, ssm_d = layer.new_states(2)
        ssm_d[1].copy_(to_dev(synth.ssm_state(shape, 7)))
        out = to_host(layer.prefill(to_dev(x), 1, False, conv_d, ssm_d))
        assert layer.check() == 0
        return out, to_host(ssm_d)[1].copy()
    finally:
        L.gdn_set_tuning(10, 0)


@pytest.mark.parametrize("shape_name,T", [("FULL", 1), ("FULL", 64), ("FULL", 333), ("FULL", 1024), ("TP2", 130)])
def test_scan_forms_agree(api, shape_name, T):
    o3, s3 = _prefill(api, shape_name, T, 3)
    o2, s2 = _prefill(api, shape_name, T, 2)
    o1, s1 = _prefill(api, shape_name, T, 1)
    for o, s in ((o2, s2), (o1, s1)):
        assert rel_l2(_bf(o3), _bf(o)) <= 1e-3
        assert rel_l2(s3, s) <= 1e-5
    o0, s0 = _prefill(api, shape_name, T, 0)  # the automatic choice is the tcgen05 form
    np.testing.assert_array_equal(o0, o3)
    np.testing.assert_array_equal(s0, s3)


def test_tcgen05_scan_matches_oracle_from_state(api):
    """A 200-token prompt (three chunks and a ragged tail) continuing from a
    non-zero recurrent state, against the oracle's token-by-token recurrence
    (the BF16-stored state form is covered by the BF16-state tests)."""
    shape = synth.FULL
    out, st = _prefill(api, "FULL", 200, 3)
    x = synth.x_tokens(shape, 7, 200)
    c = np.zeros((shape.conv_kernel - 1, shape.conv_channels), np.uint16)
    s = synth.ssm_state(shape, 7).copy()
    want = oracle_layer("FULL", 1).prefill(x, c, s, init_zero=False)
    assert rel_l2(_bf(out), _bf(want)) <= 2e-3
    assert rel_l2(st, s) <= 2e-3


@pytest.mark.parametrize("pattern", ["constant", "alternating"])
def test_chunk_forms_on_repeated_tokens(api, pattern):
    """Prompts of one repeated token (every key the same, so L is as large as
    it gets: L_ij = beta_i e^(Gamma_i - Gamma_j)) or of two alternating
    tokens: the tcgen05 chunk stages (W and U~ from an explicit (I + L)^-1)
    against the forward substitution of the warp-MMA form and against the
    oracle's token recurrence."""
    shape = synth.FULL
    T = 200
    base = synth.x_tokens(shape, 7, 2)
    x = np.stack([base[0] if (pattern == "constant" or t % 2 == 0) else base[1] for t in range(T)])
    L = api.lib()
    outs = {}
    try:
        for form in (3, 2):
            assert L.gdn_set_tuning(10, form) == 0
            layer = api.layer_from_synth(weights("FULL", 1), max_batch=1, max_prefill_tokens=T)
            conv_d, ssm_d = layer.new_states(2)
            ssm_d[1].copy_(to_dev(synth.ssm_state(shape, 7)))
            o = to_host(layer.prefill(to_dev(x), 1, False, conv_d, ssm_d))
            assert layer.check() == 0
            outs[form] = (o, to_host(ssm_d)[1].copy())
    finally:
        L.gdn_set_tuning(10, 0)
    assert rel_l2(_bf(outs[3][0]), _bf(outs[2][0])) <= 1e-3
    assert rel_l2(outs[3][1], outs[2][1]) <= 1e-5
    c = np.zeros((shape.conv_kernel - 1, shape.conv_channels), np.uint16)
    s = synth.ssm_state(shape, 7).copy()
    want = oracle_layer("FULL", 1).prefill(x, c, s, init_zero=False)
    assert rel_l2(_bf(outs[3][0]), _bf(want)) <= 2e-3
    assert rel_l2(outs[3][1], s) <= 2e-3


@pytest.mark.parametrize("scale", [1e-6, 1e6])
def test_tcgen05_scan_extreme_state_scales(api, scale):
    """The split-FP16 products scale each operand block by a power of two:
    S by its slice maximum, U and Cf by the bound max|U~| + d max|W| max|S|.
    A prompt continuing from a state scaled by 1e-6 or 1e6 (the state's
    contribution to U and to the output far below or far above the prompt's)
    must still match the warp-MMA form and the oracle's token recurrence."""
    shape = synth.FULL
    T = 200
    x = synth.x_tokens(shape, 7, T)
    s0 = (synth.ssm_state(shape, 7) * np.float32(scale)).astype(np.float32)
    L = api.lib()
    outs = {}
    try:
        for form in (3, 2):
            assert L.gdn_set_tuning(10, form) == 0
            layer = api.layer_from_synth(weights("FULL", 1), max_batch=1, max_prefill_tokens=T)
            conv_d, ssm_d = layer.new_states(2)
            ssm_d[1].copy_(to_dev(s0))
            o = to_host(layer.prefill(to_dev(x), 1, False, conv_d, ssm_d))
            assert layer.check() == 0
            outs[form] = (o, to_host(ssm_d)[1].copy())
    finally:
        L.gdn_set_tuning(10, 0)
    assert rel_l2(_bf(outs[3][0]), _bf(outs[2][0])) <= 1e-3
    assert rel_l2(outs[3][1], outs[2][1]) <= 1e-5
    c = np.zeros((shape.conv_kernel - 1, shape.conv_channels), np.uint16)
    s = s0.copy()
    want = oracle_layer("FULL", 1).prefill(x, c, s, init_zero=False)
    assert rel_l2(_bf(outs[3][0]), _bf(want)) <= 2e-3
    assert rel_l2(outs[3][1], s) <= 2e-3
