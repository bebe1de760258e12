"""The decode step with the in-projection inside the mixing kernel (up to 8
rows, tuning knob 13) against the three-kernel step on the warp-MMA
projections with four K slices (knob 0 = 1, knob 13 = 1, knob 14 = 1): the same
arithmetic in the same order,
so outputs, conv state and recurrent state must agree bit for bit, step after
step -- with padding rows, a refused (repeated or out-of-range) slot, FP32 and
BF16 state, and the two-way head-parallel shape. Both are also held to the
oracle elsewhere (the decode and graph tests run the default path)."""
import numpy as np
import pytest

from helpers import slot_inputs, to_dev, to_host, weights
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    import nvfp4_gated_deltanet_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return pkg


def _run(api, layer, knobs, x, ids, conv0, ssm0, steps):
    L = api.lib()
    for k, v in knobs.items():
        assert L.gdn_set_tuning(k, v) == 0
    try:
        conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
        idd = torch.tensor(ids, dtype=torch.int32, device="cuda")
        outs = [to_host(layer.decode_step(to_dev(x[t]), idd, conv_d, ssm_d)) for t in range(steps)]
        status = layer.check()
    finally:
        for k in knobs:
            L.gdn_set_tuning(k, 0)
    return np.stack(outs), to_host(conv_d), to_host(ssm_d), status


CASES = [
    # shape, rows' slot ids (-1 = padding), state in BF16
    ("FULL", [0], False),
    ("FULL", [1, 0], False),
    ("FULL", [2, -1, 0], False),
    ("FULL", [4, 1, 3, 0, 2], False),
    ("FULL", [7, 6, 5, 4, 3, 2, 1, 0], False),
    ("FULL", [3, -1, 1, -1, 0, 2, -1, 5], False),
    ("FULL", [0], True),
    ("FULL", [3, 1, 0, 2], True),
    ("TP2", [0], False),
    ("TP2", [2, 0, 1], False),
]


@pytest.mark.parametrize("shape_name,ids,bf16", CASES)
def test_fused_step_bit_identical_to_three_kernel_step(api, shape_name, ids, bf16):
    shape = getattr(synth, shape_name)
    layer = api.layer_from_synth(weights(shape_name, 1), max_batch=16, state_bf16=bf16)
    S = 8
    steps = 3
    x, conv0, ssm0 = slot_inputs(shape, list(range(len(ids))), steps)
    conv_all = np.stack([synth.conv_state(shape, synth.slot_seed(s)) for s in range(S)])
    ssm_all = np.stack([synth.ssm_state(shape, synth.slot_seed(s)) for s in range(S)])
    if bf16:
        ssm_all = synth.to_bf16_bits(ssm_all)
    ref = _run(api, layer, {0: 1, 13: 1, 14: 1}, x, ids, conv_all, ssm_all, steps)
    got = _run(api, layer, {13: 2}, x, ids, conv_all, ssm_all, steps)
    assert ref[3] == 0 and got[3] == 0
    for a, b, what in zip(got[:3], ref[:3], ("out", "conv", "ssm")):
        np.testing.assert_array_equal(a, b, err_msg=what)
    for r, s in enumerate(ids):
        if s < 0:
            assert (got[0][:, r] == 0).all()
    untouched = [s for s in range(S) if s not in ids]
    for s in untouched:
        np.testing.assert_array_equal(got[2][s], ssm_all[s])
        np.testing.assert_array_equal(got[1][s], conv_all[s])


def test_fused_step_refuses_repeated_and_out_of_range_slots(api):
    shape = synth.FULL
    layer = api.layer_from_synth(weights("FULL", 1), max_batch=16)
    x, conv0, ssm0 = slot_inputs(shape, [0, 1, 2], 1)
    for ids in ([1, 1, 0], [0, 9, 2]):
        ref = _run(api, layer, {0: 1, 13: 1, 14: 1}, x, ids, conv0, ssm0, 1)
        got = _run(api, layer, {13: 2}, x, ids, conv0, ssm0, 1)
        assert ref[3] == 6 and got[3] == 6                  # GDN_E_RANGE
        for a, b in zip(got[:3], ref[:3]):
            np.testing.assert_array_equal(a, b)
        bad_rows = [r for r, s in enumerate(ids) if ids.count(s) > 1 or s >= 3]
        for r in bad_rows:
            assert (got[0][:, r] == 0).all()
