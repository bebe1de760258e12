"""The large-batch decode mixing split into three kernels (conv/norms/gates,
the delta rule alone, gated norm + quantisation; tuning knob 9) performs the
fused mixing kernel's operations in the same order, so whole decode steps are
bit-identical between the two: outputs, recurrent and conv states, for FP32
and BF16 state, with padding rows and a repeated slot (both refused)."""
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


@pytest.mark.parametrize("shape_name,B,state_bf16", [("FULL", 40, False), ("FULL", 40, True), ("TINY", 7, False),
                                                     ("TP2", 33, False)])
def test_split_mixing_is_bitwise_the_fused_kernel(api, shape_name, B, state_bf16):
    shape = getattr(synth, shape_name)
    seed = 0 if shape_name == "TINY" else 1
    L = api.layer_from_synth(weights(shape_name, seed), max_batch=64, state_bf16=state_bf16)
    nslots = B + 2
    x, conv0, ssm0 = slot_inputs(shape, list(range(B)), 2)
    _, c_extra, s_extra = slot_inputs(shape, list(range(B, nslots)), 1)
    conv0 = np.concatenate([conv0, c_extra])
    ssm0 = np.concatenate([ssm0, s_extra])
    if state_bf16:
        from oracle import codecs
        ssm0 = codecs.f32_to_bf16(ssm0)
    slots = list(range(B))
    slots[1] = -1            # padding
    slots[3] = slots[4]      # a repeated slot: both rows refused
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    res = {}
    try:
        for knob in (1, 2):
            api.lib().gdn_set_tuning(9, knob)
            c, s = to_dev(conv0), to_dev(ssm0)
            outs = np.stack([to_host(L.decode_step(to_dev(x[t]), ids, c, s)) for t in range(2)])
            st = L.check()
            res[knob] = (outs, to_host(c), to_host(s), st)
    finally:
        api.lib().gdn_set_tuning(9, 0)
    assert res[1][3] == res[2][3] == 6                     # GDN_E_RANGE flagged by both
    for a, b in zip(res[1][:3], res[2][:3]):
        np.testing.assert_array_equal(a, b)
    outs, c, s, _ = res[2]
    assert not outs[:, [1, 3, 4]].any()                     # refused rows read zero
    np.testing.assert_array_equal(s[[3, 4]], ssm0[[3, 4]])  # and touch no state
