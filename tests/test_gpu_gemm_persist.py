"""The persistent forms of the tensor-core projections (tuning knob 11: one CTA
per SM walking the 128 x 128 output tiles with two TMEM accumulators; the
streaming form runs one operand ring across tiles, the weight-stationary form
keeps a weight tile and its scales resident while it walks token tiles) issue
the same MMAs in the same K order into one accumulator per tile and apply the
same scaling as the one-tile-per-CTA kernel, so prefill and large-batch decode
are bit-identical between all three: outputs, recurrent and conv states. The
sizes give each CTA several tiles (both accumulators reused, the ring wrapping
mid-tile, weight tiles reloaded mid-run) and ragged edges in both the token and
the weight-row direction."""
import numpy as np
import pytest

from helpers import slot_inputs, to_dev, to_host, weights
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

KNOB = 11


@pytest.fixture(scope="module")
def api():
    import nvfp4_gated_deltanet_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return pkg


def _all(api, run):
    res = {}
    try:
        for knob in (1, 2, 3):
            api.lib().gdn_set_tuning(KNOB, knob)
            res[knob] = run()
    finally:
        api.lib().gdn_set_tuning(KNOB, 0)
    return res


@pytest.mark.parametrize("shape_name,T", [("FULL", 1000), ("FULL", 2085), ("TP2", 333), ("TINY", 300)])
def test_persistent_prefill_is_bitwise_the_tile_kernel(api, shape_name, T):
    shape = getattr(synth, shape_name)
    seed = 0 if shape_name == "TINY" else 1
    layer = api.layer_from_synth(weights(shape_name, seed), max_batch=1, max_prefill_tokens=T)
    x = to_dev(synth.x_tokens(shape, 7, T))

    def run():
        conv, ssm = layer.new_states(1)
        out = to_host(layer.prefill(x, 0, True, conv, ssm))
        assert layer.check() == 0
        return out, to_host(conv), to_host(ssm)

    res = _all(api, run)
    for k in (2, 3):
        for a, b in zip(res[1], res[k]):
            np.testing.assert_array_equal(a, b)
    assert np.any(res[2][0])


@pytest.mark.parametrize("B", [200, 256])
def test_persistent_large_batch_is_bitwise_the_tile_kernel(api, B):
    layer = api.layer_from_synth(weights("FULL", 1), max_batch=B)
    x, conv0, ssm0 = slot_inputs(synth.FULL, list(range(B)), 2)
    ids = torch.arange(B, dtype=torch.int32, device="cuda")

    def run():
        c, s = to_dev(conv0), to_dev(ssm0)
        outs = np.stack([to_host(layer.decode_step(to_dev(x[t]), ids, c, s)) for t in range(2)])
        assert layer.check() == 0
        return outs, to_host(c), to_host(s)

    res = _all(api, run)
    for k in (2, 3):
        for a, b in zip(res[1], res[k]):
            np.testing.assert_array_equal(a, b)
