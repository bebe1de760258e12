"""A bounded device wait that runs out reports GDN_E_TIMEOUT and leaves the
context usable.

The persistent single-kernel decode step (tuning knob 3 = 2) separates its
stages with grid barriers; knob 12 sets their wait budget. With a budget of one
SM cycle the first CTA to arrive cannot see the others in time, so it gives up
and records GDN_E_TIMEOUT. These waits guard no copy in flight, so giving up is
safe: the kernel finishes with meaningless results and the status word says so.
The barrier words are cleared before every launch, so the next call, with the
default budget, must be correct again."""
import pytest

from conftest import rel_l2
from helpers import oracle_layer, slot_inputs, to_dev, to_host, weights
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GDN_E_TIMEOUT = 10


def _bf(bits):
    from oracle import codecs
    return codecs.bf16_to_f32(bits)


def test_grid_barrier_timeout_is_reported_and_the_next_call_recovers():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import nvfp4_gated_deltanet_gb300 as pkg
    sh = synth.FULL
    layer = pkg.layer_from_synth(weights("FULL", 1), max_batch=16)
    x, conv0, ssm0 = slot_inputs(sh, [0], 1)
    xd, ids = to_dev(x[0]), torch.zeros(1, dtype=torch.int32, device="cuda")
    L = pkg.lib()
    try:
        assert L.gdn_set_tuning(3, 2) == 0       # the single-kernel step
        assert L.gdn_set_tuning(12, 1) == 0      # one-cycle barrier budget
        layer.decode_step(xd, ids, to_dev(conv0), to_dev(ssm0))
        assert layer.check() == GDN_E_TIMEOUT
        assert layer.check() == 0                # cleared by the read
        assert L.gdn_set_tuning(12, 0) == 0      # default budget
        conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
        got = to_host(layer.decode_step(xd, ids, conv_d, ssm_d))
        assert layer.check() == 0
    finally:
        L.gdn_set_tuning(12, 0)
        L.gdn_set_tuning(3, 0)
    c, s = conv0.copy(), ssm0.copy()
    want = oracle_layer("FULL", 1).decode_step(x[0], [0], c, s)
    assert rel_l2(_bf(got), _bf(want)) <= 4e-3
    assert rel_l2(to_host(ssm_d), s) <= 1e-4
    assert rel_l2(_bf(to_host(conv_d)), _bf(c)) <= 4e-3
    assert L.gdn_set_tuning(12, -1) == 6          # GDN_E_RANGE
