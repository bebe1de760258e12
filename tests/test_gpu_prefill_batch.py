"""Large-batch decode (batch 64/128/256, 64 steps) and prefill (T = 1024,
4096, 16384) against the oracle.

Large batches: sequences are independent, so the oracle runs a sample of the
slots through all 64 steps and the GPU rows of those slots must match.
Prefill: at T = 1024, 4096 and 16384 against the oracle's token-by-token
recurrence over the whole output and the whole final state (rel-L2 <= 2e-3),
and against T decode steps of the same sequence on the GPU."""
import numpy as np
import pytest

from conftest import rel_l2
from helpers import oracle_layer, slot_inputs, to_dev, to_host, weights
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


@pytest.mark.parametrize("B", [64, 128, 256])
def test_large_batch_sampled_slots(api, B):
    steps = 64
    layer = api.layer_from_synth(weights("FULL", 1), max_batch=B)
    slots = list(range(B))
    x, conv0, ssm0 = slot_inputs(synth.FULL, slots, steps)
    conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    xd = to_dev(x)
    outs = np.stack([to_host(layer.decode_step(xd[t], ids, conv_d, ssm_d)) for t in range(steps)])
    assert layer.check() == 0
    O = oracle_layer("FULL", 1)
    sample = sorted({0, 1, B // 2 + 3, B - 1})
    for s in sample:
        c, st = conv0[s:s + 1].copy(), ssm0[s:s + 1].copy()
        want = np.stack([O.decode_step(x[t, s:s + 1], [0], c, st)[0] for t in range(steps)])
        assert rel_l2(_bf(outs[:, s]), _bf(want)) <= 4e-3, s
        assert rel_l2(to_host(ssm_d)[s], st[0]) <= 1e-4, s


def _prefill_vs_decode(api, T):
    """gdn_prefill of T tokens from zero state, and the same sequence as T
    gdn_decode_step calls: outputs within 2e-3, conv state bit-equal."""
    layer = api.layer_from_synth(weights("FULL", 1), max_batch=1, max_prefill_tokens=T)
    x = synth.x_tokens(synth.FULL, 7, T)
    conv_d, ssm_d = layer.new_states(2)
    out_p = to_host(layer.prefill(to_dev(x), 1, True, conv_d, ssm_d))
    assert layer.check() == 0
    conv_p, ssm_p = to_host(conv_d)[1].copy(), to_host(ssm_d)[1].copy()
    # the same sequence as T decode steps from zero state
    conv2, ssm2 = layer.new_states(2)
    ids = torch.ones(1, dtype=torch.int32, device="cuda")
    xd = to_dev(x)
    out_d = np.stack([to_host(layer.decode_step(xd[t:t + 1], ids, conv2, ssm2))[0] for t in range(T)])
    assert rel_l2(_bf(out_p), _bf(out_d)) <= 2e-3
    assert rel_l2(ssm_p, to_host(ssm2)[1]) <= 2e-3
    np.testing.assert_array_equal(conv_p, to_host(conv2)[1])
    return x, out_p, conv_p, ssm_p


@pytest.mark.parametrize("T", [1024, 4096, 16384])
def test_prefill_matches_oracle_recurrence(api, T):
    """Chunked prefill (config 4: batch 1, T = 1024 / 4096 / 16384, zero
    initial state, x seed 7) against the oracle's token-by-token recurrence
    over the whole output and the whole final state (rel-L2 <= 2e-3), and
    against T decode steps on the GPU. The oracle runs on every host core
    (oracle.parallel, bit-identical to its single-thread prefill)."""
    from oracle import parallel
    x, out_p, conv_p, ssm_p = _prefill_vs_decode(api, T)
    c = synth.conv_state(synth.FULL, 7, True)
    s = synth.ssm_state(synth.FULL, 7, True)
    want = parallel.prefill(weights("FULL", 1), x, c, s, init_zero=True)
    assert rel_l2(_bf(out_p), _bf(want)) <= 2e-3
    assert rel_l2(ssm_p, s) <= 2e-3
    assert rel_l2(_bf(conv_p), _bf(c)) <= 4e-3


@pytest.mark.parametrize("shape_name,seed,T", [("TINY", 0, 150), ("TINY", 0, 64), ("TINY", 0, 1), ("FULL", 1, 200)])
def test_prefill_ragged_and_continued_matches_oracle(api, shape_name, seed, T):
    """Ragged last chunk, a single token, and a prompt split in two calls (the
    second continues from the slot's state) against the oracle's recurrence."""
    shape = getattr(synth, shape_name)
    layer = api.layer_from_synth(weights(shape_name, seed), max_batch=1, max_prefill_tokens=T)
    O = oracle_layer(shape_name, seed)
    x = synth.x_tokens(shape, 7, T)
    conv_d, ssm_d = layer.new_states(3)
    split = max(1, T // 3)
    out1 = to_host(layer.prefill(to_dev(x[:split]), 2, True, conv_d, ssm_d))
    out2 = to_host(layer.prefill(to_dev(x[split:]), 2, False, conv_d, ssm_d)) if split < T else np.zeros((0, shape.hidden), np.uint16)
    assert layer.check() == 0
    got = np.concatenate([out1, out2])
    c = synth.conv_state(shape, 7, True)
    s = synth.ssm_state(shape, 7, True)
    want = O.prefill(x, c, s, init_zero=True)
    assert rel_l2(_bf(got), _bf(want)) <= 2e-3
    assert rel_l2(to_host(ssm_d)[2], s) <= 2e-3
    np.testing.assert_array_equal(to_host(ssm_d)[0], 0)          # other slots untouched
    assert rel_l2(_bf(to_host(conv_d)[2]), _bf(c)) <= 4e-3
