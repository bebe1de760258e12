"""The BF16-stored recurrent state (config state_bf16 = 1): the state is
loaded to FP32, updated in FP32 and stored rounded to nearest even after every
decode step; a prefill call carries it in FP32 and rounds once at the end.
Against the oracle's BF16-state layer: BF16 outputs rel-L2 <= 4e-3, the state
rel-L2 <= 4e-3; prefill outputs against the token-by-token recurrence
rel-L2 <= 2e-3. And bit-level: from a BF16-representable state, one step of
the BF16-state layer gives the FP32 layer's output and the FP32 layer's new
state rounded to BF16, bit for bit (same kernels, same order; only the store
differs)."""
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


def _to_bf16_bits(a):
    from oracle import codecs
    return codecs.f32_to_bf16(np.asarray(a, np.float32))


def _oracle16(shape_name, seed):
    from oracle import gdn
    return gdn.Layer(weights(shape_name, seed), state_bf16=True)


@pytest.mark.parametrize("B,steps", [(1, 64), (4, 4), (16, 2)])
def test_bf16_state_decode_matches_oracle(api, B, steps):
    sh = synth.FULL
    L = api.layer_from_synth(weights("FULL", 1), max_batch=16, state_bf16=True)
    O = _oracle16("FULL", 1)
    slots = list(range(B))
    x, conv0, ssm0 = slot_inputs(sh, slots, steps)
    s16 = _to_bf16_bits(ssm0)                             # the state as stored
    conv_d, ssm_d = to_dev(conv0), to_dev(s16)
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    got = np.stack([to_host(L.decode_step(to_dev(x[t]), ids, conv_d, ssm_d)) for t in range(steps)])
    assert L.check() == 0
    c, s = conv0.copy(), _bf(s16).copy()
    want = np.stack([O.decode_step(x[t], slots, c, s) for t in range(steps)])
    assert rel_l2(_bf(got), _bf(want)) <= 4e-3
    assert rel_l2(_bf(to_host(ssm_d)), s) <= 4e-3
    assert rel_l2(_bf(to_host(conv_d)), _bf(c)) <= 4e-3


def test_bf16_state_first_step_is_the_fp32_step_rounded(api):
    sh = synth.FULL
    w = weights("FULL", 1)
    L32 = api.layer_from_synth(w, max_batch=4)
    L16 = api.layer_from_synth(w, max_batch=4, state_bf16=True)
    slots = [0, 1, 2]
    x, conv0, ssm0 = slot_inputs(sh, slots, 1)
    s16 = _to_bf16_bits(ssm0)
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    ca, sa = to_dev(conv0), to_dev(_bf(s16))              # FP32 state holding BF16 values
    cb, sb = to_dev(conv0), to_dev(s16)
    oa = to_host(L32.decode_step(to_dev(x[0]), ids, ca, sa))
    ob = to_host(L16.decode_step(to_dev(x[0]), ids, cb, sb))
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(to_host(ca), to_host(cb))
    np.testing.assert_array_equal(to_host(sb), _to_bf16_bits(to_host(sa)))


def test_bf16_state_prefill_matches_oracle(api):
    sh = synth.FULL
    T = 200                                              # three chunks and a ragged tail
    L = api.layer_from_synth(weights("FULL", 1), max_batch=1, max_prefill_tokens=T, state_bf16=True)
    O = _oracle16("FULL", 1)
    x = synth.x_tokens(sh, 7, T)
    conv0 = synth.conv_state(sh, 9)
    s16 = _to_bf16_bits(synth.ssm_state(sh, 9))
    conv_d, ssm_d = to_dev(conv0[None]), to_dev(s16[None])
    out = to_host(L.prefill(to_dev(x), 0, False, conv_d, ssm_d))   # continue from the slot's state
    assert L.check() == 0
    c, s = conv0.copy(), _bf(s16).copy()
    want = O.prefill(x, c, s, init_zero=False)
    assert rel_l2(_bf(out), _bf(want)) <= 2e-3
    assert rel_l2(_bf(to_host(ssm_d)[0]), s) <= 4e-3
    assert rel_l2(_bf(to_host(conv_d)[0]), _bf(c)) <= 4e-3


def test_bf16_state_layer_refuses_fp32_state(api):
    L = api.layer_from_synth(weights("TINY", 0), max_batch=1, state_bf16=True)
    conv, _ = L.new_states(1)
    wrong = torch.zeros(1, 4, 32, 32, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        L.decode_step(torch.zeros(1, 256, dtype=torch.int16, device="cuda"),
                      torch.zeros(1, dtype=torch.int32, device="cuda"), conv, wrong)
