"""The two-way head-parallel slice of the full layer (8 key heads, 16 value
heads, hidden 2048; one rank's share, no collective) through the same kernels:
decode buckets on both projection paths and a chunked prefill, against the
oracle at the layer tolerances (BF16 outputs rel-L2 <= 4e-3, the state
rel-L2 <= 1e-4 after decode; chunked prefill against the token-by-token
recurrence rel-L2 <= 2e-3)."""
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


def _bf16(bits):
    from oracle import codecs
    return codecs.bf16_to_f32(bits)


@pytest.mark.parametrize("B", [1, 4, 16])
def test_tp2_slice_decode_matches_oracle(api, B):
    shape = synth.TP2
    L = api.layer_from_synth(weights("TP2", 1), max_batch=16)
    O = oracle_layer("TP2", 1)
    slots = list(range(B))
    x, conv0, ssm0 = slot_inputs(shape, slots, 3)
    conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    got = np.stack([to_host(L.decode_step(to_dev(x[t]), ids, conv_d, ssm_d)) for t in range(3)])
    assert L.check() == 0
    c, s = conv0.copy(), ssm0.copy()
    want = np.stack([O.decode_step(x[t], slots, c, s) for t in range(3)])
    assert rel_l2(_bf16(got), _bf16(want)) <= 4e-3
    assert rel_l2(to_host(ssm_d), s) <= 1e-4
    assert rel_l2(_bf16(to_host(conv_d)), _bf16(c)) <= 4e-3


def test_tp2_slice_prefill_matches_oracle(api):
    shape = synth.TP2
    T = 200                                              # three full chunks and a ragged tail
    L = api.layer_from_synth(weights("TP2", 1), max_batch=1, max_prefill_tokens=T)
    O = oracle_layer("TP2", 1)
    x = synth.x_tokens(shape, 7, T)
    conv_d, ssm_d = L.new_states(1)
    out = to_host(L.prefill(to_dev(x), 0, True, conv_d, ssm_d))
    assert L.check() == 0
    c = synth.conv_state(shape, 7, True)
    s = synth.ssm_state(shape, 7, True)
    want = O.prefill(x, c, s, init_zero=True)
    assert rel_l2(_bf16(out), _bf16(want)) <= 2e-3
    assert rel_l2(to_host(ssm_d)[0], s) <= 2e-3
    assert rel_l2(_bf16(to_host(conv_d)[0]), _bf16(c)) <= 4e-3
