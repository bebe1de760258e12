"""Decode buckets c1, c2, c4, c8, c16 captured as CUDA graphs: replays are
bit-identical by FNV-1a 64 of output, conv state and recurrent state, a reset
replay reproduces the hashes, and shrinking the batch zeroes inactive rows and
leaves their state untouched (Rocket blog, "A reduction barrier makes Qwen GDN
graph replay bit exact": five replays after warmup, reset replay, c16 -> c1)."""
import numpy as np
import pytest

from conftest import rel_l2
from helpers import oracle_layer, slot_inputs, to_dev, to_host, weights
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

BUCKETS = [1, 2, 4, 8, 16]


@pytest.fixture(scope="module")
def setup():
    import nvfp4_gated_deltanet_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from nvfp4_gated_deltanet_gb300.graphs import DecodeGraphs
    layer = pkg.layer_from_synth(weights("FULL", 1), max_batch=16)
    S = 16
    x, conv0, ssm0 = slot_inputs(synth.FULL, list(range(S)), 1)
    conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
    graphs = DecodeGraphs(layer, conv_d, ssm_d, buckets=BUCKETS, max_batch=16)
    return pkg, layer, graphs, x, conv0, ssm0, conv_d, ssm_d


def _hashes(out_rows, conv_d, ssm_d):
    from oracle import fnv
    return (fnv.fnv1a64(to_host(out_rows)), fnv.fnv1a64(to_host(conv_d)), fnv.fnv1a64(to_host(ssm_d)))


@pytest.mark.parametrize("B", BUCKETS)
def test_bucket_replays_bit_identical(setup, B):
    pkg, layer, graphs, x, conv0, ssm0, conv_d, ssm_d = setup
    graphs.x[:B].copy_(to_dev(x[0][:B]))
    graphs.slot_ids[:B].copy_(torch.arange(B, dtype=torch.int32))
    seen = []
    for rep in range(2):                          # a first pass and a reset replay
        conv_d.copy_(to_dev(conv0))
        ssm_d.copy_(to_dev(ssm0))
        graphs.replay(B)                          # warm-up replay
        hs = []
        for _ in range(5):
            conv_d.copy_(to_dev(conv0))           # every replay from the same state
            ssm_d.copy_(to_dev(ssm0))
            graphs.replay(B)
            torch.cuda.synchronize()
            hs.append(_hashes(graphs.out[:B], conv_d, ssm_d))
        assert len(set(hs)) == 1, hs
        seen.append(hs[0])
    assert seen[0] == seen[1]
    assert layer.check() == 0
    # and the replayed step is the oracle's step
    O = oracle_layer("FULL", 1)
    c, s = conv0.copy(), ssm0.copy()
    want = O.decode_step(x[0][:B], list(range(B)), c, s)
    from oracle import codecs
    assert rel_l2(codecs.bf16_to_f32(to_host(graphs.out[:B])), codecs.bf16_to_f32(want)) <= 4e-3
    assert rel_l2(to_host(ssm_d)[:B], s[:B]) <= 1e-4


def test_c16_to_c1_transition(setup):
    pkg, layer, graphs, x, conv0, ssm0, conv_d, ssm_d = setup
    conv_d.copy_(to_dev(conv0))
    ssm_d.copy_(to_dev(ssm0))
    graphs.x[:16].copy_(to_dev(x[0][:16]))
    graphs.slot_ids[:16].copy_(torch.arange(16, dtype=torch.int32))
    graphs.replay(16)
    torch.cuda.synchronize()
    assert (to_host(graphs.out[:16]) != 0).any(axis=1).all()
    # c16 graph with 15 rows now inactive: their output rows read zero, their state is untouched
    conv_before, ssm_before = to_host(conv_d).copy(), to_host(ssm_d).copy()
    ids = torch.full((16,), -1, dtype=torch.int32)
    ids[0] = 0
    graphs.slot_ids[:16].copy_(ids)
    graphs.replay(16)
    torch.cuda.synchronize()
    o = to_host(graphs.out[:16])
    assert (o[1:] == 0).all() and (o[0] != 0).any()
    np.testing.assert_array_equal(to_host(ssm_d)[1:], ssm_before[1:])
    np.testing.assert_array_equal(to_host(conv_d)[1:], conv_before[1:])
    # c1 graph with its only row inactive: zero output, every slot (slot 0 too) unchanged
    conv_before, ssm_before = to_host(conv_d).copy(), to_host(ssm_d).copy()
    graphs.slot_ids[:1].fill_(-1)
    graphs.replay(1)
    torch.cuda.synchronize()
    assert (to_host(graphs.out[:1]) == 0).all()
    np.testing.assert_array_equal(to_host(ssm_d), ssm_before)
    np.testing.assert_array_equal(to_host(conv_d), conv_before)
    assert layer.check() == 0


def test_negative_control_wrong_slot_changes_hash(setup):
    """Pointing a row at another slot's state must change the hashes."""
    pkg, layer, graphs, x, conv0, ssm0, conv_d, ssm_d = setup
    res = []
    for sid in (0, 5):
        conv_d.copy_(to_dev(conv0))
        ssm_d.copy_(to_dev(ssm0))
        graphs.x[:1].copy_(to_dev(x[0][:1]))
        graphs.slot_ids[:1].fill_(sid)
        graphs.replay(1)
        torch.cuda.synchronize()
        res.append(_hashes(graphs.out[:1], conv_d, ssm_d))
    assert res[0][0] != res[1][0] and res[0][2] != res[1][2]


def test_stack_graph_equals_eager_steps():
    """DecodeStackGraph (one graph of several layers' decode steps, each layer
    with its own weights and states) gives bit-identically the outputs and
    states of the same steps launched one by one, over two steps."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import nvfp4_gated_deltanet_gb300 as pkg
    from nvfp4_gated_deltanet_gb300.graphs import DecodeStackGraph
    n, B = 3, 2
    layers = [pkg.layer_from_synth(weights("TINY", 0), max_batch=4) for _ in range(n)]
    x, conv0, ssm0 = slot_inputs(synth.TINY, list(range(B)), 2)
    st_g = [(to_dev(conv0), to_dev(ssm0)) for _ in range(n)]
    st_e = [(to_dev(conv0), to_dev(ssm0)) for _ in range(n)]
    sg = DecodeStackGraph(layers, st_g, B)
    # the capture's warm-up launch stepped the graph states once from zero
    # input rows; put them back
    for (c, m) in st_g:
        c.copy_(to_dev(conv0))
        m.copy_(to_dev(ssm0))
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    for step in range(2):
        xs = torch.stack([to_dev(x[step]) for _ in range(n)])
        got = sg.step(xs).clone()
        for i, (L, (c, m)) in enumerate(zip(layers, st_e)):
            want = L.decode_step(xs[i], ids, c, m)
            np.testing.assert_array_equal(to_host(got[i]), to_host(want))
    for (cg, mg), (ce, me) in zip(st_g, st_e):
        np.testing.assert_array_equal(to_host(cg), to_host(ce))
        np.testing.assert_array_equal(to_host(mg), to_host(me))
