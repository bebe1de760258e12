"""Multi-token verify and its commit on the GPU (gdn_verify, gdn_verify_commit):
outputs and per-token state snapshots against the oracle (BF16 outputs
rel-L2 <= 4e-3, states rel-L2 <= 1e-4), bit-identity with the same number of
gdn_decode_step calls when both run their projections on the tensor cores
(tuning knob 0 = 2; the mixing kernel's order does not depend on how many rows
it serves) and agreement within tolerance under the automatic kernel choice,
commits of 0, some and all tokens, and a padding row."""
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


def _inputs(sh, B, r, nslots):
    x = np.stack([synth.x_tokens(sh, 40 + b, r) for b in range(B)])          # [B][r][H]
    conv0 = np.stack([synth.conv_state(sh, synth.slot_seed(s)) for s in range(nslots)])
    ssm0 = np.stack([synth.ssm_state(sh, synth.slot_seed(s)) for s in range(nslots)])
    return x, conv0, ssm0


def test_verify_matches_oracle_and_commits(api):
    sh, B, r = synth.FULL, 3, 4
    slots = [2, -1, 0]
    L = api.layer_from_synth(weights("FULL", 1), max_batch=16)
    O = oracle_layer("FULL", 1)
    x, conv0, ssm0 = _inputs(sh, B, r, 3)
    cd, sd = to_dev(conv0), to_dev(ssm0)
    snap_c, snap_s = L.new_snapshots(B, r)
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    out = to_host(L.verify(to_dev(x), ids, cd, sd, snap_c, snap_s))
    assert L.check() == 0
    np.testing.assert_array_equal(to_host(cd), conv0)                       # slots untouched
    np.testing.assert_array_equal(to_host(sd), ssm0)
    c, s = conv0.copy(), ssm0.copy()
    want, snaps = O.verify(x, slots, c, s)
    live = [0, 2]
    assert rel_l2(_bf(out[live]), _bf(want[live])) <= 4e-3
    assert not out[1].any()                                                   # padding row
    gs, gc = to_host(snap_s), to_host(snap_c)
    for b in live:
        for t in range(r):
            assert rel_l2(gs[b, t], snaps[b][t][1]) <= 1e-4
            assert rel_l2(_bf(gc[b, t]), _bf(snaps[b][t][0])) <= 4e-3
    # commit: row 0 (slot 2) keeps its state, row 2 (slot 0) takes token 3's
    acc = torch.tensor([0, 1, 3], dtype=torch.int32, device="cuda")
    L.verify_commit(ids, acc, snap_c, snap_s, cd, sd)
    assert L.check() == 0
    hs, hc = to_host(sd), to_host(cd)
    np.testing.assert_array_equal(hs[2], ssm0[2])
    np.testing.assert_array_equal(hs[1], ssm0[1])                             # untouched slot
    np.testing.assert_array_equal(hs[0], gs[2, 2])
    np.testing.assert_array_equal(hc[0], gc[2, 2])


@pytest.mark.parametrize("state_bf16", [False, True])
def test_verify_commit_all_is_bitwise_r_decode_steps(api, state_bf16):
    sh, B, r = synth.FULL, 3, 4
    L = api.layer_from_synth(weights("FULL", 1), max_batch=16, state_bf16=state_bf16)
    x, conv0, ssm0 = _inputs(sh, B, r, B)
    if state_bf16:
        from oracle import codecs
        ssm0 = codecs.f32_to_bf16(ssm0)
    ids = torch.arange(B, dtype=torch.int32, device="cuda")

    def run():
        # r decode steps
        ca, sa = to_dev(conv0), to_dev(ssm0)
        dec = np.stack([to_host(L.decode_step(to_dev(np.ascontiguousarray(x[:, t])), ids, ca, sa))
                        for t in range(r)], axis=1)
        # verify + commit of every token
        cb, sb = to_dev(conv0), to_dev(ssm0)
        snap_c, snap_s = L.new_snapshots(B, r)
        ver = to_host(L.verify(to_dev(x), ids, cb, sb, snap_c, snap_s))
        L.verify_commit(ids, torch.full((B,), r, dtype=torch.int32, device="cuda"), snap_c, snap_s, cb, sb)
        assert L.check() == 0
        return ver, dec, (to_host(sb), to_host(sa)), (to_host(cb), to_host(ca))

    # on the same projection kernels (tensor cores for B and for B * r rows): bit for bit
    api.lib().gdn_set_tuning(0, 2)
    try:
        ver, dec, (sv, sd), (cv, cd) = run()
    finally:
        api.lib().gdn_set_tuning(0, 0)
    np.testing.assert_array_equal(ver, dec)
    np.testing.assert_array_equal(sv, sd)
    np.testing.assert_array_equal(cv, cd)
    # with the automatic choice (B rows on the warp-MMA kernel, B * r on the tensor
    # cores) the two differ only by FP32 summation order
    ver, dec, (sv, sd), (cv, cd) = run()
    assert rel_l2(_bf(ver), _bf(dec)) <= 4e-3
    val = _bf if state_bf16 else (lambda a: a.astype(np.float64))
    assert rel_l2(val(sv), val(sd)) <= 1e-4


def test_verify_refuses_too_many_rows(api):
    L = api.layer_from_synth(weights("TINY", 0), max_batch=4)
    conv, ssm = L.new_states(2)
    snap_c, snap_s = L.new_snapshots(2, 3)
    x = torch.zeros(2, 3, 256, dtype=torch.int16, device="cuda")
    ids = torch.arange(2, dtype=torch.int32, device="cuda")
    with pytest.raises(api.GdnError):
        L.verify(x, ids, conv, ssm, snap_c, snap_s)                         # 6 rows > max_batch 4
