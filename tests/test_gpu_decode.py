"""GPU parity of the decode step against the oracle.

Tolerances (rel-L2 over the whole tensor): BF16 layer outputs 4e-3, FP32
intermediates 1e-5 (stage-wise, same inputs on both sides), the recurrent state
after 256 steps 1e-4."""
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


def _layer(api, shape_name, seed, max_batch=16, max_prefill=0):
    return api.layer_from_synth(weights(shape_name, seed), max_batch=max_batch, max_prefill_tokens=max_prefill)


def _bf16(bits):
    from oracle import codecs
    return codecs.bf16_to_f32(bits)


@pytest.mark.parametrize("shape_name,seed,steps,zero", [("TINY", 0, 8, True), ("FULL", 1, 256, False)])
def test_decode_sequence_matches_oracle(api, shape_name, seed, steps, zero):
    """configs: tiny (seed 0, 8 steps, zero state) and full width c1 (seed 1, 256 steps)."""
    shape = getattr(synth, shape_name)
    L = _layer(api, shape_name, seed)
    O = oracle_layer(shape_name, seed)
    x = synth.x_tokens(shape, seed, steps)
    conv0 = synth.conv_state(shape, seed, zero)[None]
    ssm0 = synth.ssm_state(shape, seed, zero)[None]
    conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    xd = to_dev(x)
    outs = [L.decode_step(xd[t:t + 1], slots, conv_d, ssm_d) for t in range(steps)]
    got = np.stack([to_host(o)[0] for o in outs])
    conv_o, ssm_o = conv0.copy(), ssm0.copy()
    want = np.stack([O.decode_step(x[t:t + 1], [0], conv_o, ssm_o)[0] for t in range(steps)])
    assert L.check() == 0
    assert rel_l2(_bf16(got), _bf16(want)) <= 4e-3
    assert rel_l2(to_host(ssm_d), ssm_o) <= 1e-4
    assert rel_l2(_bf16(to_host(conv_d)), _bf16(conv_o)) <= 4e-3


@pytest.mark.parametrize("shape_name,seed", [("TINY", 0), ("FULL", 1)])
def test_mix_stage_fp32_intermediates(api, shape_name, seed):
    """Same BF16 projections in, FP32 gated-norm output and state out: rel-L2 <= 1e-5."""
    shape = getattr(synth, shape_name)
    L = _layer(api, shape_name, seed)
    O = oracle_layer(shape_name, seed)
    slots_np = [3, 0, 1]
    x, conv0, ssm0 = slot_inputs(shape, slots_np, 1)
    qkvz, ba = O.projections(x[0])                        # oracle BF16 values -> GPU inputs
    from oracle import codecs
    qkvz_bits = codecs.f32_to_bf16(qkvz.astype(np.float32))
    ba_bits = codecs.f32_to_bf16(ba.astype(np.float32))
    S = 4
    conv_all = np.zeros((S,) + conv0.shape[1:], np.uint16)
    ssm_all = np.zeros((S,) + ssm0.shape[1:], np.float32)
    for i, s in enumerate(slots_np):
        conv_all[s], ssm_all[s] = conv0[i], ssm0[i]
    conv_d, ssm_d = to_dev(conv_all), to_dev(ssm_all)
    sl = torch.tensor(slots_np, dtype=torch.int32, device="cuda")
    y = L.mix_step(to_dev(qkvz_bits), to_dev(ba_bits), sl, conv_d, ssm_d)
    assert L.check() == 0
    for i, s in enumerate(slots_np):
        yw, cw, sw, _ = O.mix(qkvz[i], ba[i], conv_all[s], ssm_all[s])
        assert rel_l2(to_host(y)[i], yw) <= 1e-5
        assert rel_l2(to_host(ssm_d)[s], sw) <= 1e-5
        np.testing.assert_array_equal(to_host(conv_d)[s], cw)
    np.testing.assert_array_equal(to_host(ssm_d)[2], ssm_all[2])    # slot 2 untouched


def test_padding_rows_and_slot_errors(api):
    shape = synth.TINY
    L = _layer(api, "TINY", 0)
    O = oracle_layer("TINY", 0)
    x, conv0, ssm0 = slot_inputs(shape, [0, 1, 2], 1)
    xd = to_dev(x[0])
    conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
    out = L.decode_step(xd, torch.tensor([2, -1, 0], dtype=torch.int32, device="cuda"), conv_d, ssm_d)
    assert L.check() == 0
    o = to_host(out)
    assert (o[1] == 0).all()
    np.testing.assert_array_equal(to_host(ssm_d)[1], ssm0[1])
    np.testing.assert_array_equal(to_host(conv_d)[1], conv0[1])
    c, s = conv0.copy(), ssm0.copy()
    want = O.decode_step(x[0], [2, -1, 0], c, s)
    assert rel_l2(_bf16(o), _bf16(want)) <= 4e-3
    assert rel_l2(to_host(ssm_d), s) <= 1e-5
    # repeated slot and out-of-range slot: flagged, rows treated as padding
    before = to_host(ssm_d).copy()
    out = L.decode_step(xd, torch.tensor([1, 1, 7], dtype=torch.int32, device="cuda"), conv_d, ssm_d)
    assert L.check() == 6                                  # GDN_E_RANGE
    assert (to_host(out) == 0).all()
    np.testing.assert_array_equal(to_host(ssm_d), before)
    assert L.check() == 0                                  # cleared


def test_nonfinite_input_is_flagged(api):
    shape = synth.TINY
    L = _layer(api, "TINY", 0)
    x, conv0, ssm0 = slot_inputs(shape, [0], 1)
    xb = x[0].copy()
    xb[0, 5] = 0x7FC0                                       # BF16 NaN
    L.decode_step(to_dev(xb), torch.zeros(1, dtype=torch.int32, device="cuda"), to_dev(conv0), to_dev(ssm0))
    assert L.check() == 4                                   # GDN_E_NONFINITE
    assert L.check() == 0


@pytest.mark.parametrize("path", [1, 2, 0])
def test_batch_rows_equal_single_rows(api, path):
    """B rows in one call equal B single-row calls: bitwise when both run the
    same projection kernel (knob 0 = 1: CUDA cores, 2: tensor cores; there is
    no cross-row arithmetic and every reduction has a fixed order), and within
    the BF16 tolerance when the automatic choice runs B = 1 and B = 5 on
    different kernels."""
    shape = synth.FULL
    L = _layer(api, "FULL", 1)
    api.lib().gdn_set_tuning(0, path)
    api.lib().gdn_set_tuning(8, 1)   # one row on the same FP16 GEMV as five
    try:
        slots = [0, 1, 2, 3, 4]
        x, conv0, ssm0 = slot_inputs(shape, slots, 1)
        cb, sb = to_dev(conv0), to_dev(ssm0)
        ob = to_host(L.decode_step(to_dev(x[0]), torch.arange(5, dtype=torch.int32, device="cuda"), cb, sb))
        for i in slots:
            c1, s1 = to_dev(conv0), to_dev(ssm0)
            o1 = to_host(L.decode_step(to_dev(x[0][i:i + 1]), torch.tensor([i], dtype=torch.int32, device="cuda"),
                                       c1, s1))
            if path:
                np.testing.assert_array_equal(o1[0], ob[i])
                np.testing.assert_array_equal(to_host(s1)[i], to_host(sb)[i])
            else:
                assert rel_l2(_bf16(o1[0]), _bf16(ob[i])) <= 4e-3
                assert rel_l2(to_host(s1)[i], to_host(sb)[i]) <= 1e-5
    finally:
        api.lib().gdn_set_tuning(0, 0)
        api.lib().gdn_set_tuning(8, 0)


@pytest.mark.parametrize("shape_name,seed", [("TINY", 0), ("FULL", 1), ("TP2", 1)])
def test_one_row_warp_mma_gemv_matches_fp16_gemv_and_oracle(api, shape_name, seed):
    """The one-row projections with warp-level MMA block products (knob 8,
    the default) against the FP16x2-chain GEMV (knob 8 = 1) and the oracle:
    both exact per 16-block, FP32 across blocks in different orders, so the
    step's outputs agree to the BF16 tolerance and the states to 1e-5."""
    shape = getattr(synth, shape_name)
    L = _layer(api, shape_name, seed)
    O = oracle_layer(shape_name, seed)
    x, conv0, ssm0 = slot_inputs(shape, [0], 4)
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = {}
    try:
        for knob in (1, 2):
            api.lib().gdn_set_tuning(8, knob)
            c, s = to_dev(conv0), to_dev(ssm0)
            outs = np.stack([to_host(L.decode_step(to_dev(x[t]), ids, c, s)) for t in range(4)])
            assert L.check() == 0
            res[knob] = (outs, to_host(s))
    finally:
        api.lib().gdn_set_tuning(8, 0)
    assert rel_l2(_bf16(res[2][0]), _bf16(res[1][0])) <= 4e-3
    assert rel_l2(res[2][1], res[1][1]) <= 1e-5
    c, s = conv0.copy(), ssm0.copy()
    want = np.stack([O.decode_step(x[t], [0], c, s) for t in range(4)])
    assert rel_l2(_bf16(res[2][0]), _bf16(want)) <= 4e-3
    assert rel_l2(res[2][1], s) <= 1e-4


def test_fused_single_kernel_step_matches_oracle(api):
    """The one-launch decode step (tuning knob 3 = 2) for one and two rows."""
    shape = synth.FULL
    L = _layer(api, "FULL", 1)
    O = oracle_layer("FULL", 1)
    api.lib().gdn_set_tuning(3, 2)
    try:
        for B in (1, 2):
            x, conv0, ssm0 = slot_inputs(shape, list(range(B)), 3)
            conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
            ids = torch.arange(B, dtype=torch.int32, device="cuda")
            got = np.stack([to_host(L.decode_step(to_dev(x[t]), ids, conv_d, ssm_d)) for t in range(3)])
            assert L.check() == 0
            c, s = conv0.copy(), ssm0.copy()
            want = np.stack([O.decode_step(x[t], list(range(B)), c, s) for t in range(3)])
            assert rel_l2(_bf16(got), _bf16(want)) <= 4e-3
            assert rel_l2(to_host(ssm_d), s) <= 1e-4
            assert rel_l2(_bf16(to_host(conv_d)), _bf16(c)) <= 4e-3
    finally:
        api.lib().gdn_set_tuning(3, 0)


@pytest.mark.parametrize("shape_name,B", [("TINY", 3), ("FULL", 1), ("FULL", 7), ("FULL", 16)])
def test_in_projection_quantising_inside_the_gemm(api, shape_name, B):
    """Tensor-core decode (knob 0 = 2): the in-projection GEMM that quantises
    x itself (knob 4 = 2) gives bit-identical outputs and states to a separate
    quantisation kernel followed by the GEMM (knob 4 = 1) -- the same block
    quantiser, the same MMA order -- and so do weights streamed from the
    pre-swizzled tile copy (knob 6 = 2) or by tensor-map copies (knob 6 = 1);
    with one padding row, and matching the oracle."""
    shape = getattr(synth, shape_name)
    seed = 0 if shape_name == "TINY" else 1
    L = _layer(api, shape_name, seed)
    O = oracle_layer(shape_name, seed)
    slots = list(range(B))
    if B > 1:
        slots[1] = -1                                   # a padding row
    x, conv0, ssm0 = slot_inputs(shape, list(range(B)), 2)
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    res = {}
    api.lib().gdn_set_tuning(0, 2)
    try:
        for knob in ((1, 1), (2, 1), (1, 2), (2, 2)):
            api.lib().gdn_set_tuning(4, knob[0])
            api.lib().gdn_set_tuning(6, knob[1])
            c, s = to_dev(conv0), to_dev(ssm0)
            outs = [to_host(L.decode_step(to_dev(x[t]), ids, c, s)) for t in range(2)]
            assert L.check() == 0
            res[knob] = (np.stack(outs), to_host(c), to_host(s))
    finally:
        for k in (0, 4, 6):
            api.lib().gdn_set_tuning(k, 0)
    for knob in ((2, 1), (1, 2), (2, 2)):
        for a, b in zip(res[(1, 1)], res[knob]):
            np.testing.assert_array_equal(a, b)
    got, conv_g, ssm_g = res[(2, 2)]
    c, s = conv0.copy(), ssm0.copy()
    want = np.stack([O.decode_step(x[t], slots, c, s) for t in range(2)])
    assert rel_l2(_bf16(got), _bf16(want)) <= 4e-3
    assert rel_l2(ssm_g, s) <= 1e-4
    assert rel_l2(_bf16(conv_g), _bf16(c)) <= 4e-3
    if B > 1:
        assert not got[:, 1].any()                      # padding row: zero output
        np.testing.assert_array_equal(ssm_g[1], ssm0[1])  # and its slot untouched


def test_in_proj_stage_matches_oracle_projections(api):
    """gdn_in_proj (the in-projection alone, one row and four rows, one padding
    row): the BF16 projections against the oracle's exact W4A4 product rounded
    to BF16 -- equal up to the FP32 summation order of the blocks (rel-L2 <= 1e-5
    on the BF16 values, most elements bit-equal)."""
    shape = synth.FULL
    L = _layer(api, "FULL", 1)
    O = oracle_layer("FULL", 1)
    for B in (1, 4):
        x, _, _ = slot_inputs(shape, list(range(B)), 1)
        ids = list(range(B))
        if B > 1:
            ids[2] = -1
        got = to_host(L.in_proj(to_dev(x[0]), torch.tensor(ids, dtype=torch.int32, device="cuda")))
        qkvz, ba = O.projections(x[0])
        want = np.concatenate([qkvz, ba], axis=1)
        live = [i for i in range(B) if ids[i] >= 0]
        assert rel_l2(_bf16(got[live]), want[live]) <= 1e-5
        assert np.mean(_bf16(got[live]) == want[live]) > 0.99
        if B > 1:
            assert not got[2].any()


def test_in_proj_stage_at_prompt_size_matches_oracle_rows(api):
    """gdn_in_proj over a prompt-sized block of rows (more than max_batch, up to
    max_prefill_tokens: the persistent tensor-core GEMM with several output
    tiles per CTA and a ragged last token tile) against the oracle's W4A4
    product on sampled rows, and rows past the capacity refused."""
    shape = synth.FULL
    T = 1000
    L = api.layer_from_synth(weights("FULL", 1), max_batch=4, max_prefill_tokens=T)
    O = oracle_layer("FULL", 1)
    x = synth.x_tokens(shape, 7, T)
    got = to_host(L.in_proj(to_dev(x)))
    rows = [0, 1, 127, 128, 555, 999]
    qkvz, ba = O.projections(x[rows])
    want = np.concatenate([qkvz, ba], axis=1)
    assert rel_l2(_bf16(got[rows]), want) <= 1e-5
    assert np.mean(_bf16(got[rows]) == want) > 0.99
    with pytest.raises(api.GdnError):
        L.in_proj(to_dev(synth.x_tokens(shape, 7, T + 1)))
