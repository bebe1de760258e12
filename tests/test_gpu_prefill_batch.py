"""Large-batch decode (batch 64/128/256, 64 steps) and prefill (T = 1024,
4096, 16384) against the oracle.

Large batches: sequences are independent, so the oracle runs a sample of the
slots through all 64 steps and the GPU rows of those slots must match.
Prefill: T = 1024 against the oracle's token-by-token recurrence over the whole
output; at every T the prefill must equal T decode steps of the same sequence
(rel-L2 <= 2e-3), and the final recurrent state of sampled value heads must
match the oracle's recurrence restricted to those heads."""
import math

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


def _prefill_vs_decode(api, T, check_oracle):
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


def test_prefill_1024_matches_oracle(api):
    T = 1024
    x, out_p, conv_p, ssm_p = _prefill_vs_decode(api, T, True)
    O = oracle_layer("FULL", 1)
    c = synth.conv_state(synth.FULL, 7, True)
    s = synth.ssm_state(synth.FULL, 7, True)
    want = O.prefill(x, c, s, init_zero=True)
    assert rel_l2(_bf(out_p), _bf(want)) <= 2e-3
    assert rel_l2(ssm_p, s) <= 2e-3
    assert rel_l2(_bf(conv_p), _bf(c)) <= 4e-3


def _oracle_heads_final_state(x, heads):
    """The oracle's recurrence for a few value heads only: the projection rows
    those heads read, conv, norms, gates and the delta rule, token by token."""
    from oracle import codecs, gdn, nvfp4
    sh = synth.FULL
    w = weights("FULL", 1)
    D, Hk, Hv = sh.d_k, sh.n_k_heads, sh.n_v_heads
    G = Hv // Hk
    xf = codecs.bf16_to_f32(x)
    xc, xs = nvfp4.quantize(xf, w.act_scale_in)
    xop = nvfp4.Operand(xc, xs, w.act_scale_in)
    conv_w = codecs.bf16_to_f32(w.conv_w).astype(np.float64)
    res = {}
    for h in heads:
        kh = h // G
        rows = (list(range(kh * D, kh * D + D)) + list(range(Hk * D + kh * D, Hk * D + kh * D + D))
                + list(range(2 * Hk * D + h * D, 2 * Hk * D + h * D + D)))
        wop = nvfp4.Operand(w.qkvz.codes[rows], w.qkvz.scales[rows], w.qkvz.tensor_scale)
        pre = codecs.round_bf16(nvfp4.gemm_op(xop, wop))                       # [T][3D] BF16 values
        ba_rows = [h, Hv + h]
        bop = nvfp4.Operand(w.ba.codes[ba_rows], w.ba.scales[ba_rows], w.ba.tensor_scale)
        ba = codecs.round_bf16(nvfp4.gemm_op(xop, bop))
        T = x.shape[0]
        win = np.zeros((3, 3 * D))
        cw = conv_w[rows]
        S = np.zeros((1, D, D), np.float32)
        beta, g = gdn.gates(ba[:, 0], ba[:, 1], w.A_log[h:h + 1].repeat(T), w.dt_bias[h:h + 1].repeat(T))
        for t in range(T):
            y, win = gdn.conv_step(win, pre[t], cw)
            q, k, v = y[:D], y[D:2 * D], y[2 * D:]
            kh_ = gdn.l2norm(k[None], w.l2_eps)
            qh_ = gdn.l2norm(q[None], w.l2_eps) / math.sqrt(D)
            _, S64 = gdn.delta_step(S.astype(np.float64), qh_, kh_, v[None], beta[t:t + 1], g[t:t + 1])
            S = S64.astype(np.float32)
        res[h] = S[0]
    return res


@pytest.mark.parametrize("T", [4096, 16384])
def test_prefill_long_vs_decode_and_sampled_heads(api, T):
    x, out_p, conv_p, ssm_p = _prefill_vs_decode(api, T, False)
    heads = [0, 31] if T == 4096 else [17]
    want = _oracle_heads_final_state(x, heads)
    for h in heads:
        assert rel_l2(ssm_p[h], want[h]) <= 2e-3, h


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
