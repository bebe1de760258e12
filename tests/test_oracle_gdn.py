"""Pins of the oracle's layer stages: closed forms, invariants the definition
fixes, and the chunked form against the token recurrence."""
import math

import numpy as np
import pytest

from conftest import rel_l2
from nvfp4_gated_deltanet_gb300 import synth
from oracle import codecs, gdn


# ------------------------------------------------------------------ conv

def test_conv_one_hot_taps_shift():
    C = 6
    rng = np.random.default_rng(0)
    state = rng.standard_normal((3, C))
    xn = rng.standard_normal(C)
    window = np.concatenate([state, xn[None]], 0)
    for j in range(4):
        w = np.zeros((C, 4))
        w[:, j] = 1.0
        y, st = gdn.conv_step(state, xn, w)
        np.testing.assert_allclose(y, window[j] / (1 + np.exp(-window[j])), rtol=1e-15)
        np.testing.assert_array_equal(st, window[1:])


def test_conv_impulse_response():
    C = 3
    w = np.array([[0.1, 0.2, 0.3, 0.4], [1, -1, 2, -2], [0, 0, 0, 5]], dtype=np.float64)
    st = np.zeros((3, C))
    pres = []
    for t in range(5):
        xn = np.ones(C) if t == 0 else np.zeros(C)
        y, st = gdn.conv_step(st, xn, w)
        pres.append(y)
    # the impulse meets tap 3 at t=0, tap 2 at t=1, ..., nothing at t=4
    for t in range(5):
        pre = w[:, 3 - t] if t < 4 else np.zeros(C)
        np.testing.assert_allclose(pres[t], pre / (1 + np.exp(-pre)), rtol=1e-15)


# ------------------------------------------------------------------ norms, gates

def test_l2norm_unit_and_scale_invariant():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 128)) * 10
    n = gdn.l2norm(x, 1e-6)
    np.testing.assert_allclose(np.linalg.norm(n, axis=1), 1.0, atol=1e-7)
    np.testing.assert_allclose(gdn.l2norm(3.0 * x, 1e-6), n, rtol=1e-7)
    assert (gdn.l2norm(np.zeros((1, 8)), 1e-6) == 0).all()


def test_gates_closed_forms():
    beta, g = gdn.gates(np.array([0.0, 50.0, -50.0]), np.array([0.0, 30.0, -40.0]),
                        np.array([0.0, math.log(2), 0.0]), np.array([0.0, 0.0, 0.0]))
    np.testing.assert_allclose(beta, [0.5, 1.0, 0.0], atol=1e-20)
    np.testing.assert_allclose(g[0], -math.log(2), rtol=1e-15)       # softplus(0) = ln 2
    assert g[1] == -2 * 30.0                                           # above the threshold: identity
    np.testing.assert_allclose(g[2], -math.log1p(math.exp(-40.0)), rtol=1e-15)


def test_gated_rmsnorm_constant_o():
    c = 0.37
    o = np.full((2, 8), c)
    z = np.linspace(-3, 3, 16).reshape(2, 8)
    w = np.linspace(0.5, 1.5, 8)
    y = gdn.gated_rmsnorm(o, z, w, 1e-6)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + 1e-6) * w * z / (1 + np.exp(-z)), rtol=1e-14)


# ------------------------------------------------------------------ delta rule

def _rand_heads(rng, Hk, Hv, d):
    q = gdn.l2norm(rng.standard_normal((Hk, d)), 1e-6)
    k = gdn.l2norm(rng.standard_normal((Hk, d)), 1e-6)
    v = rng.standard_normal((Hv, d))
    S = rng.standard_normal((Hv, d, d))
    return q, k, v, S


def test_delta_g0_beta0_leaves_state_unchanged():
    rng = np.random.default_rng(2)
    q, k, v, S = _rand_heads(rng, 2, 4, 16)
    S32 = S.astype(np.float32).astype(np.float64)
    o, S2 = gdn.delta_step(S32, q, k, v, np.zeros(4), np.zeros(4))
    np.testing.assert_array_equal(S2.astype(np.float32), S32.astype(np.float32))


def test_delta_beta1_unit_key_stores_v_exactly():
    # dyadic inputs: S k = v holds exactly after the update
    rng = np.random.default_rng(3)
    Hk, Hv, d = 2, 4, 8
    S = rng.integers(-8, 8, (Hv, d, d)) / 4.0
    v = rng.integers(-8, 8, (Hv, d)) / 8.0
    k = np.zeros((Hk, d))
    k[0, 3] = 1.0
    k[1, 6] = 1.0
    q = np.ones((Hk, d)) / 4.0
    for g in (0.0, math.log(0.5)):
        o, S2 = gdn.delta_step(S, q, k, v, np.ones(Hv), np.full(Hv, g))
        for h in range(Hv):
            np.testing.assert_array_equal(S2[h] @ k[h // 2], v[h])


def test_delta_alpha0_closed_form_and_gqa_mapping():
    rng = np.random.default_rng(4)
    Hk, Hv, d = 2, 4, 16
    q, k, v, S = _rand_heads(rng, Hk, Hv, d)
    o, S2 = gdn.delta_step(S, q, k, v, np.ones(Hv), np.full(Hv, -np.inf))
    for h in range(Hv):
        kk = k[h // 2]                    # value heads 0,1 -> key head 0; 2,3 -> key head 1
        np.testing.assert_allclose(S2[h], np.outer(v[h], kk), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(o[h], v[h] * (kk @ q[h // 2]), rtol=1e-13, atol=1e-15)


def test_delta_scalar_case():
    # dk = dv = 1, k = q = 1: S' = a S + b (v - a S), o = S'
    for S0, a, b, v in [(0.5, 0.25, 0.75, 2.0), (-1.0, 1.0, 0.5, 0.0)]:
        o, S2 = gdn.delta_step(np.array([[[S0]]]), np.ones((1, 1)), np.ones((1, 1)), np.array([[v]]),
                               np.array([b]), np.array([math.log(a)]))
        want = a * S0 + b * (v - a * S0)
        assert abs(S2[0, 0, 0] - want) < 1e-15 and abs(o[0, 0] - want) < 1e-15


def test_chunked_form_equals_recurrence():
    rng = np.random.default_rng(5)
    T, d = 150, 16            # two full chunks of 64 and a ragged tail of 22
    for gscale in (0.05, 3.0, 240.0):
        q = gdn.l2norm(rng.standard_normal((T, d)), 1e-6) / math.sqrt(d)
        k = gdn.l2norm(rng.standard_normal((T, d)), 1e-6)
        v = rng.standard_normal((T, d))
        beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
        g = -gscale * rng.uniform(0, 1, T)
        S0 = rng.standard_normal((d, d)) * 0.1
        S = S0.copy()
        O = np.empty((T, d))
        for t in range(T):
            o, S4 = gdn.delta_step(S[None], q[t:t + 1], k[t:t + 1], v[t:t + 1], beta[t:t + 1], g[t:t + 1])
            S = S4[0]
            O[t] = o[0]
        Oc, Sc = gdn.chunked_delta(q, k, v, beta, g, S0)
        assert rel_l2(Oc, O) < 1e-12, gscale
        assert rel_l2(Sc, S) < 1e-12, gscale


# ------------------------------------------------------------------ whole layer

@pytest.fixture(scope="module")
def tiny():
    return gdn.Layer(synth.layer_weights(synth.TINY, 0))


def test_layer_padding_row_zero_and_state_untouched(tiny):
    sh = synth.TINY
    x = synth.x_tokens(sh, 0, 3)
    cs = np.stack([synth.conv_state(sh, 100 + s) for s in range(2)])
    ss = np.stack([synth.ssm_state(sh, 100 + s) for s in range(2)])
    cs0, ss0 = cs.copy(), ss.copy()
    out = tiny.decode_step(x, [-1, 1, -1], cs, ss)
    assert (out[0] == 0).all() and (out[2] == 0).all() and (out[1] != 0).any()
    np.testing.assert_array_equal(cs[0], cs0[0])
    np.testing.assert_array_equal(ss[0], ss0[0])
    assert (cs[1] != cs0[1]).any() and (ss[1] != ss0[1]).any()


def test_layer_batch_rows_equal_single_rows(tiny):
    sh = synth.TINY
    x = np.stack([synth.x_tokens(sh, 100 + s, 1)[0] for s in range(3)])
    cs = np.stack([synth.conv_state(sh, 100 + s) for s in range(3)])
    ss = np.stack([synth.ssm_state(sh, 100 + s) for s in range(3)])
    csb, ssb = cs.copy(), ss.copy()
    outb = tiny.decode_step(x, [0, 1, 2], csb, ssb)
    for s in range(3):
        c1, s1 = cs.copy(), ss.copy()
        o1 = tiny.decode_step(x[s:s + 1], [s], c1, s1)
        np.testing.assert_array_equal(o1[0], outb[s])
        np.testing.assert_array_equal(s1[s], ssb[s])


def test_prefill_is_decode_and_continues(tiny):
    sh = synth.TINY
    x = synth.x_tokens(sh, 7, 10)
    # T = 1 prefill equals one decode step
    c1, s1 = synth.conv_state(sh, 0, True), synth.ssm_state(sh, 0, True)
    o1 = tiny.prefill(x[:1], c1, s1, init_zero=True)
    c2, s2 = synth.conv_state(sh, 0, True)[None].copy(), synth.ssm_state(sh, 0, True)[None].copy()
    o2 = tiny.decode_step(x[:1], [0], c2, s2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2[0])
    # prefill(4) then prefill(6, continuing) equals prefill(10)
    ca, sa = synth.conv_state(sh, 0, True), synth.ssm_state(sh, 0, True)
    oa = np.concatenate([tiny.prefill(x[:4], ca, sa, True), tiny.prefill(x[4:], ca, sa, False)])
    cb, sb = synth.conv_state(sh, 0, True), synth.ssm_state(sh, 0, True)
    ob = tiny.prefill(x, cb, sb, True)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(sa, sb)
    np.testing.assert_array_equal(ca, cb)


def test_layer_stage_extras_consistent(tiny):
    # the mix stage's intermediates obey the stage definitions
    sh = synth.TINY
    x = synth.x_tokens(sh, 0, 1)
    qkvz, ba = tiny.projections(x)
    y, cst, S, ex = tiny.mix(qkvz[0], ba[0], synth.conv_state(sh, 1), synth.ssm_state(sh, 1))
    np.testing.assert_allclose(np.linalg.norm(ex["k_hat"], axis=1), 1.0, atol=1e-6)
    np.testing.assert_allclose(np.linalg.norm(ex["q_hat"], axis=1), 1 / math.sqrt(sh.d_k), atol=1e-6)
    assert (ex["g"] <= 0).all() and ((ex["beta"] > 0) & (ex["beta"] < 1)).all()
    # conv state holds the raw BF16 projection inputs, newest last
    nqkv = 2 * sh.n_k_heads * sh.d_k + sh.n_v_heads * sh.d_v
    np.testing.assert_array_equal(codecs.bf16_to_f32(cst[-1]), qkvz[0, :nqkv].astype(np.float32))


# ------------------------------------------------------------------ BF16-stored state

def _bf16_state(sh, seed):
    """A recurrent state whose values are BF16-representable (float32 array)."""
    s = synth.ssm_state(sh, seed)
    return codecs.bf16_to_f32(codecs.f32_to_bf16(s))


def test_bf16_state_decode_rounds_the_updated_state_once():
    """A decode step of the BF16-state layer equals the FP32-state layer's step
    from the same state, with the updated state rounded FP32 -> BF16 (nearest
    even): the outputs are identical and the state is rounded after the
    update, not before it or inside it."""
    sh = synth.TINY
    w = synth.layer_weights(sh, 0)
    L32, L16 = gdn.Layer(w), gdn.Layer(w, state_bf16=True)
    x = synth.x_tokens(sh, 3, 2)
    c0 = synth.conv_state(sh, 3)[None]
    s0 = _bf16_state(sh, 3)[None]
    ca, sa, cb, sb = c0.copy(), s0.copy(), c0.copy(), s0.copy()
    out32 = L32.decode_step(x[0:1], [0], ca, sa)
    out16 = L16.decode_step(x[0:1], [0], cb, sb)
    np.testing.assert_array_equal(out32, out16)
    np.testing.assert_array_equal(ca, cb)
    np.testing.assert_array_equal(sb, codecs.bf16_to_f32(codecs.f32_to_bf16(sa)))
    assert (sb != sa).any()                      # the rounding did something
    # every stored value is BF16: its low 16 bits are zero
    assert not (sb.view(np.uint32) & 0xFFFF).any()


def test_bf16_state_identity_update_leaves_state_bit_unchanged():
    """beta = 0 and g = 0 (A_log = -inf, b -> -inf): the update is the identity,
    so a BF16 state comes back bit-identical."""
    sh = synth.TINY
    w = synth.layer_weights(sh, 0)
    w.A_log[:] = -np.inf
    L16 = gdn.Layer(w, state_bf16=True)
    qkvz = codecs.bf16_to_f32(synth.bf16_normal(1, sh.qkvz_out, 5)[0]).astype(np.float64)
    ba = np.concatenate([np.full(sh.n_v_heads, -1e4), np.zeros(sh.n_v_heads)])
    s0 = _bf16_state(sh, 4)
    with np.errstate(over="ignore"):                 # sigmoid(-1e4) = 1/(1+inf) = 0
        _, _, s1, ex = L16.mix(qkvz, ba, synth.conv_state(sh, 4), s0)
    assert (ex["beta"] == 0).all() and (ex["g"] == 0).all()
    np.testing.assert_array_equal(s1, s0)


def test_bf16_state_prefill_carries_fp32_and_rounds_at_the_end():
    """A prefill call of the BF16-state layer: the FP32 layer's prefill from the
    same state, the final state rounded once to BF16; outputs identical."""
    sh = synth.TINY
    w = synth.layer_weights(sh, 0)
    L32, L16 = gdn.Layer(w), gdn.Layer(w, state_bf16=True)
    x = synth.x_tokens(sh, 6, 20)
    c0, s0 = synth.conv_state(sh, 6), _bf16_state(sh, 6)
    ca, sa, cb, sb = c0.copy(), s0.copy(), c0.copy(), s0.copy()
    o32 = L32.prefill(x, ca, sa, init_zero=False)
    o16 = L16.prefill(x, cb, sb, init_zero=False)
    np.testing.assert_array_equal(o32, o16)
    np.testing.assert_array_equal(sb, codecs.bf16_to_f32(codecs.f32_to_bf16(sa)))
    # and differs from rounding after every token (the decode-step semantics)
    cc, sc = c0.copy(), s0.copy()
    for t in range(20):
        L16.decode_step(x[t:t + 1], [0], cc[None], sc[None])
    assert rel_l2(sc, sb) > 0


# ------------------------------------------------------------------ verify / commit

def test_verify_then_commit_equals_decode_steps(tiny):
    """r candidate tokens through verify, then commit of n of them: the outputs
    are the first decode steps' outputs and the slot ends as after n decode
    steps; n = 0 leaves the slot as it was; a padding row reads zero."""
    sh = synth.TINY
    r = 3
    slots = [0, -1, 1]
    x = np.stack([synth.x_tokens(sh, 40 + b, r) for b in range(3)])          # [B][r][H]
    conv0 = np.stack([synth.conv_state(sh, 100 + s) for s in range(2)])
    ssm0 = np.stack([synth.ssm_state(sh, 100 + s) for s in range(2)])
    c, s = conv0.copy(), ssm0.copy()
    out, snaps = tiny.verify(x, slots, c, s)
    np.testing.assert_array_equal(c, conv0)                                  # slots untouched
    np.testing.assert_array_equal(s, ssm0)
    assert not out[1].any() and snaps[1] is None
    # decode reference: rows 0 and 2 stepped r times
    cd, sd = conv0.copy(), ssm0.copy()
    dec = [tiny.decode_step(x[[0, 2], t], [0, 1], cd, sd) for t in range(r)]
    for t in range(r):
        np.testing.assert_array_equal(out[0, t], dec[t][0])
        np.testing.assert_array_equal(out[2, t], dec[t][1])
    # commit 0 tokens for slot 0 and 2 tokens for slot 1
    gdn.Layer.verify_commit(slots, [0, 0, 2], snaps, c, s)
    np.testing.assert_array_equal(s[0], ssm0[0])
    c2, s2 = conv0.copy(), ssm0.copy()
    for t in range(2):
        tiny.decode_step(x[[0, 2], t], [-1, 1], c2, s2)
    np.testing.assert_array_equal(s[1], s2[1])
    np.testing.assert_array_equal(c[1], c2[1])
    # commit all r for slot 0
    gdn.Layer.verify_commit(slots, [r, 0, 0], snaps, c, s)
    np.testing.assert_array_equal(s[0], sd[0])
    np.testing.assert_array_equal(c[0], cd[0])
