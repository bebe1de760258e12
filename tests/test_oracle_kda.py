"""Pins of the oracle's KDA-style recurrent step (per-channel gated delta rule)."""
import numpy as np

from nvfp4_gated_deltanet_gb300 import synth
from oracle import codecs, gdn, kda


def test_equal_channel_decays_reduce_to_the_gdn_delta_rule():
    """With one log-decay shared by every key channel the step is the GDN delta
    rule (gdn.delta_step, pinned on its own)."""
    M, H, D = 2, 3, 8
    q, k, v, g, beta, S = synth.kda_inputs(M, H, D, 1)
    gs = g[:, :, :1]                                     # one decay per head
    o, Sn = kda.kda_step(q, k, v, np.broadcast_to(gs, g.shape), beta, S)
    for m in range(M):
        o_ref, S_ref = gdn.delta_step(S[m].astype(np.float64), q[m].astype(np.float64), k[m].astype(np.float64),
                                      v[m].astype(np.float64), beta[m].astype(np.float64),
                                      gs[m, :, 0].astype(np.float64))
        np.testing.assert_allclose(o[m], o_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(Sn[m], S_ref.astype(np.float32), rtol=1e-7, atol=1e-9)


def test_beta_zero_is_a_pure_per_channel_decay():
    M, H, D = 1, 2, 8
    q, k, v, g, beta, S = synth.kda_inputs(M, H, D, 2)
    o, Sn = kda.kda_step(q, k, v, g, np.zeros_like(beta), S)
    want = (S.astype(np.float64) * np.exp(g.astype(np.float64))[:, :, None, :])
    np.testing.assert_array_equal(Sn, want.astype(np.float32))
    np.testing.assert_allclose(o, np.einsum("mhvk,mhk->mhv", want, q.astype(np.float64)), rtol=1e-12)


def test_unit_key_no_decay_stores_v():
    """beta = 1, k = e_j, g = 0: afterwards S k = v (exactly, dyadic inputs)."""
    D = 8
    S = np.full((1, 1, D, D), 0.25, np.float32)
    k = np.zeros((1, 1, D), np.float32)
    k[0, 0, 3] = 1.0
    v = (np.arange(D, dtype=np.float32) - 2.5)[None, None]
    _, Sn = kda.kda_step(np.zeros_like(k), k, v, np.zeros_like(k), np.ones((1, 1), np.float32), S)
    np.testing.assert_array_equal(Sn[0, 0] @ k[0, 0], v[0, 0])


def test_matches_the_transition_matrix_form():
    """The same step written as the KDA paper's transition on P = S^T:
    P' = (I - beta k k^T) diag(alpha) P + beta k v^T, o = P'^T q."""
    M, H, D = 1, 2, 6
    q, k, v, g, beta, S = synth.kda_inputs(M, H, D, 3)
    o, Sn = kda.kda_step(q, k, v, g, beta, S)
    for h in range(H):
        kk = k[0, h].astype(np.float64)
        P = S[0, h].astype(np.float64).T
        A = np.eye(D) - beta[0, h] * np.outer(kk, kk)
        Pn = A @ np.diag(np.exp(g[0, h].astype(np.float64))) @ P + beta[0, h] * np.outer(kk, v[0, h])
        np.testing.assert_allclose(Sn[0, h], Pn.T.astype(np.float32), rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(o[0, h], Pn.T @ q[0, h].astype(np.float64), rtol=1e-10, atol=1e-12)


def test_bf16_store_rounds_the_fp32_result():
    q, k, v, g, beta, S = synth.kda_inputs(1, 2, 8, 4)
    _, S32 = kda.kda_step(q, k, v, g, beta, S)
    _, S16 = kda.kda_step(q, k, v, g, beta, S, "bf16")
    np.testing.assert_array_equal(S16, codecs.bf16_to_f32(codecs.f32_to_bf16(S32)))
