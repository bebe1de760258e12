"""The gate extremes of the gated delta rule, driven through the GPU's token
mixing (gdn_mix_step: conv, norms, gates, delta rule, gated norm) and checked
against the oracle and against closed forms of the definition.

The mixing stage takes the BF16 projections directly, so b and a can be set to
values that put the gates at their limits (value heads h, cycling):
  h % 4 == 0  b = a = -1e4:   beta = 0, alpha = 1  -> the state is bit-unchanged
  h % 4 == 1  b = +1e4, a = -1e4: beta = 1, alpha = 1 with a unit key k = e_j
              -> after the update S k = v (the stored value is read back)
  h % 4 == 2  b = a = +1e4:   beta = 1, alpha = 0  -> S = v k^T exactly
  h % 4 == 3  ordinary gates, and A_log = -inf for two of them (alpha = 1)
The keys are made one-hot by the conv: zero conv state on the k channels and
one large input per key head through the newest tap, so SiLU leaves exactly
one non-zero channel."""
import dataclasses

import numpy as np
import pytest

from conftest import rel_l2
from helpers import to_dev, to_host, weights
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    import nvfp4_gated_deltanet_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return pkg


def _case(B):
    from oracle import codecs
    sh = synth.FULL
    D, Hk, Hv = sh.d_k, sh.n_k_heads, sh.n_v_heads
    w = weights("FULL", 1)
    A_log = w.A_log.copy()
    A_log[[3, 7]] = -np.inf
    w = dataclasses.replace(w, A_log=A_log)
    conv_w = codecs.bf16_to_f32(w.conv_w)
    r = np.random.default_rng(11)
    qkvz = r.standard_normal((B, sh.qkvz_out)).astype(np.float32)
    conv = np.stack([synth.conv_state(sh, 200 + b) for b in range(B)])
    onehot = [(7 * kh + 3) % D for kh in range(Hk)]
    for kh in range(Hk):
        ch = slice(Hk * D + kh * D, Hk * D + (kh + 1) * D)
        qkvz[:, ch] = 0.0
        j = Hk * D + kh * D + onehot[kh]
        qkvz[:, j] = 8.0 * np.sign(conv_w[j, sh.conv_kernel - 1])   # SiLU(w * 8 * sign w) > 0
        conv[:, :, ch] = 0
    ba = r.standard_normal((B, 2 * Hv)).astype(np.float32)
    for h in range(Hv):
        if h % 4 == 0:
            ba[:, h], ba[:, Hv + h] = -1e4, -1e4
        elif h % 4 == 1:
            ba[:, h], ba[:, Hv + h] = 1e4, -1e4
        elif h % 4 == 2:
            ba[:, h], ba[:, Hv + h] = 1e4, 1e4
    ssm = np.stack([synth.ssm_state(sh, 200 + b) for b in range(B)])
    return w, codecs.f32_to_bf16(qkvz), codecs.f32_to_bf16(ba), conv, ssm, onehot


@pytest.mark.filterwarnings("ignore:overflow encountered in exp")   # the oracle's sigmoid(-1e4) = 0
@pytest.mark.parametrize("B", [1, 3])
def test_gate_extremes_match_oracle_and_closed_forms(api, B):
    from oracle import codecs, gdn
    w, qkvz_bits, ba_bits, conv0, ssm0, onehot = _case(B)
    sh = w.shape
    D, Hv, G = sh.d_k, sh.n_v_heads, sh.n_v_heads // sh.n_k_heads
    layer = api.layer_from_synth(w, max_batch=16)
    conv_d, ssm_d = to_dev(conv0), to_dev(ssm0)
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    y = to_host(layer.mix_step(to_dev(qkvz_bits), to_dev(ba_bits), ids, conv_d, ssm_d))
    assert layer.check() == 0
    S_gpu, conv_gpu = to_host(ssm_d), to_host(conv_d)
    O = gdn.Layer(w)
    for b in range(B):
        yw, cw, sw, ex = O.mix(codecs.bf16_to_f32(qkvz_bits[b]).astype(np.float64),
                               codecs.bf16_to_f32(ba_bits[b]).astype(np.float64), conv0[b], ssm0[b])
        assert rel_l2(y[b], yw) <= 1e-5
        assert rel_l2(S_gpu[b], sw) <= 1e-5
        np.testing.assert_array_equal(conv_gpu[b], cw)
        assert np.all(ex["beta"][0::4] == 0.0) and np.all(ex["beta"][1::4] == 1.0)
        for h in range(Hv):
            kh = h // G
            j = onehot[kh]
            v = ex["v"][h]
            if h % 4 == 0:          # beta = 0, alpha = 1: untouched, bit for bit
                np.testing.assert_array_equal(S_gpu[b, h], ssm0[b, h])
            elif h % 4 == 1:        # beta = 1, alpha = 1, unit key: S k = v
                np.testing.assert_allclose(S_gpu[b, h][:, j], v, rtol=1e-5, atol=1e-6)
            elif h % 4 == 2:        # beta = 1, alpha = 0: S = v k^T, zero off the key's column
                assert np.all(np.delete(S_gpu[b, h], j, axis=1) == 0.0)
                np.testing.assert_allclose(S_gpu[b, h][:, j], v * ex["k_hat"][kh][j], rtol=1e-6, atol=1e-7)
        # A_log = -inf: g = 0, alpha = 1 (the decay leaves S as it was before the delta)
        assert ex["g"][3] == 0.0 and ex["g"][7] == 0.0
