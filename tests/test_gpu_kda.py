"""KDA-style recurrent step (per-channel gated delta rule) against the oracle:
o rel-L2 <= 1e-5 and state rel-L2 <= 1e-5 with an FP32 state; with a BF16
state, from the same BF16 values, o and the state rel-L2 <= 4e-3 (the KDA
entry's tolerances for BF16 storage: a BF16 half-ulp with slack, since a
one-ulp difference in one step's stored state carries into the next). Shapes: the pages' 64 heads x 128 at M = 1 and 8, ragged small
heads, several steps in a row."""
import numpy as np
import pytest

from conftest import rel_l2
from helpers import to_dev, to_host
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def api():
    import nvfp4_gated_deltanet_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return pkg


@pytest.mark.parametrize("M,H,D,steps", [(1, 64, 128, 3), (8, 64, 128, 2), (3, 5, 64, 4), (2, 7, 32, 4)])
@pytest.mark.parametrize("bf16", [False, True])
def test_kda_step_matches_oracle(api, M, H, D, steps, bf16):
    from oracle import codecs, kda
    q, k, v, g, beta, S = synth.kda_inputs(M, H, D, 11)
    if bf16:
        S = codecs.bf16_to_f32(codecs.f32_to_bf16(S))
    Sd = to_dev(codecs.f32_to_bf16(S)) if bf16 else to_dev(S)
    Sref = S.copy()
    for t in range(steps):
        # new inputs each step (same generator, shifted seed)
        q, k, v, g, beta, _ = synth.kda_inputs(M, H, D, 11 + t)
        o = to_host(api.kda_step(to_dev(q), to_dev(k), to_dev(v), to_dev(g), to_dev(beta), Sd))
        o_ref, Sref = kda.kda_step(q, k, v, g, beta, Sref, "bf16" if bf16 else "f32")
        assert rel_l2(o, o_ref) <= (4e-3 if bf16 else 1e-5)
    got = codecs.bf16_to_f32(to_host(Sd)) if bf16 else to_host(Sd)
    assert rel_l2(got, Sref) <= (4e-3 if bf16 else 1e-5)


def test_kda_step_refuses_bad_shapes(api):
    z = torch.zeros(1, 1, 48, dtype=torch.float32, device="cuda")
    with pytest.raises(api.GdnError):
        api.kda_step(z, z, z, z, torch.zeros(1, 1, device="cuda"), torch.zeros(1, 1, 48, 48, device="cuda"))
