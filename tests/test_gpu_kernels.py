"""GPU parity of the standalone entry points: the NVFP4 quantiser (bit-exact)
and the W4A4 product (FP32 rel-L2 <= 1e-5) against the oracle."""
import numpy as np
import pytest

from conftest import rel_l2
from helpers import to_dev, to_host
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def g():
    import nvfp4_gated_deltanet_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return pkg


def _oracle_q(x32, ts):
    from oracle import nvfp4
    return nvfp4.quantize(x32, ts)


@pytest.mark.parametrize("rows,cols,ts", [(1, 2048, 2.0 ** -8), (64, 2048, 2.0 ** -8), (37, 4096, 2.0 ** -4),
                                          (3, 16, 1.0)])
def test_quantize_bf16_bit_exact(g, rows, cols, ts):
    from oracle import codecs
    xb = synth.bf16_normal(rows, cols, seed=rows * 7 + cols, std=1.0)
    codes, scales = g.nvfp4_quantize(to_dev(xb), ts)
    oc, os_ = _oracle_q(codecs.bf16_to_f32(xb), ts)
    np.testing.assert_array_equal(to_host(scales), os_)
    np.testing.assert_array_equal(to_host(codes), oc)


def test_quantize_f32_edge_cases_bit_exact(g):
    rng = np.random.default_rng(0)
    # wide dynamic range (subnormal, normal and saturating E4M3 scales), signed zeros,
    # E2M1 ties at every grid midpoint, and blocks from the hand-worked fixture
    ts = 2.0 ** -8
    mags = np.exp2(rng.uniform(-40, 12, (512, 16)))
    sign = np.where(rng.uniform(size=(512, 16)) < 0.5, -1.0, 1.0)
    wide = (mags * sign).astype(np.float32)
    ties = np.zeros((8, 16), np.float32)
    mid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    for i in range(8):                          # amax 6 -> scale 1 * ts * 2^k, x*r lands on midpoints
        ties[i, :8] = mid * 2.0 ** (i - 4) * 6 * ts / 6
        ties[i, 8:] = -ties[i, :8]
        ties[i, 15] = 6 * ts * 2.0 ** (i - 4)
    zeros = np.zeros((2, 16), np.float32)
    zeros[1] = -0.0
    zeros[1, 3] = -1e-30
    x = np.concatenate([wide, ties, zeros]).astype(np.float32)
    codes, scales = g.nvfp4_quantize(to_dev(x), ts)
    oc, os_ = _oracle_q(x, ts)
    np.testing.assert_array_equal(to_host(scales), os_)
    np.testing.assert_array_equal(to_host(codes), oc)


def test_quantize_nonfinite_flags_status(g):
    x = np.ones((4, 32), np.float32)
    x[1, 3] = np.nan
    x[2, 20] = np.inf
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales = g.nvfp4_quantize(to_dev(x), 1.0, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 4                      # GDN_E_NONFINITE
    s = to_host(scales)
    assert s[1, 0] == 0 and s[2, 1] == 0 and s[0, 0] != 0 and s[1, 1] != 0
    assert (to_host(codes)[1, :8] == 0).all()


# K % 256 == 0 runs on the tcgen05 block-scaled kernel (N-tile 16/32/64/128, split-K
# clusters, ragged M and N); other K on the CUDA-core kernel.
@pytest.mark.parametrize("M,N,K", [(1, 384, 256), (5, 100, 128), (16, 2048, 4096), (33, 64, 64), (2, 12352, 2048),
                                   (128, 256, 256), (200, 384, 512), (64, 1024, 2048), (40, 300, 256),
                                   (256, 12352, 2048), (3, 2048, 4096)])
def test_gemm_fp32_matches_exact_product(g, M, N, K):
    from oracle import nvfp4
    a = synth.nvfp4_random(M, K, seed=M + 1000, prefix="mat", tensor_scale=2.0 ** -8)
    b = synth.nvfp4_random(N, K, seed=N + 2000, prefix="mat", tensor_scale=2.0 ** -6)
    want = nvfp4.gemm(a.codes, a.scales, a.tensor_scale, b.codes, b.scales, b.tensor_scale)
    got = g.nvfp4_gemm(to_dev(a.codes), to_dev(a.scales), a.tensor_scale, to_dev(b.codes), to_dev(b.scales),
                       b.tensor_scale, out_dtype=torch.float32)
    assert rel_l2(to_host(got), want) <= 1e-5
    gotb = g.nvfp4_gemm(to_dev(a.codes), to_dev(a.scales), a.tensor_scale, to_dev(b.codes), to_dev(b.scales),
                        b.tensor_scale, out_dtype=torch.bfloat16)
    gb = gotb.float().cpu().numpy()
    assert rel_l2(gb, want) <= 4e-3


def test_gemm_zero_rows_give_exact_zero(g):
    b = synth.nvfp4_random(64, 128, seed=5)
    a_codes = torch.zeros(3, 64, dtype=torch.uint8, device="cuda")
    a_scales = torch.zeros(3, 8, dtype=torch.uint8, device="cuda")
    got = g.nvfp4_gemm(a_codes, a_scales, 1.0, to_dev(b.codes), to_dev(b.scales), b.tensor_scale,
                       out_dtype=torch.float32)
    assert (got == 0).all()
