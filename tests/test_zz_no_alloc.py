"""gdn_decode_step_static -- the decode step for callers that cannot allocate
device memory or keep a context -- gives the same results as gdn_decode_step.

Both entry points are called through the C ABI on the same weights and the
same inputs, two steps in a row, for one, two and four rows. The static entry
point keeps its intermediates in a fixed device array shared by all its calls,
so the second call also checks that nothing left behind by the first one leaks
into it. The first step is also compared with the oracle, and the calls after
the first must leave the device's allocated and free memory unchanged. This
file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from conftest import rel_l2
from helpers import oracle_layer, slot_inputs, to_dev, to_host, weights
from nvfp4_gated_deltanet_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _bf(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("B", [1, 2, 4])
def test_static_step_matches_context_step(B):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import nvfp4_gated_deltanet_gb300 as pkg
    w = weights("FULL", 1)
    sh = w.shape
    # device copies of the weights, kept alive for the static entry point
    dev = {"qkvz": (to_dev(w.qkvz.codes), to_dev(w.qkvz.scales)), "ba": (to_dev(w.ba.codes), to_dev(w.ba.scales)),
           "out": (to_dev(w.out.codes), to_dev(w.out.scales)), "conv_w": to_dev(w.conv_w),
           "A_log": to_dev(w.A_log), "dt_bias": to_dev(w.dt_bias), "norm_w": to_dev(w.norm_w)}
    nv = lambda k, m: pkg.GdnNVFP4(dev[k][0].data_ptr(), dev[k][1].data_ptr(), float(m.tensor_scale))
    gw = pkg.GdnWeights(nv("qkvz", w.qkvz), nv("ba", w.ba), nv("out", w.out), dev["conv_w"].data_ptr(),
                        dev["A_log"].data_ptr(), dev["dt_bias"].data_ptr(), dev["norm_w"].data_ptr())
    cfg = pkg.GdnConfig(sh.hidden, sh.n_k_heads, sh.n_v_heads, sh.d_k, sh.d_v, sh.conv_kernel, 16, 0, w.rms_eps,
                        w.l2_eps, w.act_scale_in, w.act_scale_out)
    layer = pkg.layer_from_synth(w, max_batch=16)

    slots = list(range(B))
    x, conv0, ssm0 = slot_inputs(sh, slots, 2)
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    conv_a, ssm_a = to_dev(conv0), to_dev(ssm0)   # context path
    conv_b, ssm_b = to_dev(conv0), to_dev(ssm0)   # static path
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    L = pkg.lib()
    xs = [to_dev(x[step]) for step in range(2)]
    outs = [torch.empty(B, sh.hidden, dtype=torch.int16, device="cuda") for _ in range(2)]
    conv_o, ssm_o = conv0.copy(), ssm0.copy()     # the oracle's first step
    want0 = oracle_layer("FULL", 1).decode_step(x[0], slots, conv_o, ssm_o)
    mem = None
    for step in range(2):                          # two calls in a row
        want = layer.decode_step(xs[step], ids, conv_a, ssm_a)
        got = outs[step]
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        st = L.gdn_decode_step_static(ctypes.byref(cfg), ctypes.byref(gw), xs[step].data_ptr(), ids.data_ptr(), B,
                                      got.data_ptr(), conv_b.data_ptr(), ssm_b.data_ptr(), B, status.data_ptr(),
                                      stream)
        assert st == 0, pkg.STATUS_NAMES[st]
        torch.cuda.synchronize()
        after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        if step > 0:                               # the first call may set up the array's address
            assert after == before, (before, after)
        assert int(status.item()) == 0
        assert rel_l2(_bf(to_host(got)), _bf(to_host(want))) <= 4e-3
        assert rel_l2(to_host(ssm_b), to_host(ssm_a)) <= 1e-4
        assert rel_l2(_bf(to_host(conv_b)), _bf(to_host(conv_a))) <= 4e-3
        if step == 0:                              # against the oracle, on its own
            assert rel_l2(_bf(to_host(got)), _bf(want0)) <= 4e-3
            assert rel_l2(to_host(ssm_b), ssm_o) <= 1e-4
    assert layer.check() == 0


def test_static_step_refuses_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import nvfp4_gated_deltanet_gb300 as pkg
    good = 0x10000  # never dereferenced: the size check fails first
    A = pkg.GdnNVFP4(good, good, 1.0)
    gw = pkg.GdnWeights(A, A, A, good, good, good, good)
    for field, val in [("hidden", 4096), ("n_v_heads", 64)]:
        cfg = pkg.GdnConfig(2048, 16, 32, 128, 128, 4, 16, 0, 1e-6, 1e-6, 2 ** -8, 2 ** -4)
        setattr(cfg, field, val)
        assert pkg.lib().gdn_decode_step_static(ctypes.byref(cfg), ctypes.byref(gw), good, good, 1, good, good, good,
                                                1, None, None) == 2
    cfg = pkg.GdnConfig(2048, 16, 32, 128, 128, 4, 16, 0, 1e-6, 1e-6, 2 ** -8, 2 ** -4)
    assert pkg.lib().gdn_decode_step_static(ctypes.byref(cfg), ctypes.byref(gw), good, good, 17, good, good, good,
                                            17, None, None) == 2
