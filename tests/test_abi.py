"""The C-ABI library loads, exports every function include/gdn.h declares, and
refuses bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def L():
    from nvfp4_gated_deltanet_gb300 import build
    build.build()
    import nvfp4_gated_deltanet_gb300 as g
    return g.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["gdn_create", "gdn_destroy", "nvfp4_quantize", "nvfp4_gemm", "gdn_decode_step", "gdn_prefill",
              "gdn_mix_step", "gdn_check", "gdn_status_string"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(L):
    import nvfp4_gated_deltanet_gb300 as g
    for n in declared_functions():
        assert hasattr(L, n), n
        assert n in g.SIGNATURES, f"binding lacks {n}"


def test_status_strings(L):
    assert L.gdn_status_string(0) == b"GDN_OK"
    assert L.gdn_status_string(2) == b"GDN_E_SHAPE"
    assert L.gdn_status_string(99) == b"GDN_E_UNKNOWN"


def test_host_refusals_before_any_launch(L):
    import nvfp4_gated_deltanet_gb300 as g
    good = 0x10000  # never dereferenced: every call below fails validation first
    # quantiser
    assert L.nvfp4_quantize(good, 0, 4, 24, 1.0, good, good, None, None) == 2          # cols % 16
    assert L.nvfp4_quantize(None, 0, 4, 32, 1.0, good, good, None, None) == 1          # NULL x
    assert L.nvfp4_quantize(good + 2, 0, 4, 32, 1.0, good, good, None, None) == 3      # misaligned
    assert L.nvfp4_quantize(good, 0, 4, 32, float("nan"), good, good, None, None) == 4
    assert L.nvfp4_quantize(good, 0, 4, 32, -1.0, good, good, None, None) == 5
    assert L.nvfp4_quantize(None, 0, 0, 32, 1.0, None, None, None, None) == 0          # empty is a no-op
    # gemm
    A = g.GdnNVFP4(good, good, 1.0)
    B = g.GdnNVFP4(good, good, 1.0)
    assert L.nvfp4_gemm(ctypes.byref(A), 4, ctypes.byref(B), 4, 48, good, 1, None) == 2   # K % 64
    assert L.nvfp4_gemm(ctypes.byref(A), 0, ctypes.byref(B), 4, 64, None, 1, None) == 0   # M = 0
    Bz = g.GdnNVFP4(good, good, 0.0)
    assert L.nvfp4_gemm(ctypes.byref(A), 4, ctypes.byref(Bz), 4, 64, good, 1, None) == 5
    Bn = g.GdnNVFP4(None, good, 1.0)
    assert L.nvfp4_gemm(ctypes.byref(A), 4, ctypes.byref(Bn), 4, 64, good, 1, None) == 1
    # context
    out = ctypes.c_void_p()
    assert L.gdn_create(None, None, None, ctypes.byref(out)) == 1
    cfg = g.GdnConfig(2048, 16, 32, 128, 128, 4, 16, 0, 1e-6, 1e-6, 2 ** -8, 2 ** -4)
    w = g.GdnWeights(A, A, A, good, good, good, good)
    for field, val, code in [("d_k", 48, 2), ("conv_kernel", 7, 2), ("max_batch", 0, 2), ("hidden", 100, 2),
                             ("n_v_heads", 24, 2), ("rms_eps", float("inf"), 4), ("act_scale_in", 0.0, 5)]:
        bad = g.GdnConfig.from_buffer_copy(cfg)
        setattr(bad, field, val)
        if field == "d_k":
            bad.d_v = val
        assert L.gdn_create(ctypes.byref(bad), ctypes.byref(w), None, ctypes.byref(out)) == code, field
        assert out.value is None
    wn = g.GdnWeights(A, A, A, None, good, good, good)
    assert L.gdn_create(ctypes.byref(cfg), ctypes.byref(wn), None, ctypes.byref(out)) == 1
    wa = g.GdnWeights(A, g.GdnNVFP4(good + 8, good, 1.0), A, good, good, good, good)
    assert L.gdn_create(ctypes.byref(cfg), ctypes.byref(wa), None, ctypes.byref(out)) == 3
    # calls on a NULL context
    assert L.gdn_decode_step(None, good, good, 1, good, good, good, 1, None) == 1
    assert L.gdn_prefill(None, good, 8, 0, 1, good, good, good, 1, None) == 1
    assert L.gdn_mix_step(None, good, good, good, 1, good, good, good, 1, None) == 1
    assert L.gdn_check(None, 0, None) == 1
    assert L.gdn_destroy(None) == 0


def test_python_binding_raises_without_library(tmp_path, monkeypatch):
    import nvfp4_gated_deltanet_gb300 as g
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        g.lib()


def test_tuning_knob_ranges(L):
    """Every knob takes its documented values and refuses the rest (GDN_E_RANGE
    = 6); each is put back to its default (0) afterwards."""
    valid = {0: (0, 1, 2), 1: (0, 1, 2, 4, 8), 2: (0, 1, 2, 4, 8), 3: (0, 1, 2), 4: (0, 1, 2), 5: (0, 1, 2),
             6: (0, 1, 2), 7: (0, 1, 2, 4), 8: (0, 1, 2), 9: (0, 1, 2), 10: (0, 1, 2, 3), 11: (0, 1, 2, 3),
             13: (0, 1, 2), 14: (0, 1, 2, 3), 15: (0, 1, 2, 3), 16: (0, 1, 2)}
    try:
        for knob, values in valid.items():
            for v in range(-1, 10):
                assert L.gdn_set_tuning(knob, v) == (0 if v in values else 6), (knob, v)
        for v in (0, 1, 1000, 2 ** 31 - 1):                    # knob 12: a wait budget in cycles
            assert L.gdn_set_tuning(12, v) == 0, v
        assert L.gdn_set_tuning(12, -1) == 6
        assert L.gdn_set_tuning(17, 0) == 6
        assert L.gdn_set_tuning(-1, 0) == 6
    finally:
        for knob in list(valid) + [12]:
            L.gdn_set_tuning(knob, 0)
