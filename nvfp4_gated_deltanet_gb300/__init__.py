"""NVFP4 W4A4 Gated DeltaNet layer step for GB300 (sm_103a).

A thin ctypes binding over ``libgdn.so`` (C ABI in ``include/gdn.h``): argument
marshalling only. Every step of the layer runs in the library's CUDA kernels;
PyTorch supplies device memory and streams. There is no CPU fallback: if the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_OK = 0
STATUS_NAMES = ["GDN_OK", "GDN_E_NULL", "GDN_E_SHAPE", "GDN_E_ALIGN", "GDN_E_NONFINITE", "GDN_E_BAD_SCALE",
                "GDN_E_RANGE", "GDN_E_OVERFLOW", "GDN_E_CUDA", "GDN_E_OOM", "GDN_E_TIMEOUT", "GDN_E_STATE"]

# Every entry point the header declares, with its ctypes signature.
_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


class GdnConfig(ctypes.Structure):
    _fields_ = [("hidden", _i), ("n_k_heads", _i), ("n_v_heads", _i), ("d_k", _i), ("d_v", _i),
                ("conv_kernel", _i), ("max_batch", _i), ("max_prefill_tokens", _i),
                ("rms_eps", _f), ("l2_eps", _f), ("act_scale_in", _f), ("act_scale_out", _f),
                ("state_bf16", _i)]


class GdnNVFP4(ctypes.Structure):
    _fields_ = [("codes", _vp), ("scales", _vp), ("tensor_scale", _f)]


class GdnWeights(ctypes.Structure):
    _fields_ = [("qkvz", GdnNVFP4), ("ba", GdnNVFP4), ("out", GdnNVFP4), ("conv_w", _vp),
                ("A_log", _vp), ("dt_bias", _vp), ("norm_w", _vp)]


SIGNATURES = {
    "gdn_status_string": (ctypes.c_char_p, [_i]),
    "gdn_create": (_i, [ctypes.POINTER(GdnConfig), ctypes.POINTER(GdnWeights), _vp, ctypes.POINTER(_vp)]),
    "gdn_destroy": (_i, [_vp]),
    "nvfp4_quantize": (_i, [_vp, _i, _i, _i, _f, _vp, _vp, _vp, _vp]),
    "nvfp4_gemm": (_i, [ctypes.POINTER(GdnNVFP4), _i, ctypes.POINTER(GdnNVFP4), _i, _i, _vp, _i, _vp]),
    "gdn_decode_step": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _vp]),
    "gdn_mix_step": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i, _vp]),
    "gdn_prefill": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _i, _vp]),
    "gdn_verify": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _i, _vp, _vp, _vp]),
    "gdn_verify_commit": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp]),
    "kda_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "gdn_in_proj": (_i, [_vp, _vp, _vp, _i, _vp, _vp]),
    "gdn_in_mix": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _vp]),
    "gdn_out_proj": (_i, [_vp, _vp, _vp, _i, _vp, _vp]),
    "gdn_check": (_i, [_vp, _i, _vp]),
    "gdn_set_tuning": (_i, [_i, _i]),
    "gdn_decode_step_static": (_i, [ctypes.POINTER(GdnConfig), ctypes.POINTER(GdnWeights), _vp, _vp, _i, _vp, _vp,
                                    _vp, _i, _vp, _vp]),
}

_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{call} failed: {name}")


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with nvfp4_gated_deltanet_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, call: str):
    if status != GDN_OK:
        raise GdnError(status, call)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


from .api import *  # noqa: E402,F401,F403
