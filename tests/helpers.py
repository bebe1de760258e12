"""Shared test plumbing: device upload of seeded inputs and the oracle runs the
GPU tests compare against. Nothing here computes any part of the layer."""
from __future__ import annotations

import functools

import numpy as np

from nvfp4_gated_deltanet_gb300 import synth


def to_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def to_host(t) -> np.ndarray:
    import torch
    a = t.detach().cpu().numpy()
    if t.dtype == torch.int16:
        a = a.view(np.uint16)
    return a


@functools.lru_cache(maxsize=4)
def weights(shape_name: str, seed: int):
    return synth.layer_weights(getattr(synth, shape_name), seed)


@functools.lru_cache(maxsize=4)
def oracle_layer(shape_name: str, seed: int):
    from oracle import gdn
    return gdn.Layer(weights(shape_name, seed))


def slot_inputs(shape, slots, steps, zero_state=False):
    """Per-slot x [steps][B][H] and initial states for the multi-sequence workloads."""
    x = np.stack([synth.x_tokens(shape, synth.slot_seed(s), steps) for s in slots], axis=1)
    conv = np.stack([synth.conv_state(shape, synth.slot_seed(s), zero_state) for s in slots])
    ssm = np.stack([synth.ssm_state(shape, synth.slot_seed(s), zero_state) for s in slots])
    return x, conv, ssm
