"""KDA-style recurrent step (per-channel gated delta rule), float64.

TEST INFRASTRUCTURE ONLY: imported by tests/ and bench.py's CPU baseline, never
by the library.

Rocket blog, "Moving the KDA state tile out of shared memory is 4.6x at M=8":
a KDA layer carries a 64 x 128 x 128 recurrent state per stream that every
step reads and writes, stored in FP32 (or BF16 in the storage lane's
contract); the step is checked against a double-precision evaluation with
o and state tolerances of 4e-3 and 1e-5 (FP32 state) / 4e-3 (BF16 state). The
entry does not print the recurrence. The reading taken here is the gated delta
rule of this library with the scalar decay of a head replaced by one decay per
key channel (the "fine-grained" gate of Kimi Delta Attention), in the state
layout S[d_v][d_k]:

    S <- S diag(exp(g));  u = beta (v - S k);  S <- S + u k^T;  o = S q

g is the per-channel log-decay [d_k], beta a scalar per head; q, k, v as given
(no normalisation inside the step). With every g_j equal this is exactly the
GDN delta rule of ``gdn.delta_step``.
"""
from __future__ import annotations

import numpy as np

from . import codecs


def kda_step(q, k, v, g, beta, S, state_store: str = "f32"):
    """One step for M streams x H heads.

    q, k, g: [M][H][dk]; v: [M][H][dv]; beta: [M][H]; S: [M][H][dv][dk].
    Returns (o float64 [M][H][dv], S' [M][H][dv][dk] float32 rounded to the
    storage type: "f32", or "bf16" (FP32 then BF16))."""
    q, k, v, g = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g))
    beta = np.asarray(beta, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    Sd = S * np.exp(g)[:, :, None, :]                        # decay each key column
    Sk = np.einsum("mhvk,mhk->mhv", Sd, k)
    u = beta[:, :, None] * (v - Sk)
    Sn = Sd + u[:, :, :, None] * k[:, :, None, :]
    o = np.einsum("mhvk,mhk->mhv", Sn, q)
    S32 = Sn.astype(np.float32)
    if state_store == "bf16":
        S32 = codecs.bf16_to_f32(codecs.f32_to_bf16(S32))
    return o, S32
