"""The oracle's token-by-token prefill and decode steps on every host core.

TEST INFRASTRUCTURE, like the rest of ``oracle/``. This module adds no
arithmetic: it runs the layer's own stages (``gdn.Layer.projections``,
``gdn.Layer.mix`` and ``gdn.Layer.out_proj``) in worker processes and puts
their results together. Two facts of the layer's definition make the split
exact, so the result is bit-identical to ``gdn.Layer.prefill`` (pinned on the
CPU by comparing the two):

* up to the gated norm, the value heads of one key head read only their own
  projection rows, conv channels, gates and recurrent state. The recurrence of
  that group is therefore the recurrence of a layer with one key head whose
  weight rows are the full layer's rows for it (the grouped-query map of the
  Rocket blog's GDN entry: value head h reads key head h / (Hv / Hk));
* the NVFP4 quantisers and the W4A4 products treat every token row on its own
  (one tensor scale per site, set in advance), so token ranges of the
  projections and of the out-projection can run apart, and the rows of a
  decode batch (each with its own state) can too.

Workers are started with the ``spawn`` method (safe in a process that already
uses a GPU) and import numpy and the oracle only. BLAS threads are pinned to
one per worker, so the worker count is the core count used.
"""
from __future__ import annotations

import dataclasses
import multiprocessing as mp
import os

import numpy as np

from . import gdn

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
_TOKEN_CHUNK = 1024  # projection rows per pass inside a worker (bounds its memory)


# ------------------------------------------------------------------ plain weight records
# Field-for-field copies of what gdn.Layer reads from a weight set, so that the
# workers need nothing but numpy and this package.

@dataclasses.dataclass(frozen=True)
class Shape:
    hidden: int
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    conv_kernel: int

    @property
    def value_dim(self) -> int:
        return self.n_v_heads * self.d_v


@dataclasses.dataclass
class Matrix:
    codes: np.ndarray
    scales: np.ndarray
    tensor_scale: float


@dataclasses.dataclass
class Weights:
    shape: Shape
    qkvz: Matrix
    ba: Matrix
    out: Matrix
    conv_w: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray
    norm_w: np.ndarray
    act_scale_in: float
    act_scale_out: float
    rms_eps: float
    l2_eps: float


def plain(w) -> Weights:
    """A weight set with the attributes gdn.Layer reads, as a ``Weights`` record."""
    s = w.shape
    m = lambda x: Matrix(np.asarray(x.codes), np.asarray(x.scales), float(x.tensor_scale))
    return Weights(Shape(s.hidden, s.n_k_heads, s.n_v_heads, s.d_k, s.d_v, s.conv_kernel), m(w.qkvz), m(w.ba),
                   m(w.out), np.asarray(w.conv_w), np.asarray(w.A_log), np.asarray(w.dt_bias), np.asarray(w.norm_w),
                   float(w.act_scale_in), float(w.act_scale_out), float(w.rms_eps), float(w.l2_eps))


def group_rows(shape: Shape, kh: int):
    """Rows of key head kh's group: (qkvz rows q|k|v|z, ba rows b|a, conv
    channels q|k|v, value heads), each in the full layer's order."""
    D, Hk, Hv = shape.d_k, shape.n_k_heads, shape.n_v_heads
    G = Hv // Hk
    heads = list(range(kh * G, (kh + 1) * G))
    q = list(range(kh * D, (kh + 1) * D))
    k = [Hk * D + r for r in q]
    v = [2 * Hk * D + h * D + i for h in heads for i in range(D)]
    z = [2 * Hk * D + Hv * D + h * D + i for h in heads for i in range(D)]
    ba = heads + [Hv + h for h in heads]
    return q + k + v + z, ba, q + k + v, heads


def group_weights(w: Weights, kh: int) -> Weights:
    """The layer restricted to key head kh: one key head, its G value heads,
    the full layer's weight rows for them (out-projection: their columns)."""
    s = w.shape
    rows, ba_rows, chans, heads = group_rows(s, kh)
    G = len(heads)
    c0, c1 = heads[0] * s.d_v, (heads[-1] + 1) * s.d_v  # the group's columns of y (heads are contiguous)
    sub = lambda m, r: Matrix(m.codes[r], m.scales[r], m.tensor_scale)
    out = Matrix(w.out.codes[:, c0 // 2:c1 // 2], w.out.scales[:, c0 // 16:c1 // 16], w.out.tensor_scale)
    return Weights(Shape(s.hidden, 1, G, s.d_k, s.d_v, s.conv_kernel), sub(w.qkvz, rows), sub(w.ba, ba_rows),
                   out, w.conv_w[chans], w.A_log[heads],
                   w.dt_bias[heads], w.norm_w, w.act_scale_in, w.act_scale_out, w.rms_eps, w.l2_eps)


# ------------------------------------------------------------------ tasks

def group_recurrence(wg: Weights, x_bits: np.ndarray, conv_g: np.ndarray, ssm_g: np.ndarray):
    """gdn.Layer.prefill's token loop for one key head's group, stopped before
    the out-projection: returns (y float64 [T][G*d_v], conv state, recurrent
    state) with the states as the prefill leaves them (FP32 within the call)."""
    L = gdn.Layer(wg)
    conv, S = conv_g.copy(), ssm_g.copy()
    T = x_bits.shape[0]
    y = np.empty((T, wg.shape.value_dim), dtype=np.float64)
    for t0 in range(0, T, _TOKEN_CHUNK):
        qkvz, ba = L.projections(x_bits[t0:t0 + _TOKEN_CHUNK])
        for i in range(qkvz.shape[0]):
            y[t0 + i], conv, S, _ = L.mix(qkvz[i], ba[i], conv, S, "f32")
    return y, conv, S


_W = None  # the worker's weight set (set once per worker)
_L = None  # the worker's full layer, built on first use


def _init_worker(w: Weights):
    global _W, _L
    _W, _L = w, None


def _layer():
    global _L
    if _L is None:
        _L = gdn.Layer(_W)
    return _L


def _task(job):
    kind = job[0]
    if kind == "group":
        _, kh, x_bits, conv_g, ssm_g = job
        return group_recurrence(group_weights(_W, kh), x_bits, conv_g, ssm_g)
    if kind == "out":
        return _layer().out_proj(job[1])
    if kind == "rows":   # decode rows with their own states (slots 0..n-1 of the job)
        _, x_bits, ids, conv, ssm = job
        out = _layer().decode_step(x_bits, ids, conv, ssm)
        return out, conv, ssm
    raise ValueError(kind)


def _pool(n: int, w: Weights):
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    for v in _THREAD_VARS:
        os.environ[v] = "1"
    try:
        return mp.get_context("spawn").Pool(n, initializer=_init_worker, initargs=(w,))
    finally:
        for v, val in saved.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val


def make_pool(weights, workers: int | None = None):
    """A worker pool holding ``weights`` for repeated calls (pass it as
    ``pool=``; the caller closes it). Its size is the core count used."""
    n = (os.cpu_count() or 1) if workers is None else workers
    return _pool(n, plain(weights)), n


def decode_step(weights, x_bits: np.ndarray, slot_ids, conv_state: np.ndarray, ssm_state: np.ndarray,
                workers: int | None = None, pool=None) -> np.ndarray:
    """Same contract and result as ``gdn.Layer(weights).decode_step``: the rows
    are split over ``workers`` processes (rows are independent: per-row
    quantisation, products, state). 0 runs in this process; ``pool`` (from
    make_pool with the same weights, and its size as ``workers``) is reused."""
    w = plain(weights)
    x_bits = np.asarray(x_bits, dtype=np.uint16).reshape(len(slot_ids), w.shape.hidden)
    n = (os.cpu_count() or 1) if workers is None else workers
    rows = list(range(len(slot_ids)))
    parts = [rows[i::max(1, n)] for i in range(max(1, n))]
    jobs, index = [], []
    for part in parts:
        if not part:
            continue
        live = [r for r in part if slot_ids[r] >= 0]
        ids = [live.index(r) if slot_ids[r] >= 0 else -1 for r in part]
        sl = [slot_ids[r] for r in live]
        jobs.append(("rows", x_bits[part], ids, conv_state[sl].copy(), ssm_state[sl].copy()))
        index.append((part, sl))
    if n <= 0:
        _init_worker(w)
        res = [_task(j) for j in jobs]
    elif pool is not None:
        res = pool.map(_task, jobs, chunksize=1)
    else:
        own = _pool(n, w)
        try:
            res = own.map(_task, jobs, chunksize=1)
        finally:
            own.close()
            own.join()
    out = np.zeros((len(slot_ids), w.shape.hidden), np.uint16)
    for (part, sl), (o, c, s) in zip(index, res):
        out[part] = o
        conv_state[sl] = c
        ssm_state[sl] = s
    return out


def prefill(weights, x_bits: np.ndarray, conv_state: np.ndarray, ssm_state: np.ndarray, init_zero: bool,
            workers: int | None = None, pool=None) -> np.ndarray:
    """Same contract and result as ``gdn.Layer(weights).prefill`` for an FP32
    state: x_bits BF16 [T][H]; conv_state [K-1][C] and ssm_state [Hv][dv][dk]
    updated in place; returns out BF16 bits [T][H]. ``workers`` processes (by
    default one per host core, at most one per key head for the recurrence);
    0 runs every task in this process; ``pool`` as for decode_step."""
    w = plain(weights)
    s = w.shape
    if init_zero:
        conv_state[...] = 0
        ssm_state[...] = 0
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T = x_bits.shape[0]
    groups = []
    for kh in range(s.n_k_heads):
        _, _, chans, heads = group_rows(s, kh)
        groups.append(("group", kh, x_bits, conv_state[:, chans].copy(), ssm_state[heads].copy()))
    n = (os.cpu_count() or 1) if workers is None else workers
    own = None
    if n <= 0:
        _init_worker(w)
        run = lambda jobs: [_task(j) for j in jobs]
    else:
        if pool is None:
            pool = own = _pool(n, w)
        run = lambda jobs: pool.map(_task, jobs, chunksize=1)
    res = run(groups)
    try:
        y = np.empty((T, s.value_dim), dtype=np.float64)
        for (_, kh, _, _, _), (yg, cg, sg) in zip(groups, res):
            _, _, chans, heads = group_rows(s, kh)
            y[:, heads[0] * s.d_v:(heads[-1] + 1) * s.d_v] = yg
            conv_state[:, chans] = cg
            ssm_state[heads] = sg
        parts = max(1, n)
        bounds = np.linspace(0, T, parts + 1).astype(int)
        outs = run([("out", y[a:b]) for a, b in zip(bounds[:-1], bounds[1:]) if b > a])
    finally:
        if own is not None:
            own.close()
            own.join()
    return np.concatenate(outs, axis=0) if outs else np.zeros((0, s.hidden), np.uint16)
