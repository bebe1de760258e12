"""The all-cores prefill of the oracle (``oracle.parallel``) is the oracle's own
token-by-token prefill, bit for bit: outputs, conv state and recurrent state.

The split it relies on (key-head groups independent up to the out-projection,
token rows independent in the quantisers and products) is a property of the
layer's definition; these cases would fail on a wrong row, channel or column
map, a dropped group, a token range off by one, or a state not carried
between token chunks."""
import numpy as np
import pytest

from nvfp4_gated_deltanet_gb300 import synth
from oracle import gdn, parallel


def _both(shape_name, seed, T, workers, init_zero=False, state_seed=3):
    shape = getattr(synth, shape_name)
    w = synth.layer_weights(shape, seed)
    x = synth.x_tokens(shape, 7, T)
    c1, s1 = synth.conv_state(shape, state_seed), synth.ssm_state(shape, state_seed)
    c2, s2 = c1.copy(), s1.copy()
    want = gdn.Layer(w).prefill(x, c1, s1, init_zero)
    got = parallel.prefill(w, x, c2, s2, init_zero, workers=workers)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(c2, c1)
    np.testing.assert_array_equal(s2, s1)


@pytest.mark.parametrize("T", [1, 150])
def test_parallel_prefill_equals_oracle_prefill_tiny(T):
    _both("TINY", 0, T, workers=0)


def test_parallel_prefill_in_worker_processes():
    _both("TINY", 0, 70, workers=2, init_zero=True)


def test_parallel_prefill_equals_oracle_prefill_full_width():
    _both("FULL", 1, 3, workers=0)


def test_parallel_prefill_crosses_token_chunks(monkeypatch):
    """Token chunks of 16 inside a worker: the states carry across them."""
    monkeypatch.setattr(parallel, "_TOKEN_CHUNK", 16)
    _both("TINY", 0, 53, workers=0)


@pytest.mark.parametrize("workers", [0, 2])
def test_parallel_decode_step_equals_oracle_decode_step(workers):
    """Rows split over workers, with padding rows and slots out of row order."""
    shape = synth.TINY
    w = synth.layer_weights(shape, 0)
    ids = [3, -1, 0, 5, 1]
    S = 6
    x = np.stack([synth.x_tokens(shape, 40 + r, 1)[0] for r in range(len(ids))])
    c1 = np.stack([synth.conv_state(shape, 50 + s) for s in range(S)])
    s1 = np.stack([synth.ssm_state(shape, 50 + s) for s in range(S)])
    c2, s2 = c1.copy(), s1.copy()
    want = gdn.Layer(w).decode_step(x, ids, c1, s1)
    got = parallel.decode_step(w, x, ids, c2, s2, workers=workers)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(c2, c1)
    np.testing.assert_array_equal(s2, s1)
