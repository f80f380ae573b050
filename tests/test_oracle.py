"""The fp64 oracle against the pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


def rec(q, k, v, g, beta, h0):
    return oracle.recurrence(q, k, v, g, beta, h0)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_recurrence_pin(pin):
    pin(rec)


@pytest.mark.parametrize("chunk", [1, 2, 16, 32, 64])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 33, 49, 64, 97])
def test_chunked_wy_equals_recurrence(chunk, T):
    """The chunkwise WY/UT form (an independent derivation: prefix sums, a
    unit-lower triangular solve and a state carry) reaches the recurrence's
    result for every chunk size, including a ragged last chunk."""
    q, k, v, g, beta, h0 = pins.random_problem(100 + T, B=1, T=T, HK=1, HV=2, dk=8, dv=6)
    o, ht = rec(q, k, v, g, beta, h0)
    oc, hc = oracle.chunked_wy(q, k, v, g, beta, h0, chunk=chunk)
    scale = max(np.abs(o).max(), 1.0)
    np.testing.assert_allclose(oc, o, atol=1e-12 * scale)
    np.testing.assert_allclose(hc, ht, atol=1e-12 * max(np.abs(ht).max(), 1.0))


def test_chunked_wy_is_pinned_too():
    """The chunked restatement passes the same pins as the recurrence."""
    for pin in pins.ALL_PINS:
        pin(lambda q, k, v, g, beta, h0: oracle.chunked_wy(q, k, v, g, beta, h0, chunk=4))


def test_strong_decay_chunked_no_overflow():
    """Strong decay (|g| ~ 8 per token) over a 64-token chunk: the chunked form
    keeps every exponent <= 0 and still matches."""
    q, k, v, g, beta, h0 = pins.random_problem(11, T=64, dk=4, dv=3, g_scale=8.0)
    o, ht = rec(q, k, v, g, beta, h0)
    oc, hc = oracle.chunked_wy(q, k, v, g, beta, h0, chunk=64)
    np.testing.assert_allclose(oc, o, atol=1e-12)
    np.testing.assert_allclose(hc, ht, atol=1e-12)


def test_threads_do_not_change_result():
    q, k, v, g, beta, h0 = pins.random_problem(12, B=3, T=20, HK=2, HV=4, dk=6, dv=5)
    o1, h1 = oracle.recurrence(q, k, v, g, beta, h0, threads=1)
    o4, h4 = oracle.recurrence(q, k, v, g, beta, h0, threads=5)
    assert np.array_equal(o1, o4) and np.array_equal(h1, h4)


def test_heads_subset_matches_full():
    q, k, v, g, beta, h0 = pins.random_problem(13, B=2, T=9, HK=2, HV=4, dk=4, dv=3)
    o, ht = rec(q, k, v, g, beta, h0)
    sub = oracle.recurrence_heads(q, k, v, g, beta, h0, [(0, 3), (1, 0), (1, 2)])
    for (b, hv), (ob, hb) in sub.items():
        assert np.array_equal(ob, o[b, :, hv]) and np.array_equal(hb, ht[b, hv])


def test_empty_sequence_returns_initial_state():
    q, k, v, g, beta, h0 = pins.random_problem(14, B=1, T=0, dk=4, dv=3)
    o, ht = rec(q, k, v, g, beta, h0)
    assert o.shape == (1, 0, 1, 3)
    assert np.array_equal(ht, h0)


def test_bad_arguments_rejected():
    q, k, v, g, beta, h0 = pins.random_problem(15, B=1, T=3, HK=2, HV=3, dk=4, dv=3)
    with pytest.raises(RuntimeError):
        rec(q, k, v, g, beta, None)
