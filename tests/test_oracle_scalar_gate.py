"""Scalar-gate oracle against pins (CPU only).

The definition (g broadcast over key channels through the pinned recurrence)
is checked against the per-key-head-gram chunked form, against a closed form
for beta = 0, and against a hand-worked scalar case; a channelwise g that is
not constant over channels must NOT match (the broadcast is the only link)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


def problem(seed, T, B=1, HK=2, HV=4, dk=6, dv=5, h0=True):
    q, k, v, gc, beta, s0 = pins.random_problem(seed, B=B, T=T, HK=HK, HV=HV, dk=dk, dv=dv, h0=h0)
    g = gc[..., 0].copy()            # one log-decay per token and value head
    return q, k, v, g, beta, s0


def close(a, b, rel=1e-12):
    np.testing.assert_allclose(a, b, rtol=0, atol=rel * max(np.abs(b).max(), 1.0))


@pytest.mark.parametrize("T,chunk", [(1, 4), (13, 4), (33, 16), (64, 64), (97, 32)])
def test_key_head_gram_form_equals_definition(T, chunk):
    q, k, v, g, beta, s0 = problem(900 + T, T)
    o, ht = oracle.scalar_gate_recurrence(q, k, v, g, beta, s0)
    o2, h2 = oracle.scalar_gate_wy(q, k, v, g, beta, s0, chunk=chunk)
    close(o2, o, 1e-11)
    close(h2, ht, 1e-11)


def test_pure_decay_closed_form():
    """beta = 0: the state only decays, by exp(sum of g) as a scalar, so
    o_t = exp(G_t) S0^T q_t and ht = exp(G_T) S0."""
    q, k, v, g, beta, s0 = problem(910, 9, HK=1, HV=2)
    beta[:] = 0.0
    o, ht = oracle.scalar_gate_recurrence(q, k, v, g, beta, s0)
    G = np.cumsum(g[0], axis=0)                       # [T, HV]
    for hv in range(2):
        for t in range(9):
            close(o[0, t, hv], np.exp(G[t, hv]) * s0[0, hv].T @ q[0, t, 0])
        close(ht[0, hv], np.exp(G[-1, hv]) * s0[0, hv])


def test_hand_worked_scalar_case():
    """dk = 2, dv = 1, one head, h0 = [1, 2]^T, k = q = e1, beta = 1/2,
    g = ln(1/2) then 0, v = (3, 0).  By hand:
      t0: state [0.5, 1]; predict k.S = 0.5; u = (3 - 0.5)/2 = 1.25;
          state [1.75, 1]; o = q.S = 1.75
      t1: no decay; predict 1.75; u = (0 - 1.75)/2 = -0.875;
          state [0.875, 1]; o = 0.875."""
    e1 = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)
    q = np.repeat(e1, 2, axis=1)
    k = q.copy()
    v = np.array([3.0, 0.0]).reshape(1, 2, 1, 1)
    g = np.array([np.log(0.5), 0.0]).reshape(1, 2, 1)
    beta = np.full((1, 2, 1), 0.5)
    h0 = np.array([1.0, 2.0]).reshape(1, 1, 2, 1)
    o, ht = oracle.scalar_gate_recurrence(q, k, v, g, beta, h0)
    close(o.ravel(), np.array([1.75, 0.875]))
    close(ht.ravel(), np.array([0.875, 1.0]))
    o2, h2 = oracle.scalar_gate_wy(q, k, v, g, beta, h0, chunk=2)
    close(o2.ravel(), np.array([1.75, 0.875]))
    close(h2.ravel(), np.array([0.875, 1.0]))


def test_channel_varying_decay_differs():
    """Mutant check: the key-head gram form assumes one decay for all
    channels; with channelwise g it is not the channelwise result."""
    q, k, v, gc, beta, s0 = pins.random_problem(920, B=1, T=16, HK=1, HV=2, dk=6, dv=5)
    o_c, _ = oracle.recurrence(q, k, v, gc, beta, s0)
    o_s, _ = oracle.scalar_gate_wy(q, k, v, gc[..., 0], beta, s0, chunk=8)
    assert np.abs(o_c - o_s).max() > 1e-3
