"""Chunk-parallel scan oracle against pins (CPU only).

``affine_map`` is pinned to the token recurrence (itself pinned in
test_oracle.py) through the facts that make the split possible: the end
state is affine in the start state with the same M for every start, c is the
end state from a zero start, M is the end state of a zero-value run from the
identity, and two closed forms (no delta update; orthonormal keys with no
decay) fix M outright.  ``segmented_forward`` must then give the recurrence's
outputs and final state for every segment count."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


def problem(seed, T, B=1, HK=1, HV=2, dk=5, dv=4, h0=True):
    return pins.random_problem(seed, B=B, T=T, HK=HK, HV=HV, dk=dk, dv=dv, h0=h0)


def close(a, b, rel=1e-12):
    np.testing.assert_allclose(a, b, rtol=0, atol=rel * max(np.abs(b).max(), 1.0))


def apply(M, S, c):
    return np.einsum("bhij,bhjv->bhiv", M, S) + c


def test_one_token_map_is_one_step():
    q, k, v, g, beta, h0 = problem(1, 1)
    M, c = oracle.affine_map(k, v, g, beta, 0, 1)
    _, s1 = oracle.recurrence(q, k, v, g, beta, h0)
    close(apply(M, h0, c), s1)


@pytest.mark.parametrize("t0,t1", [(0, 9), (3, 17), (17, 18), (5, 5)])
def test_end_state_is_affine_in_the_start(t0, t1):
    """Two random starts and the zero start give M S + c with one (M, c)."""
    q, k, v, g, beta, h0 = problem(2, 18, B=2, HK=1, HV=2)
    M, c = oracle.affine_map(k, v, g, beta, t0, t1)
    sl = slice(t0, t1)
    rng = np.random.default_rng(3)
    for S in (h0, rng.standard_normal(h0.shape), np.zeros_like(h0)):
        _, end = oracle.recurrence(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S)
        close(apply(M, S, c), end)


def test_identity_start_with_zero_values_gives_the_map():
    """dk = dv: a run from h0 = I with v = 0 ends in M (how the map is
    obtained from a plain state run), and one from h0 = 0 ends in c."""
    T, d = 11, 6
    q, k, v, g, beta, _ = problem(4, T, HK=1, HV=3, dk=d, dv=d)
    M, c = oracle.affine_map(k, v, g, beta, 0, T)
    eye = np.broadcast_to(np.eye(d), (1, 3, d, d)).copy()
    _, end_m = oracle.recurrence(q, k, np.zeros_like(v), g, beta, eye)
    _, end_c = oracle.recurrence(q, k, v, g, beta, None)
    close(end_m, M)
    close(end_c, c)


def test_no_update_is_pure_decay():
    """beta = 0: M = diag(exp(sum of g)), c = 0."""
    T = 7
    q, k, v, g, beta, _ = problem(5, T)
    M, c = oracle.affine_map(k, v, g, np.zeros_like(beta), 0, T)
    want = np.zeros_like(M)
    for hv in range(M.shape[1]):
        want[0, hv] = np.diag(np.exp(g[0, :, hv].sum(axis=0)))
    close(M, want)
    assert np.abs(c).max() == 0.0


def test_orthonormal_keys_project_out():
    """g = 0, beta = 1, orthonormal keys: each token removes its key's
    direction, so M = I - sum_t k_t k_t^T and c = sum_t k_t v_t^T."""
    d, T = 6, 4
    rng = np.random.default_rng(6)
    basis, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = basis[:T].reshape(1, T, 1, d)
    v = rng.standard_normal((1, T, 1, 3))
    g = np.zeros((1, T, 1, d))
    beta = np.ones((1, T, 1))
    M, c = oracle.affine_map(k, v, g, beta, 0, T)
    K = k[0, :, 0]
    close(M[0, 0], np.eye(d) - K.T @ K)
    close(c[0, 0], K.T @ v[0, :, 0])


@pytest.mark.parametrize("segments", [1, 2, 3, 4, 7, 50])
@pytest.mark.parametrize("T,chunk", [(37, 4), (64, 16), (5, 16)])
def test_segmented_equals_recurrence(segments, T, chunk):
    q, k, v, g, beta, h0 = problem(10 + T, T, B=2, HK=1, HV=2)
    o, ht = oracle.recurrence(q, k, v, g, beta, h0)
    o2, ht2 = oracle.segmented_forward(q, k, v, g, beta, h0, segments=segments, chunk=chunk)
    close(o2, o, rel=1e-11)
    close(ht2, ht, rel=1e-11)


def test_segmented_grouped_heads_no_initial_state():
    T = 40
    q, k, v, g, beta, _ = problem(20, T, HK=2, HV=4, h0=False)
    o, ht = oracle.recurrence(q, k, v, g, beta, None)
    o2, ht2 = oracle.segmented_forward(q, k, v, g, beta, None, segments=4, chunk=8)
    close(o2, o, rel=1e-11)
    close(ht2, ht, rel=1e-11)


def test_segment_bounds():
    assert oracle.segment_bounds(0, 64, 3) == []
    assert oracle.segment_bounds(100, 64, 3) == [(0, 64), (64, 100)]
    assert oracle.segment_bounds(4096, 64, 3) == [(0, 1408), (1408, 2816), (2816, 4096)]
    b = oracle.segment_bounds(1000, 16, 5)
    assert b[0][0] == 0 and b[-1][1] == 1000
    assert all(x[1] == y[0] for x, y in zip(b, b[1:]))
    assert all(t0 % 16 == 0 for t0, _ in b)


def test_wrong_composition_order_is_caught():
    """Composing the token maps on the wrong side (M <- M A_t) breaks the
    affine pin: the check above would see it."""
    T = 6
    q, k, v, g, beta, h0 = problem(30, T, HV=1)
    M, c = oracle.affine_map(k, v, g, beta, 0, T)
    wrong = np.eye(M.shape[-1])
    for t in range(T):
        kt = k[0, t, 0]
        wrong = wrong @ ((np.eye(len(kt)) - beta[0, t, 0] * np.outer(kt, kt))
                         * np.exp(g[0, t, 0])[None, :])
    assert np.abs(wrong - M[0, 0]).max() > 1e-3
