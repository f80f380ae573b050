"""Tree-verification oracle against pins (CPU only).

The definition (tree_recurrence) is pinned to the chain oracle, which has its
own pins: a chain-shaped tree is a plain sequence, a star is independent
single-token steps, and a hand-worked scalar tree fixes which state each
token sees.  The ancestor-masked WY form (tree_wy) must then reach the
definition on random and beam-shaped trees."""
import numpy as np
import pytest

import oracle
from channelwise_gated_delta_gb300.inputs import draw_parents
from tests import oracle_pins as pins


def problem(seed, T, B=1, HK=1, HV=2, dk=6, dv=5, h0=True):
    return pins.random_problem(seed, B=B, T=T, HK=HK, HV=HV, dk=dk, dv=dv, h0=h0)


def close(a, b, rel=1e-12):
    np.testing.assert_allclose(a, b, rtol=0, atol=rel * max(np.abs(b).max(), 1.0))


def test_hand_worked_scalar_tree():
    """dk = dv = 1, k = q = 1, beta = 1/2, h0 = 0, tokens 1 and 2 both
    children of token 0, g = (0, ln 1/2, 0), v = (1, 2, 3).  By hand:
      token 0: state 0 -> predict 0, u = (1 - 0)/2 = 0.5, state 0.5, o = 0.5
      token 1: decays 0.5 to 0.25, predict 0.25, u = (2 - 0.25)/2 = 0.875,
               state 1.125, o = 1.125
      token 2: starts again from token 0's 0.5 (not from token 1),
               predict 0.5, u = (3 - 0.5)/2 = 1.25, state 1.75, o = 1.75.
    (In sequence order token 2 would see 1.125 and give 2.0625.)"""
    one = np.ones((1, 3, 1, 1))
    v = np.array([1.0, 2.0, 3.0]).reshape(1, 3, 1, 1)
    g = np.array([0.0, np.log(0.5), 0.0]).reshape(1, 3, 1, 1)
    beta = np.full((1, 3, 1), 0.5)
    parent = np.array([[-1, 0, 0]])
    want = np.array([0.5, 1.125, 1.75]).reshape(1, 3, 1, 1)
    close(oracle.tree_recurrence(one, one, v, g, beta, None, parent), want)
    close(oracle.tree_wy(one, one, v, g, beta, None, parent), want)
    o_seq, _ = oracle.recurrence(one, one, v, g, beta, None)
    assert abs(o_seq[0, 2, 0, 0] - 2.0625) < 1e-15


@pytest.mark.parametrize("T", [1, 7, 20])
def test_chain_tree_is_the_sequence(T):
    q, k, v, g, beta, h0 = problem(200 + T, T)
    parent = draw_parents(1, T, "chain").numpy()
    o, _ = oracle.recurrence(q, k, v, g, beta, h0)
    close(oracle.tree_recurrence(q, k, v, g, beta, h0, parent), o)
    close(oracle.tree_wy(q, k, v, g, beta, h0, parent), o)


def test_star_tree_is_independent_steps():
    T = 9
    q, k, v, g, beta, h0 = problem(300, T)
    parent = draw_parents(1, T, "star").numpy()
    got = oracle.tree_recurrence(q, k, v, g, beta, h0, parent)
    for t in range(T):
        sl = slice(t, t + 1)
        o1, _ = oracle.recurrence(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], h0)
        close(got[:, sl], o1)


@pytest.mark.parametrize("kind,T,seed", [("random", 12, 0), ("random", 24, 1), ("beam", 21, 2),
                                         ("beam", 13, 3), ("random", 1, 4)])
def test_tree_wy_equals_definition(kind, T, seed):
    q, k, v, g, beta, h0 = problem(400 + seed, T, B=2, HK=1, HV=2)
    parent = draw_parents(2, T, kind, seed=seed).numpy()
    close(oracle.tree_wy(q, k, v, g, beta, h0, parent),
          oracle.tree_recurrence(q, k, v, g, beta, h0, parent), rel=1e-11)


def test_tree_wy_no_initial_state_and_grouped_heads():
    T = 15
    q, k, v, g, beta, h0 = problem(500, T, HK=2, HV=4, h0=False)
    parent = draw_parents(1, T, "random", seed=5).numpy()
    close(oracle.tree_wy(q, k, v, g, beta, None, parent),
          oracle.tree_recurrence(q, k, v, g, beta, None, parent), rel=1e-11)


def test_only_ancestors_matter():
    """Changing a token's inputs changes exactly the outputs of itself and
    its descendants."""
    T = 16
    q, k, v, g, beta, h0 = problem(600, T)
    parent = draw_parents(1, T, "random", seed=6).numpy()
    base = oracle.tree_recurrence(q, k, v, g, beta, h0, parent)
    t0 = 3
    v2 = v.copy()
    v2[0, t0] += 1.0
    moved = oracle.tree_recurrence(q, k, v2, g, beta, h0, parent)
    for t in range(T):
        path = []
        u = t
        while u >= 0:
            path.append(u)
            u = parent[0, u]
        changed = not np.array_equal(moved[0, t], base[0, t])
        assert changed == (t0 in path), t


def test_relabelling_permutes_outputs():
    """Another topological numbering of the same tree gives the same output
    per node."""
    T = 10
    q, k, v, g, beta, h0 = problem(700, T)
    parent = np.array([[-1, 0, 0, 1, 1, 2, -1, 6, 3, 7]])
    # new order: swap the subtrees' numbering while keeping parents first
    perm = [0, 6, 2, 1, 7, 5, 4, 3, 9, 8]    # new index n holds old node perm[n]
    inv = {old: new for new, old in enumerate(perm)}
    parent2 = np.array([[(-1 if parent[0, o] < 0 else inv[parent[0, o]]) for o in perm]])
    for n in range(T):
        assert parent2[0, n] < n
    take = lambda x: x[:, perm]
    base = oracle.tree_recurrence(q, k, v, g, beta, h0, parent)
    re = oracle.tree_recurrence(take(q), take(k), take(v), take(g), take(beta), h0, parent2)
    close(re, base[:, perm])
    close(oracle.tree_wy(take(q), take(k), take(v), take(g), take(beta), h0, parent2),
          base[:, perm], rel=1e-11)


def test_causal_mask_mutant_is_caught():
    """The plausible slip of keeping the causal mask on a tree is detected by
    the comparison with the definition."""
    T = 12
    q, k, v, g, beta, h0 = problem(800, T)
    parent = draw_parents(1, T, "beam", seed=8).numpy()
    want = oracle.tree_recurrence(q, k, v, g, beta, h0, parent)
    causal, _ = oracle.chunked_wy(q, k, v, g, beta, h0, chunk=T)
    assert np.abs(causal - want).max() > 1e-3
