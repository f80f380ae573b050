"""Checks that pin the fp64 oracle to facts outside itself.

Each ``pin_*`` function takes a recurrence callable
``rec(q, k, v, g, beta, h0) -> (o, ht)`` (numpy float64 in and out, layouts of
the oracle) and raises AssertionError if the callable disagrees with what the
mathematics of the method fixes.  They are run on the real oracle
(test_oracle.py) and on deliberately broken builds of it
(test_oracle_mutants.py), which must each fail at least one of them.

The method (page "Reorder channelwise gated delta rule chunked hot loops for
autovectorization", pytorch/executorch PR #21021, first commit summary): per
value head a state S[dk][dv] is decayed per key channel by exp(g_t), a value
is predicted from the decayed state, a beta-weighted rank-one update moves
the prediction toward v_t, and the output is read from the updated state.
"""
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x, axis=-1):
    return x / np.linalg.norm(x, axis=axis, keepdims=True)


def random_problem(seed, B=1, T=5, HK=1, HV=1, dk=5, dv=3, h0=True, g_scale=1.0):
    r = _rng(seed)
    q = _unit(r.standard_normal((B, T, HK, dk)))
    k = _unit(r.standard_normal((B, T, HK, dk)))
    v = r.standard_normal((B, T, HV, dv))
    g = -np.log1p(np.exp(r.standard_normal((B, T, HV, dk)))) * g_scale
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, HV))))
    s0 = 0.3 * r.standard_normal((B, HV, dk, dv)) if h0 else None
    return q, k, v, g, beta, s0


# ---------------------------------------------------------------- golden files
def load_golden(name):
    """Parses a hand-worked fixture: 'shape' line plus one line per tensor."""
    vals, shape = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split(None, 1)
            if key == "shape":
                for tok in rest.split():
                    a, b = tok.split("=")
                    shape[a] = int(b)
                continue
            toks = []
            for tok in rest.split():
                if tok == "ln2":
                    toks.append(math.log(2.0))
                elif tok == "-ln2":
                    toks.append(-math.log(2.0))
                else:
                    toks.append(float(tok))
            vals[key] = np.array(toks)
    B, T, HK, HV, dk, dv = (shape[x] for x in ("B", "T", "HK", "HV", "dk", "dv"))
    out = dict(
        q=vals["q"].reshape(B, T, HK, dk), k=vals["k"].reshape(B, T, HK, dk),
        v=vals["v"].reshape(B, T, HV, dv), g=vals["g"].reshape(B, T, HV, dk),
        beta=vals["beta"].reshape(B, T, HV), h0=vals["h0"].reshape(B, HV, dk, dv),
        o=vals["o"].reshape(B, T, HV, dv), ht=vals["ht"].reshape(B, HV, dk, dv))
    return out


def pin_golden(rec):
    """Hand-worked examples (tests/golden/*.txt), every value derived by hand."""
    for name in ("hand_worked_dk2_dv3_t2.txt", "hand_worked_gqa_hk2_hv4.txt"):
        d = load_golden(name)
        o, ht = rec(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
        np.testing.assert_allclose(o, d["o"], rtol=0, atol=1e-12, err_msg=name + " o")
        np.testing.assert_allclose(ht, d["ht"], rtol=0, atol=1e-12, err_msg=name + " ht")


# ---------------------------------------------------------------- closed forms
def pin_beta_zero_is_pure_decay(rec):
    """beta = 0: no update happens, so S_t = diag(exp(sum_{s<=t} g_s)) h0 and
    o_t = S_t^T q_t.  dk != dv and per-channel g catch a decay applied along
    the wrong axis."""
    q, k, v, g, beta, h0 = random_problem(1, B=2, T=6, HK=1, HV=2, dk=5, dv=3)
    beta = np.zeros_like(beta)
    o, ht = rec(q, k, v, g, beta, h0)
    G = np.cumsum(g, axis=1)  # [B, T, HV, dk]
    for b in range(2):
        for hv in range(2):
            for t in range(6):
                St = np.exp(G[b, t, hv])[:, None] * h0[b, hv]
                np.testing.assert_allclose(o[b, t, hv], St.T @ q[b, t, 0], atol=1e-13)
            np.testing.assert_allclose(ht[b, hv], np.exp(G[b, -1, hv])[:, None] * h0[b, hv],
                                       atol=1e-13)


def pin_delta_step(rec):
    """One token with a unit key: the delta update moves the prediction a
    fraction beta of the way to v, so with q = k
    o = (1 - beta) (D h0)^T k + beta v, D = diag(exp(g)).  It fixes the
    decay-before-predict order, the sign of the correction, the beta scale and
    that the output is read after the update."""
    for seed in range(3):
        q, k, v, g, beta, h0 = random_problem(10 + seed, T=1, dk=6, dv=4)
        q = k.copy()
        o, ht = rec(q, k, v, g, beta, h0)
        D = np.exp(g[0, 0, 0])[:, None]
        kk = k[0, 0, 0]
        pred = (D * h0[0, 0]).T @ kk
        expect = (1.0 - beta[0, 0, 0]) * pred + beta[0, 0, 0] * v[0, 0, 0]
        np.testing.assert_allclose(o[0, 0, 0], expect, atol=1e-13)
        # and the state is exactly decay plus a rank-one term along k
        R = ht[0, 0] - D * h0[0, 0]
        np.testing.assert_allclose(R, np.outer(kk, kk @ R), atol=1e-13)


def pin_orthonormal_keys_write_exactly(rec):
    """g = 0, beta = 1 and orthonormal keys: each update overwrites the value
    stored along its key without disturbing the others, so at the end
    S^T k_t = v_t for every t, and with h0 = 0, S = sum_t k_t v_t^T."""
    r = _rng(3)
    dk, dv, T = 8, 5, 6
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    k = Qm[:T][None, :, None, :]
    q = _unit(r.standard_normal((1, T, 1, dk)))
    v = r.standard_normal((1, T, 1, dv))
    g = np.zeros((1, T, 1, dk))
    beta = np.ones((1, T, 1))
    h0 = 0.3 * r.standard_normal((1, 1, dk, dv))
    _, ht = rec(q, k, v, g, beta, h0)
    for t in range(T):
        np.testing.assert_allclose(ht[0, 0].T @ k[0, t, 0], v[0, t, 0], atol=1e-12)
    _, ht0 = rec(q, k, v, g, beta, None)
    np.testing.assert_allclose(ht0[0, 0], sum(np.outer(k[0, t, 0], v[0, t, 0]) for t in range(T)),
                               atol=1e-12)


def pin_reset(rec):
    """exp(g_t) = 0 on every channel erases the state: S_t = beta_t k_t v_t^T,
    and every later output equals a fresh run started at token t."""
    q, k, v, g, beta, h0 = random_problem(4, T=7, dk=4, dv=3)
    t = 3
    g = g.copy()
    g[:, t] = -1.0e4  # exp underflows to exactly 0 in float64
    o, ht = rec(q, k, v, g, beta, h0)
    o_fresh, ht_fresh = rec(q[:, t:], k[:, t:], v[:, t:], g[:, t:], beta[:, t:], None)
    np.testing.assert_allclose(o[:, t:], o_fresh, atol=1e-13)
    np.testing.assert_allclose(ht, ht_fresh, atol=1e-13)
    o1, ht1 = rec(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], g[:, :t + 1], beta[:, :t + 1], h0)
    np.testing.assert_allclose(ht1[0, 0], beta[0, t, 0] * np.outer(k[0, t, 0], v[0, t, 0]),
                               atol=1e-13)


# ---------------------------------------------------------------- invariants
def pin_linearity(rec):
    """For fixed q, k, g, beta the map (V, h0) -> (O, ht) is linear."""
    q, k, v1, g, beta, h1 = random_problem(5, B=1, T=9, HK=1, HV=2, dk=4, dv=3)
    _, _, v2, _, _, h2 = random_problem(6, B=1, T=9, HK=1, HV=2, dk=4, dv=3)
    a = -1.7
    oa, ha = rec(q, k, a * v1 + v2, g, beta, a * h1 + h2)
    o1, s1 = rec(q, k, v1, g, beta, h1)
    o2, s2 = rec(q, k, v2, g, beta, h2)
    np.testing.assert_allclose(oa, a * o1 + o2, atol=1e-12)
    np.testing.assert_allclose(ha, a * s1 + s2, atol=1e-12)


def pin_value_columns_independent(rec):
    """Permuting the value channels of v and h0 permutes o and ht the same way."""
    q, k, v, g, beta, h0 = random_problem(7, T=8, dk=4, dv=6)
    perm = np.array([3, 0, 5, 1, 4, 2])
    o, ht = rec(q, k, v, g, beta, h0)
    op, hp = rec(q, k, v[..., perm], g, beta, h0[..., perm])
    np.testing.assert_allclose(op, o[..., perm], atol=1e-13)
    np.testing.assert_allclose(hp, ht[..., perm], atol=1e-13)


def pin_gqa_is_repeated_heads(rec):
    """Grouped heads equal ungrouped heads with each key/query head repeated
    over its G = HV/HK consecutive value heads."""
    q, k, v, g, beta, h0 = random_problem(8, B=2, T=5, HK=2, HV=6, dk=4, dv=3)
    o, ht = rec(q, k, v, g, beta, h0)
    qr, kr = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    o2, ht2 = rec(qr, kr, v, g, beta, h0)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(ht, ht2, atol=1e-14)


def pin_resume(rec):
    """Running T1 + T2 tokens equals running T2 tokens from the final state of
    the first T1 (the final state is the only thing carried)."""
    q, k, v, g, beta, h0 = random_problem(9, B=2, T=11, HK=1, HV=2, dk=4, dv=3)
    o, ht = rec(q, k, v, g, beta, h0)
    c = 4
    oa, ha = rec(q[:, :c], k[:, :c], v[:, :c], g[:, :c], beta[:, :c], h0)
    ob, hb = rec(q[:, c:], k[:, c:], v[:, c:], g[:, c:], beta[:, c:], ha)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-13)
    np.testing.assert_allclose(hb, ht, atol=1e-13)


ALL_PINS = [pin_golden, pin_beta_zero_is_pure_decay, pin_delta_step,
            pin_orthonormal_keys_write_exactly, pin_reset, pin_linearity,
            pin_value_columns_independent, pin_gqa_is_repeated_heads, pin_resume]
