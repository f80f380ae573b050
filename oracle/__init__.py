"""fp64 CPU oracle for the channelwise gated delta rule forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library.

Two routines, both in float64:

``recurrence``
    The definition: the per-token four-sweep recurrence (decay, predict,
    rank-one delta update, output) of the page "Reorder channelwise gated
    delta rule chunked hot loops for autovectorization" (pytorch/executorch
    PR #21021, first commit summary).  Implemented in C (gdr_oracle.c),
    threaded over (batch, value head).  This is THE oracle.

``chunked_wy``
    The chunkwise WY/UT restatement named in the second commit summary of the
    same page (per-channel log-decay prefixes, causal query/key terms, the
    beta-folded triangular transform, WY pseudo-values, inter-chunk state
    carry, ragged last chunk).  Written from the algebra of unrolling the
    recurrence over a chunk; it exists to pin the recurrence (the two must
    agree to rounding for every chunk size) and is never the parity target.

``tree_recurrence`` / ``tree_wy``
    Tree verification, the workload of the page "Support TreeUpdateSolve
    kernel" (trymirai/uzu PR #576): the tokens form a tree of draft tokens
    (parents before children) and the tree's ancestor relation takes the
    place of the causal order.  ``tree_recurrence`` is the definition: each
    token's output is the last output of the token recurrence run along its
    root path.  ``tree_wy`` is the same WY/UT algebra as ``chunked_wy`` with
    the ancestor mask and path prefix sums, over the whole tree at once; it
    exists to pin the form the GPU computes.

``scalar_gate_recurrence`` / ``scalar_gate_wy``
    The scalar-gate variant (one log-decay per token and value head, the
    same for every key channel), the case in which the review thread of
    "Support TreeUpdateSolve kernel" weighs a per-key-head gram against a
    per-value-head one.  The definition is the recurrence with g broadcast
    over the key channels; ``scalar_gate_wy`` is the chunked form with the
    decay factored out of the dot products, so that one gram K K^T per key
    head serves all of its value heads.

``affine_map`` / ``segmented_forward``
    The chunk-parallel state scan.  Over any run of tokens the recurrence is
    an affine map of the state, S_end = M S_start + c, with M [dk, dk]
    depending only on (k, g, beta) and c the end state from a zero start.
    ``affine_map`` composes it token by token from the one-token map
    S -> (I - beta k k^T) diag(exp g) S + beta k v^T (the unrolled update of
    the first commit summary of the executorch page).  ``segmented_forward``
    cuts the sequence into segments of whole chunks, takes the maps of the
    middle segments, runs the first segment from h0, chains the maps to get
    every segment's start state, and runs the other segments from those
    starts: the order of work the GPU's segmented route follows.  The pages
    only name the chunked pieces; this split of the serial carry is derived
    from the algebra, and its result is the definition's.

Array layouts (numpy, C-contiguous):
    q, k [B, T, HK, dk]; v [B, T, HV, dv]; g [B, T, HV, dk]; beta [B, T, HV];
    h0 [B, HV, dk, dv] or None.  Returns (o [B, T, HV, dv], ht [B, HV, dk, dv]).
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None


def _open(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gdr_oracle_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp] + [ctypes.c_long] * 6 + [
        ctypes.c_int]
    lib.gdr_oracle_f64.restype = ctypes.c_int
    lib.gdr_oracle_default_threads.argtypes = []
    lib.gdr_oracle_default_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _open(_build.build())
    return _lib


def default_threads() -> int:
    """Number of host threads the oracle uses when ``threads`` is not given."""
    return int(_load().gdr_oracle_default_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def recurrence(q, k, v, g, beta, h0=None, threads=None, _lib_override=None):
    """fp64 sequential token recurrence (the oracle).  See module docstring.

    ``_lib_override`` lets the oracle's own tests run a deliberately broken
    build of gdr_oracle.c through the same pins (mutation testing)."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and v.shape[:2] == (B, T)
    assert g.shape == (B, T, HV, dk) and beta.shape == (B, T, HV)
    if h0 is not None:
        h0 = _f64(h0)
        assert h0.shape == (B, HV, dk, dv)
    out = np.zeros((B, T, HV, dv), dtype=np.float64)
    ht = np.zeros((B, HV, dk, dv), dtype=np.float64)
    lib = _load() if _lib_override is None else _lib_override
    rc = lib.gdr_oracle_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                            _ptr(out), _ptr(ht), B, T, HK, HV, dk, dv,
                            0 if threads is None else int(threads))
    if rc != 0:
        raise RuntimeError("gdr_oracle_f64 failed with status %d" % rc)
    return out, ht


def recurrence_heads(q, k, v, g, beta, h0, heads, threads=None):
    """Oracle on a subset of (b, hv) pairs.

    Heads are independent, so slicing the inputs down to one (b, hv) and its
    key head gives exactly that head's result.  Returns a dict
    {(b, hv): (o [T, dv], ht [dk, dv])}.
    """
    HK = q.shape[2]
    HV = v.shape[2]
    group = HV // HK
    res = {}
    for (b, hv) in heads:
        hk = hv // group
        sl = lambda x, h: x[b:b + 1, :, h:h + 1]
        o, ht = recurrence(sl(q, hk), sl(k, hk), sl(v, hv), sl(g, hv), beta[b:b + 1, :, hv:hv + 1],
                           None if h0 is None else h0[b:b + 1, hv:hv + 1], threads=threads)
        res[(b, hv)] = (o[0, :, 0], ht[0, 0])
    return res


def chunked_wy(q, k, v, g, beta, h0=None, chunk=64):
    """fp64 chunkwise WY/UT restatement of the same forward pass.

    Per (b, hv) and per chunk of L <= chunk tokens, with S0 the state at the
    chunk start and r, s local token indices:
      G       = inclusive prefix sum of g over the chunk, per key channel
      A[r,s]  = beta_r * sum_i k_ri k_si exp(G_ri - G_si)      (s < r, else 0)
      P[r,s]  = sum_i q_ri k_si exp(G_ri - G_si)                (s <= r, else 0)
      Kt      = exp(G) * k,   Qt = exp(G) * q,   Kh = exp(G_L - G) * k
      (I + A) U = diag(beta) (V - Kt S0)          (unit-lower triangular solve)
      O       = Qt S0 + P U
      S_next  = diag(exp(G_L)) S0 + Kh^T U
    The ragged final chunk (L < chunk) runs through the same code.
    """
    from scipy.linalg import solve_triangular

    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    group = HV // HK
    out = np.zeros((B, T, HV, dv))
    ht = np.zeros((B, HV, dk, dv))
    for b in range(B):
        for hv in range(HV):
            hk = hv // group
            S = np.zeros((dk, dv)) if h0 is None else _f64(h0)[b, hv].copy()
            for t0 in range(0, T, chunk):
                t1 = min(T, t0 + chunk)
                L = t1 - t0
                K = k[b, t0:t1, hk]          # [L, dk]
                Q = q[b, t0:t1, hk]
                V = v[b, t0:t1, hv]          # [L, dv]
                bet = beta[b, t0:t1, hv]     # [L]
                G = np.cumsum(g[b, t0:t1, hv], axis=0)   # [L, dk]
                causal = np.tril(np.ones((L, L)), 0)
                strict = np.tril(np.ones((L, L)), -1)
                # [r, s, i] = exp(G_ri - G_si) on s <= r; the exponent is masked
                # to -inf above the diagonal so it can never overflow there
                D = np.where(causal[:, :, None] > 0, G[:, None, :] - G[None, :, :], -np.inf)
                E = np.exp(D)
                A = bet[:, None] * np.einsum("ri,si,rsi->rs", K, K, E) * strict
                P = np.einsum("ri,si,rsi->rs", Q, K, E) * causal
                Kt = np.exp(G) * K
                Qt = np.exp(G) * Q
                Kh = np.exp(G[-1][None, :] - G) * K
                rhs = bet[:, None] * (V - Kt @ S)
                U = solve_triangular(np.eye(L) + A, rhs, lower=True, unit_diagonal=True)
                out[b, t0:t1, hv] = Qt @ S + P @ U
                S = np.exp(G[-1])[:, None] * S + Kh.T @ U
            ht[b, hv] = S
    return out, ht


def _check_parent(parent, B, T):
    parent = np.asarray(parent, dtype=np.int64).reshape(B, T)
    for b in range(B):
        for t in range(T):
            assert -1 <= parent[b, t] < t, "parents must precede their children"
    return parent


def _path(parent_b, t):
    """Root-to-t token indices (ancestors first, t last)."""
    path = []
    while t >= 0:
        path.append(t)
        t = parent_b[t]
    return path[::-1]


def tree_recurrence(q, k, v, g, beta, h0, parent, threads=None):
    """Tree verification by definition: o[b, t] is the output of the last
    token when the token recurrence runs over the root path of t (its
    ancestors from the root down, then t), starting from h0[b] (zeros if
    None).  parent [B, T] ints, parent[b, t] in [-1, t-1], -1 for a token
    whose parent is the state h0.  Returns o [B, T, HV, dv].

    All paths of a tree run as one batch of `recurrence`: a path shorter than
    the deepest is padded at its front with tokens of zero decay (g = 0) and
    beta = 0, which leave the state unchanged exactly (multiplied by
    exp(0) = 1 and added beta * ... = 0), and their outputs are discarded."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    parent = _check_parent(parent, B, T)
    out = np.zeros((B, T, HV, dv))
    for b in range(B):
        if T == 0:
            continue
        paths = [_path(parent[b], t) for t in range(T)]
        depth = max(len(p) for p in paths)
        qp = np.zeros((T, depth, HK, dk))
        kp = np.zeros((T, depth, HK, dk))
        vp = np.zeros((T, depth, HV, dv))
        gp = np.zeros((T, depth, HV, dk))
        bp = np.zeros((T, depth, HV))
        for t, p in enumerate(paths):
            off = depth - len(p)
            qp[t, off:] = q[b, p]
            kp[t, off:] = k[b, p]
            vp[t, off:] = v[b, p]
            gp[t, off:] = g[b, p]
            bp[t, off:] = beta[b, p]
        hp = None if h0 is None else np.repeat(_f64(h0)[b:b + 1], T, axis=0)
        o, _ = recurrence(qp, kp, vp, gp, bp, hp, threads=threads)
        out[b] = o[:, -1]
    return out


def tree_wy(q, k, v, g, beta, h0, parent):
    """The WY/UT form of tree verification, one solve over the whole tree.

    Per (b, hv), with anc(r) the strict ancestors of token r:
      G_r     = sum of g over the root path of r (inclusive), per channel
      A[r,s]  = beta_r * sum_i k_ri k_si exp(G_ri - G_si)      (s in anc(r))
      P[r,s]  = sum_i q_ri k_si exp(G_ri - G_si)                (s in anc(r) or s = r)
      Kt = exp(G) * k,  Qt = exp(G) * q
      (I + A) U = diag(beta) (V - Kt S0)     (unit lower triangular: parents first)
      O = Qt S0 + P U
    Returns o [B, T, HV, dv]."""
    from scipy.linalg import solve_triangular

    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    group = HV // HK
    parent = _check_parent(parent, B, T)
    out = np.zeros((B, T, HV, dv))
    for b in range(B):
        anc = np.zeros((T, T))
        for r in range(T):
            for s in _path(parent[b], r)[:-1]:
                anc[r, s] = 1.0
        path_or_self = anc + np.eye(T)
        for hv in range(HV):
            hk = hv // group
            S = np.zeros((dk, dv)) if h0 is None else _f64(h0)[b, hv]
            K, Q, V = k[b, :, hk], q[b, :, hk], v[b, :, hv]
            bet = beta[b, :, hv]
            G = np.zeros((T, dk))
            for r in range(T):
                G[r] = g[b, r, hv] + (G[parent[b, r]] if parent[b, r] >= 0 else 0.0)
            D = np.where(path_or_self[:, :, None] > 0, G[:, None, :] - G[None, :, :], -np.inf)
            E = np.exp(D)
            A = bet[:, None] * np.einsum("ri,si,rsi->rs", K, K, E) * anc
            P = np.einsum("ri,si,rsi->rs", Q, K, E) * path_or_self
            Kt = np.exp(G) * K
            Qt = np.exp(G) * Q
            rhs = bet[:, None] * (V - Kt @ S)
            U = solve_triangular(np.eye(T) + A, rhs, lower=True, unit_diagonal=True)
            out[b, :, hv] = Qt @ S + P @ U
    return out


def scalar_gate_recurrence(q, k, v, g, beta, h0=None, threads=None):
    """Scalar-gate forward by definition: g [B, T, HV] (one log-decay per
    token and value head) applied to every key channel, i.e. the recurrence
    with g repeated over dk.  Returns (o, ht)."""
    g = _f64(g)
    dk = np.asarray(q).shape[3]
    return recurrence(q, k, v, np.repeat(g[..., None], dk, axis=3), beta, h0, threads=threads)


def scalar_gate_wy(q, k, v, g, beta, h0=None, chunk=64):
    """Scalar-gate chunked form with the gram per key head.

    Per chunk of L tokens, with G the inclusive prefix of the scalar g of a
    value head and Gamma[r, s] = exp(G_r - G_s) (s <= r):
      KK = K K^T and QK = Q K^T, once per KEY head (shared by its G value heads)
      A = diag(beta) (KK * Gamma), strictly lower;  P = QK * Gamma, lower
      (I + A) U = diag(beta) (V - exp(G) K S0)
      O = exp(G) Q S0 + P U
      S_next = exp(G_L) S0 + (exp(G_L - G) K)^T U
    Returns (o [B, T, HV, dv], ht [B, HV, dk, dv])."""
    from scipy.linalg import solve_triangular

    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    group = HV // HK
    out = np.zeros((B, T, HV, dv))
    ht = np.zeros((B, HV, dk, dv))
    for b in range(B):
        S = {hv: (np.zeros((dk, dv)) if h0 is None else _f64(h0)[b, hv].copy())
             for hv in range(HV)}
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            L = t1 - t0
            for hk in range(HK):
                K = k[b, t0:t1, hk]
                Q = q[b, t0:t1, hk]
                KK = K @ K.T            # the key-head gram, shared below
                QK = Q @ K.T
                for hv in range(hk * group, (hk + 1) * group):
                    G = np.cumsum(g[b, t0:t1, hv])                      # [L]
                    diff = G[:, None] - G[None, :]
                    Gamma = np.exp(np.where(np.tril(np.ones((L, L))) > 0, diff, -np.inf))
                    bet = beta[b, t0:t1, hv]
                    A = bet[:, None] * KK * Gamma * np.tril(np.ones((L, L)), -1)
                    P = QK * Gamma
                    V = v[b, t0:t1, hv]
                    eG = np.exp(G)[:, None]
                    rhs = bet[:, None] * (V - (eG * K) @ S[hv])
                    U = solve_triangular(np.eye(L) + A, rhs, lower=True, unit_diagonal=True)
                    out[b, t0:t1, hv] = (eG * Q) @ S[hv] + P @ U
                    S[hv] = np.exp(G[-1]) * S[hv] + (np.exp(G[-1] - G)[:, None] * K).T @ U
        for hv in range(HV):
            ht[b, hv] = S[hv]
    return out, ht


def segment_bounds(T, chunk, segments):
    """Token ranges [t0, t1) of at most ``segments`` segments of whole chunks:
    ceil(chunks / segments) chunks each, the last one shorter (and ragged
    when T is not a multiple of the chunk).  No segment is empty."""
    nch = -(-T // chunk)
    if nch == 0:
        return []
    per = -(-nch // max(1, segments))
    return [(c * chunk, min(T, (c + per) * chunk)) for c in range(0, nch, per)]


def affine_map(k, v, g, beta, t0, t1):
    """The map of tokens t0 .. t1-1 on the state of every (b, hv):
    S_end = M S_start + c, M [B, HV, dk, dk], c [B, HV, dk, dv], composed
    one token at a time: with a = exp(g_t) per key channel,
      S -> (I - beta_t k_t k_t^T) diag(a) S + beta_t k_t v_t^T
    (decay, then the delta update with the prediction (diag(a) S)^T k_t)."""
    k, v, g, beta = (_f64(x) for x in (k, v, g, beta))
    B, _, HK, dk = k.shape
    HV, dv = v.shape[2], v.shape[3]
    group = HV // HK
    M = np.zeros((B, HV, dk, dk))
    c = np.zeros((B, HV, dk, dv))
    eye = np.eye(dk)
    for b in range(B):
        for hv in range(HV):
            hk = hv // group
            Mb, cb = eye.copy(), np.zeros((dk, dv))
            for t in range(t0, t1):
                kt = k[b, t, hk]
                bt = beta[b, t, hv]
                A = (eye - bt * np.outer(kt, kt)) * np.exp(g[b, t, hv])[None, :]
                Mb = A @ Mb
                cb = A @ cb + bt * np.outer(kt, v[b, t, hv])
            M[b, hv], c[b, hv] = Mb, cb
    return M, c


def segmented_forward(q, k, v, g, beta, h0=None, segments=3, chunk=64):
    """The chunk-parallel scan in the GPU's order of work; returns (o, ht).

    With segments p = 0 .. P-1 (``segment_bounds``) and S_p the state at the
    start of segment p:
      1. (M_p, c_p) = affine_map over segment p, for p = 1 .. P-2
      2. segment 0 runs from S_0 = h0 (or 0): its outputs and S_1
      3. S_{p+1} = M_p S_p + c_p for p = 1 .. P-2
      4. segment p >= 1 runs from S_p: its outputs (and, last, ht)
    The runs are the token recurrence."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    bounds = segment_bounds(T, chunk, segments)
    start = np.zeros((B, HV, dk, dv)) if h0 is None else _f64(h0).copy()
    if not bounds:
        return np.zeros((B, 0, HV, dv)), start
    maps = {p: affine_map(k, v, g, beta, *bounds[p]) for p in range(1, len(bounds) - 1)}
    out = np.zeros((B, T, HV, dv))

    def run(p, S):
        t0, t1 = bounds[p]
        sl = slice(t0, t1)
        o, S_end = recurrence(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S)
        out[:, sl] = o
        return S_end

    S = run(0, start)
    starts = [S]
    for p in range(1, len(bounds) - 1):
        M, c = maps[p]
        S = np.einsum("bhij,bhjv->bhiv", M, S) + c
        starts.append(S)
    ht = S if len(bounds) == 1 else None
    for p in range(1, len(bounds)):
        ht = run(p, starts[p - 1])
    return out, ht
