"""GPU parity of tree verification (gdr_forward_tree) against the oracle's
definition: each token's output is the recurrence run along its root path."""
import numpy as np
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_CHUNKED, GDR_FLAG_FORCE_GENERIC,
                                           GDR_FLAG_TREE_BLOCKED,
                                           GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD, GdrError,
                                           gdr_device_check,
                                           gdr_forward, gdr_forward_tree, gdr_trace_enable,
                                           gdr_trace_read)
from channelwise_gated_delta_gb300.inputs import draw, draw_parents, to_f64
from tests.parity_util import assert_close, to_cuda

pytestmark = pytest.mark.gpu


def run_tree(d, parent, flags=0):
    c = to_cuda(d)
    out = gdr_forward_tree(c["q"], c["k"], c["v"], c["g"], c["beta"], parent, h0=c["h0"],
                           flags=flags)
    gdr_device_check()
    return out


def check(d, parent, flags=0):
    ref = oracle.tree_recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                 to_f64(d["h0"]), parent.numpy())
    assert_close("o", run_tree(d, parent, flags), ref, d["q"].dtype)


# --------------------------- tensor-core route (bf16, dk = dv = 128)
@pytest.mark.parametrize("kind", ["random", "beam", "star", "chain"])
@pytest.mark.parametrize("T", [1, 5, 16, 17, 33, 64])
def test_tc_tree_shapes(kind, T):
    d = draw(2, T, 2, 4, 128, 128, dtype=torch.bfloat16, seed=100 + T)
    check(d, draw_parents(2, T, kind, seed=T))


def test_tc_tree_no_initial_state():
    d = draw(3, 48, 1, 2, 128, 128, dtype=torch.bfloat16, h0=False, seed=101)
    check(d, draw_parents(3, 48, "random", seed=101))


@pytest.mark.parametrize("kind", ["chain", "random"])
def test_tc_tree_strong_decay(kind):
    """|g| ~ 3 per token: a 64-deep chain decays by ~190 nats (the exact
    path), a random tree's shallow paths stay in range (the fast path)."""
    d = draw(2, 64, 1, 2, 128, 128, dtype=torch.bfloat16, seed=102, g_mu=3.0)
    check(d, draw_parents(2, 64, kind, seed=102))


def test_tc_and_cuda_core_routes_agree():
    d = draw(4, 64, 2, 4, 128, 128, dtype=torch.bfloat16, seed=103)
    par = draw_parents(4, 64, "beam", seed=103, branching=3)
    tc = run_tree(d, par).float()
    cc = run_tree(d, par, flags=GDR_FLAG_FORCE_GENERIC).float()
    assert (tc - cc).abs().max().item() <= 2e-2 * cc.abs().max().item()


@pytest.mark.parametrize("kind", ["random", "beam", "star", "chain"])
@pytest.mark.parametrize("T", [1, 5, 16, 17, 33, 64])
def test_tree_shapes(kind, T):
    d = draw(2, T, 2, 4, 64, 64, dtype=torch.float32, seed=T)
    check(d, draw_parents(2, T, kind, seed=T))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_tree_dims_and_dtypes(dtype, dk, dv):
    d = draw(2, 40, 1, 2, dk, dv, dtype=dtype, seed=dk + dv)
    check(d, draw_parents(2, 40, "random", seed=dk))


def test_tree_no_initial_state_grouped_heads():
    d = draw(3, 24, 2, 6, 64, 64, dtype=torch.float32, h0=False, seed=11)
    check(d, draw_parents(3, 24, "beam", seed=11, branching=2))


def test_tree_verify_shape():
    """A draft-tree verify step at model shapes: 8 trees of 64 tokens,
    HK = 16, HV = 32, dk = dv = 128, bf16, with an initial state."""
    d = draw(8, 64, 16, 32, 128, 128, dtype=torch.bfloat16, seed=12)
    check(d, draw_parents(8, 64, "beam", seed=12, branching=4))


def test_tree_slow_decay_beta_near_one():
    """The conditioning stress recipe (beta near 1, slow decay) on a deep tree."""
    d = draw(2, 64, 1, 2, 128, 128, dtype=torch.float32, seed=13, g_mu=-3.0, beta_mu=2.0,
             beta_sigma=0.5)
    check(d, draw_parents(2, 64, "random", seed=13))


@pytest.mark.parametrize("T,chunk", [(16, 16), (30, 32), (64, 64)])
def test_chain_tree_equals_chunked_sequence(T, chunk):
    """A chain is a sequence: the tree route and the CUDA-core chunked route
    over one chunk agree to float32 rounding (they factor the decay around
    different reference rows: the tree's start and the chunk's middle)."""
    d = draw(2, T, 1, 2, 64, 64, dtype=torch.float32, seed=14)
    c = to_cuda(d)
    tree = gdr_forward_tree(c["q"], c["k"], c["v"], c["g"], c["beta"],
                            draw_parents(2, T, "chain"), h0=c["h0"])
    seq, _ = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=chunk,
                         flags=GDR_FLAG_FORCE_CHUNKED | GDR_FLAG_FORCE_GENERIC)
    gdr_device_check()
    assert (tree - seq).abs().max().item() <= 1e-5 * seq.abs().max().item()


def test_bad_trees_rejected():
    d = to_cuda(draw(1, 4, 1, 1, 32, 32, seed=15))
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
    with pytest.raises(GdrError) as e:
        gdr_forward_tree(*args, [[-1, 0, 2, 0]], h0=d["h0"])   # parent not before child
    assert e.value.status == 2
    with pytest.raises(GdrError) as e:
        gdr_forward_tree(*args, [[-1, 0, -2, 0]], h0=d["h0"])  # below -1
    assert e.value.status == 2
    big = to_cuda(draw(1, 513, 1, 1, 32, 32, seed=16))
    with pytest.raises(GdrError) as e:
        gdr_forward_tree(big["q"], big["k"], big["v"], big["g"], big["beta"],
                         draw_parents(1, 513, "chain"))
    assert e.value.status == 3


# --------------------------- blocked solve: trees of up to 512 tokens
def oracle_tree(d, parent, kind):
    args = [to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")]
    scalar = d["g"].dim() == 3
    if kind == "chain":
        # a chain's root paths are the prefixes of one sequence
        rec = oracle.scalar_gate_recurrence if scalar else oracle.recurrence
        return rec(*args, to_f64(d["h0"]))[0]
    if scalar:  # the definition on a channelwise copy of the gate
        args[3] = np.repeat(args[3][..., None], args[0].shape[-1], axis=-1)
    return oracle.tree_recurrence(*args, to_f64(d["h0"]), parent.numpy())


def check_blocked(d, kind, seed, flags=0, branching=3):
    B, T = d["q"].shape[:2]
    par = draw_parents(B, T, kind, seed=seed, branching=branching)
    c = to_cuda(d)
    gdr_trace_enable(True)
    try:
        out = gdr_forward_tree(c["q"], c["k"], c["v"], c["g"], c["beta"], par, h0=c["h0"],
                               flags=flags)
        gdr_device_check()
        tr = gdr_trace_read()
    finally:
        gdr_trace_enable(False)
    assert "gdr_tree_solve_kernel" in tr and "gdr_tree_gram_kernel" in tr, tr
    assert_close("o", out, oracle_tree(d, par, kind), d["q"].dtype)
    return out


@pytest.mark.parametrize("kind", ["random", "beam", "chain"])
@pytest.mark.parametrize("B,T", [(1, 65), (8, 128), (1, 256), (8, 512), (1, 512)])
def test_blocked_tree_shapes(kind, B, T):
    check_blocked(draw(B, T, 1, 2, 128, 128, dtype=torch.bfloat16, seed=200 + T + B), kind, T)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (32, 32), (128, 64)])
@pytest.mark.parametrize("kind", ["random", "chain"])
def test_blocked_tree_f32(dk, dv, kind):
    """float32 q/k/v: bf16 pairs hi + lo, at the float32 bound."""
    check_blocked(draw(2, 200, 1, 2, dk, dv, dtype=torch.float32, seed=210 + dk + dv), kind, dk)


def test_blocked_tree_f32_full_size():
    check_blocked(draw(1, 512, 1, 2, 128, 128, dtype=torch.float32, seed=215), "random", 5)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("kind", ["random", "chain"])
def test_blocked_tree_scalar_gate(dtype, kind):
    """The gram once per key head, shared by its two value heads (the
    default), and once per value head: both at the oracle's bound, and the
    same up to the order of float additions."""
    d = draw(2, 300, 2, 4, 128, 128, dtype=dtype, seed=220, scalar_gate=True)
    per_kh = check_blocked(d, kind, 220)
    per_hv = check_blocked(d, kind, 220, flags=GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD)
    assert torch.equal(per_kh, per_hv)


def test_blocked_tree_no_initial_state_grouped_heads():
    check_blocked(draw(2, 150, 2, 6, 64, 64, dtype=torch.bfloat16, h0=False, seed=221),
                  "beam", 221, branching=2)


@pytest.mark.parametrize("kind,g_mu", [("chain", 6.0), ("chain", 3.0), ("random", 6.0),
                                       ("beam", 3.0)])
def test_blocked_tree_strong_decay(kind, g_mu):
    """About 6 nats a token: 16-token blocks of a chain spread past 60 nats
    and take one pass per row; 3 nats: factored blocks near the limit."""
    check_blocked(draw(2, 130, 1, 2, 128, 128, dtype=torch.bfloat16, seed=222, g_mu=g_mu,
                       g_sigma=0.5), kind, 222)


def test_blocked_tree_slow_decay_beta_near_one():
    """The conditioning stress recipe (beta near 1, slow decay) on a deep tree."""
    check_blocked(draw(2, 400, 1, 2, 128, 128, dtype=torch.float32, seed=223, g_mu=-3.0,
                       beta_mu=2.0, beta_sigma=0.5), "random", 223)


@pytest.mark.parametrize("kind", ["random", "beam", "star", "chain"])
@pytest.mark.parametrize("T", [1, 5, 17, 64])
def test_blocked_route_forced_on_one_chunk_trees(kind, T):
    """GDR_FLAG_TREE_BLOCKED at T <= 64: parity with the oracle, and agreement
    with the one-chunk tensor-core route."""
    d = draw(2, T, 2, 4, 128, 128, dtype=torch.bfloat16, seed=230 + T)
    out = check_blocked(d, kind, T, flags=GDR_FLAG_TREE_BLOCKED)
    ref = run_tree(d, draw_parents(2, T, kind, seed=T)).float()
    assert (out.float() - ref).abs().max().item() <= 2e-2 * ref.abs().max().item()


def test_blocked_tree_verify_shape():
    """Model shapes: 8 trees of 512 draft tokens, HK = 16, HV = 32, dk = dv = 128."""
    d = draw(8, 512, 16, 32, 128, 128, dtype=torch.bfloat16, seed=240)
    check_blocked(d, "beam", 240, branching=4)
