"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle,
element by element on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_CHUNKED, GDR_FLAG_FORCE_GENERIC,
                                           gdr_device_check, gdr_forward)
from channelwise_gated_delta_gb300.inputs import WORKLOADS, draw, draw_workload, to_f64
from tests.parity_util import assert_close, to_cuda

pytestmark = pytest.mark.gpu


def run_gpu(d, chunk, flags=0, inplace=False, store_ht=True):
    c = to_cuda(d)
    ht = c["h0"] if (inplace and c["h0"] is not None) else None
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], ht=ht, chunk=chunk,
                          flags=flags, store_ht=store_ht)
    gdr_device_check()
    return out, ht


def run_oracle(d):
    return oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                             to_f64(d["h0"]))


def check(d, chunk, flags=0, inplace=False):
    dtype = d["q"].dtype
    ref_o, ref_h = run_oracle(d)
    out, ht = run_gpu(d, chunk, flags=flags, inplace=inplace)
    assert_close("o", out, ref_o, dtype)
    assert_close("ht", ht, ref_h, dtype)


# ------------------------------------------------------------ named workloads
def test_tiny():
    w = WORKLOADS["tiny"]
    check(draw_workload(w), w.chunk)


def test_decode_b64_in_place():
    w = WORKLOADS["decode_b64"]
    d = draw_workload(w)
    check(d, w.chunk, inplace=True)


def test_ragged_b8_each_sequence():
    w = WORKLOADS["ragged_b8"]
    for d in draw_workload(w):
        check(d, w.chunk)


def test_prefill_t4k_full():
    w = WORKLOADS["prefill_t4k"]
    check(draw_workload(w), w.chunk)


@pytest.mark.slow
def test_prefill_t16k_all_heads():
    """Full-size long prefill in the launch configuration the benchmark times,
    every (batch, value head) of o and ht against the oracle (one batch
    element at a time to bound the oracle's memory)."""
    w = WORKLOADS["prefill_t16k"]
    d = draw_workload(w)
    out, ht = run_gpu(d, w.chunk)
    for b in range(w.B):
        one = lambda x: to_f64(x[b:b + 1])
        ro, rh = oracle.recurrence(*(one(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                   one(d["h0"]))
        assert_close("o[%d]" % b, out[b:b + 1], ro, w.dtype)
        assert_close("ht[%d]" % b, ht[b:b + 1], rh, w.dtype)


@pytest.mark.slow
def test_prefill_t16k_f32_all_heads():
    """The long-prefill stress recipe at full size with float32 q/k/v (the
    chunk prep and the state scan on the tensor cores, BF16x3), every
    (batch, value head) of o and ht against the oracle at the float32 bound."""
    w = WORKLOADS["prefill_t16k"]
    d = draw(w.B, w.T, w.HK, w.HV, w.dk, w.dv, dtype=torch.float32, h0=True, seed=31,
             g_mu=w.g_mu, g_sigma=w.g_sigma, beta_mu=w.beta_mu, beta_sigma=w.beta_sigma)
    out, ht = run_gpu(d, w.chunk)
    for b in range(w.B):
        one = lambda x: to_f64(x[b:b + 1])
        ro, rh = oracle.recurrence(*(one(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                   one(d["h0"]))
        assert_close("o[%d]" % b, out[b:b + 1], ro, torch.float32)
        assert_close("ht[%d]" % b, ht[b:b + 1], rh, torch.float32)


@pytest.mark.slow
def test_prefill_t16k_f32_few_heads_segmented():
    """16384 float32 tokens on four value heads: the automatic choice cuts
    the tensor-core scan into many segments (the maps chained over ~20
    segments of the stress recipe); every head against the oracle."""
    w = WORKLOADS["prefill_t16k"]
    d = draw(1, w.T, 2, 4, w.dk, w.dv, dtype=torch.float32, h0=True, seed=32,
             g_mu=w.g_mu, g_sigma=w.g_sigma, beta_mu=w.beta_mu, beta_sigma=w.beta_sigma)
    check(d, w.chunk)


# ------------------------------------------------------------ shapes and edges
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128), (32, 128)])
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_shapes_and_chunks(dtype, dk, dv, chunk):
    d = draw(2, 83, 2, 4, dk, dv, dtype=dtype, seed=dk + dv + chunk)
    check(d, chunk)


@pytest.mark.parametrize("T", [2, 15, 16, 17, 31, 33, 63, 64, 65, 97])
def test_ragged_lengths(T):
    check(draw(1, T, 1, 2, 64, 64, dtype=torch.float32, seed=T), 16)


@pytest.mark.parametrize("HK,HV", [(1, 1), (1, 4), (2, 4), (4, 4), (3, 6)])
def test_head_groupings(HK, HV):
    check(draw(2, 40, HK, HV, 32, 64, dtype=torch.bfloat16, seed=HK * 10 + HV), 32)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_no_initial_state(dtype):
    check(draw(2, 50, 2, 4, 64, 64, dtype=dtype, h0=False, seed=5), 16)


@pytest.mark.parametrize("T", [1, 70])
def test_in_place_state(T):
    check(draw(2, T, 2, 4, 64, 32, dtype=torch.float32, seed=6), 32, inplace=True)


def test_no_final_state():
    d = draw(1, 30, 1, 2, 32, 32, seed=7)
    ref_o, _ = run_oracle(d)
    out, ht = run_gpu(d, 16, store_ht=False)
    assert ht is None
    assert_close("o", out, ref_o, torch.float32)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_equals_forced_chunked(dtype):
    """T == 1 routed to the decode kernel and forced through the chunked
    prefill give the same result (both checked against the oracle too)."""
    d = draw(4, 1, 2, 4, 128, 128, dtype=dtype, seed=8)
    o1, h1 = run_gpu(d, 64)
    o2, h2 = run_gpu(d, 64, flags=GDR_FLAG_FORCE_CHUNKED)
    ref_o, ref_h = run_oracle(d)
    for o, h in ((o1, h1), (o2, h2)):
        assert_close("o", o, ref_o, dtype)
        assert_close("ht", h, ref_h, dtype)
    assert_close("o decode vs chunked", o1, to_f64(o2), dtype)


def test_empty_sequence_copies_state():
    d = draw(2, 0, 1, 2, 32, 32, seed=9)
    out, ht = run_gpu(d, 16)
    assert out.shape[1] == 0
    assert torch.equal(ht.cpu(), d["h0"])
    d0 = draw(2, 0, 1, 2, 32, 32, seed=9, h0=False)
    out, ht = run_gpu(d0, 16)
    assert torch.count_nonzero(ht).item() == 0


def test_empty_batch():
    d = draw(0, 5, 1, 2, 32, 32, seed=10)
    out, ht = run_gpu(d, 16)
    assert out.numel() == 0 and ht.numel() == 0


def test_strong_decay():
    """|g| ~ 6 per token: cumulative decay over a chunk far below float32's
    range; every exponent the kernels take stays <= 0."""
    d = draw(1, 64, 1, 2, 32, 32, dtype=torch.float32, seed=11, g_mu=6.0, g_sigma=0.5)
    check(d, 64)


@pytest.mark.parametrize("g_mu", [0.6, 1.0, 1.3, 1.6])
def test_tensor_core_decay_near_range_limit(g_mu):
    """Channelwise decays of ~1-2 nats per token: the tensor-core kernel's
    reference-row factors reach e^{+-50} and beyond, some chunks take the
    exact path and neighbours of both kinds meet; the carry between chunks
    must not lose the state to underflow."""
    d = draw(2, 320, 1, 2, 128, 128, dtype=torch.bfloat16, seed=13, g_mu=g_mu)
    check(d, 64)


def test_resume_matches_single_call():
    d = draw(1, 100, 1, 2, 64, 64, dtype=torch.float32, seed=12)
    c = to_cuda(d)
    o_all, h_all = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=32)
    sl = lambda x, a, b: x[:, a:b].clone()  # fresh, aligned allocations
    oa, ha = gdr_forward(*(sl(c[n], 0, 37) for n in ("q", "k", "v", "g", "beta")), c["h0"], chunk=32)
    ob, hb = gdr_forward(*(sl(c[n], 37, 100) for n in ("q", "k", "v", "g", "beta")), ha, chunk=32)
    ref_o, ref_h = run_oracle(d)
    assert_close("o resumed", torch.cat([oa, ob], dim=1), ref_o, torch.float32)
    assert_close("ht resumed", hb, ref_h, torch.float32)
    assert_close("o single", o_all, ref_o, torch.float32)
