"""GPU parity of the scalar-gate variant (g [B, T, HV]: one log-decay per
token and value head) against the oracle's definition, on every route:
single-token decode, tensor-core prefill (fast and exact paths), CUDA-core
chunks, packed variable-length batches and trees."""
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_GENERIC, gdr_device_check, gdr_forward,
                                           gdr_forward_tree, gdr_forward_varlen)
from channelwise_gated_delta_gb300.inputs import draw, draw_parents, pack, to_f64
from tests.parity_util import assert_close, to_cuda

pytestmark = pytest.mark.gpu


def ref(d):
    return oracle.scalar_gate_recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))


def check(d, chunk=64, flags=0):
    c = to_cuda(d)
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=chunk,
                          flags=flags)
    gdr_device_check()
    ro, rh = ref(d)
    assert_close("o", out, ro, d["q"].dtype)
    assert_close("ht", ht, rh, d["q"].dtype)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("h0", [True, False])
def test_tensor_core_route(T, h0):
    check(draw(2, T, 2, 4, 128, 128, dtype=torch.bfloat16, h0=h0, seed=T, scalar_gate=True))


@pytest.mark.parametrize("g_mu,beta_mu", [(-3.0, 2.0), (3.0, 0.0), (1.5, 0.0)])
def test_tensor_core_decay_regimes(g_mu, beta_mu):
    """Slow decay with beta near 1 (the conditioning stress), and decays of
    ~3 and ~1.7 nats per token, which leave the 80-nat range inside a chunk
    (the exact path) or near its edge."""
    check(draw(2, 300, 1, 2, 128, 128, dtype=torch.bfloat16, seed=7, g_mu=g_mu, beta_mu=beta_mu,
               beta_sigma=0.5, scalar_gate=True))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv,chunk", [(32, 32, 16), (64, 128, 32), (128, 64, 64),
                                         (128, 128, 64)])
def test_cuda_core_route(dtype, dk, dv, chunk):
    check(draw(2, 97, 2, 4, dk, dv, dtype=dtype, seed=dk + dv, scalar_gate=True), chunk,
          flags=GDR_FLAG_FORCE_GENERIC)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode(dtype):
    check(draw(16, 1, 4, 8, 128, 128, dtype=dtype, seed=3, scalar_gate=True))


def test_decode_in_place_model_shape():
    d = draw(64, 1, 16, 32, 128, 128, dtype=torch.bfloat16, seed=4, scalar_gate=True)
    c = to_cuda(d)
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], ht=c["h0"])
    gdr_device_check()
    ro, rh = ref(d)
    assert_close("o", out, ro, torch.bfloat16)
    assert_close("ht", ht, rh, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_varlen(dtype):
    gen = torch.Generator()
    gen.manual_seed(5)
    seqs = [draw(1, L, 2, 4, 128, 128, dtype=dtype, generator=gen, scalar_gate=True)
            for L in (1, 33, 0, 64, 65, 150, 1)]
    packed, cu = pack(seqs)
    c = to_cuda(packed)
    out, ht = gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, h0=c["h0"])
    gdr_device_check()
    for n, d in enumerate(seqs):
        ro, rh = ref(d)
        assert_close("o[%d]" % n, out[:, cu[n]:cu[n + 1]], ro, dtype)
        assert_close("ht[%d]" % n, ht[n:n + 1], rh, dtype)


def test_tree():
    d = draw(2, 40, 2, 4, 128, 128, dtype=torch.bfloat16, seed=6, scalar_gate=True)
    par = draw_parents(2, 40, "random", seed=6)
    c = to_cuda(d)
    out = gdr_forward_tree(c["q"], c["k"], c["v"], c["g"], c["beta"], par, h0=c["h0"])
    gdr_device_check()
    dk = d["q"].shape[3]
    g_full = to_f64(d["g"])[..., None].repeat(dk, axis=3)
    want = oracle.tree_recurrence(to_f64(d["q"]), to_f64(d["k"]), to_f64(d["v"]), g_full,
                                  to_f64(d["beta"]), to_f64(d["h0"]), par.numpy())
    assert_close("o", out, want, torch.bfloat16)


def test_scalar_gate_equals_broadcast_channelwise_on_cuda_cores():
    """On the CUDA-core route a scalar gate reads the same value for every
    channel: the same bits as the channelwise path given g repeated over dk."""
    d = draw(2, 70, 1, 2, 64, 64, dtype=torch.float32, seed=8, scalar_gate=True)
    c = to_cuda(d)
    gs, hs = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=32,
                         flags=GDR_FLAG_FORCE_GENERIC)
    g_full = c["g"][..., None].expand(-1, -1, -1, 64).contiguous()
    gc, hc = gdr_forward(c["q"], c["k"], c["v"], g_full, c["beta"], c["h0"], chunk=32,
                         flags=GDR_FLAG_FORCE_GENERIC)
    gdr_device_check()
    assert torch.equal(gs, gc) and torch.equal(hs, hc)
