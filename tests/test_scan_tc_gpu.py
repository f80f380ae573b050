"""The state scan of the chunked prefill on the tensor cores (gdr_chunk_scan_tc:
tcgen05 products in BF16x3, the state in tensor memory), the route of float32
q/k/v and of the shapes the fused bf16 kernel does not take: parity with the
fp64 oracle at the float32 bound, agreement with the CUDA-core scan
(GDR_FLAG_FORCE_GENERIC), and the route actually taken."""
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_GENERIC, GDR_FLAG_NO_SEGMENTS,
                                           gdr_device_check, gdr_forward, gdr_forward_varlen,
                                           gdr_trace_enable, gdr_trace_read)
from channelwise_gated_delta_gb300.inputs import WORKLOADS, draw, draw_workload, pack, to_f64
from tests.parity_util import assert_close, to_cuda

pytestmark = pytest.mark.gpu


def forward(d, chunk, flags=0):
    c = to_cuda(d)
    gdr_trace_enable(True)
    try:
        out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=chunk,
                              flags=flags | GDR_FLAG_NO_SEGMENTS)
        gdr_device_check()
        tr = gdr_trace_read()
    finally:
        gdr_trace_enable(False)
    return out, ht, tr


def check(d, chunk):
    ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d["h0"]))
    out, ht, tr = forward(d, chunk)
    assert "gdr_chunk_scan_tc" in tr and "gdr_chunk_scan" not in tr, tr
    assert_close("o", out, ref_o, d["q"].dtype)
    assert_close("ht", ht, ref_h, d["q"].dtype)
    return out, ht


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (32, 32), (32, 128)])
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_f32_shapes_and_chunks(dk, dv, chunk):
    check(draw(2, 150, 2, 4, dk, dv, dtype=torch.float32, seed=500 + dk + dv + chunk), chunk)


def test_tiny_workload():
    w = WORKLOADS["tiny"]
    check(draw_workload(w), w.chunk)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129, 1000])
def test_f32_lengths(T):
    """T = 1 forced through the chunked route; ragged last chunks."""
    d = draw(1, T, 2, 4, 128, 128, dtype=torch.float32, seed=510 + T)
    ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d["h0"]))
    from channelwise_gated_delta_gb300 import GDR_FLAG_FORCE_CHUNKED
    out, ht, tr = forward(d, 64, flags=GDR_FLAG_FORCE_CHUNKED)
    assert "gdr_chunk_scan_tc" in tr, tr
    assert_close("o", out, ref_o, torch.float32)
    assert_close("ht", ht, ref_h, torch.float32)


def test_conditioning_stress_f32():
    """beta near 1 and slow decay (||A|| ~ 1 within chunks) over 2048 tokens
    at the model's head shape, float32."""
    check(draw(1, 2048, 2, 4, 128, 128, dtype=torch.float32, seed=520, g_mu=-3.0,
               beta_mu=2.0, beta_sigma=0.5), 64)


@pytest.mark.parametrize("g_mu", [6.0, 2.0])
def test_strong_decay_f32(g_mu):
    check(draw(1, 300, 1, 2, 128, 128, dtype=torch.float32, seed=521, g_mu=g_mu, g_sigma=0.5), 64)


def test_no_initial_state_and_no_final_state():
    d = draw(2, 200, 1, 2, 128, 128, dtype=torch.float32, h0=False, seed=522)
    ref_o, _ = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")), None)
    c = to_cuda(d)
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], None, chunk=64,
                          store_ht=False)
    gdr_device_check()
    assert ht is None
    assert_close("o", out, ref_o, torch.float32)


def test_bf16_inputs_off_the_fused_shape():
    """bf16 q/k/v with dk = 64: the chunked route with the tensor-core scan."""
    check(draw(2, 300, 2, 4, 64, 128, dtype=torch.bfloat16, seed=523), 64)


def test_agrees_with_cuda_core_scan():
    """Same records arithmetic, the scan on CUDA cores (3xTF32) and on the
    tensor cores (BF16x3): well inside the float32 bound of each other."""
    d = draw(2, 700, 2, 4, 128, 128, dtype=torch.float32, seed=524)
    o1, h1, _ = forward(d, 64)
    o2, h2, tr = forward(d, 64, flags=GDR_FLAG_FORCE_GENERIC)
    assert "gdr_chunk_scan" in tr and "gdr_chunk_scan_tc" not in tr, tr
    assert (o1 - o2).abs().max().item() <= 2e-4 * o2.abs().max().item()
    assert (h1 - h2).abs().max().item() <= 2e-4 * h2.abs().max().item()


def test_ragged_b8_packed_f32():
    """The ragged workload (lengths 1 .. 512, float32) through the packed entry:
    the prefill sequences on the tensor-core scan, each against the oracle."""
    w = WORKLOADS["ragged_b8"]
    seqs = draw_workload(w)
    packed, cu = pack(seqs)
    c = to_cuda(packed)
    gdr_trace_enable(True)
    try:
        out, ht = gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, h0=c["h0"],
                                     chunk=w.chunk)
        gdr_device_check()
        tr = gdr_trace_read()
    finally:
        gdr_trace_enable(False)
    assert "gdr_chunk_scan_tc" in tr, tr
    for n, d in enumerate(seqs):
        ref_o, ref_h = oracle.recurrence(*(to_f64(d[x]) for x in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))
        assert_close("o[%d]" % n, out[:, cu[n]:cu[n + 1]], ref_o, torch.float32)
        assert_close("ht[%d]" % n, ht[n:n + 1], ref_h, torch.float32)
