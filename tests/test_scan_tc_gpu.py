"""The state scan of the chunked prefill on the tensor cores (gdr_chunk_scan_tc:
tcgen05 products in BF16x3, the state in tensor memory), the route of float32
q/k/v and of the shapes the fused bf16 kernel does not take: parity with the
fp64 oracle at the float32 bound, agreement with the CUDA-core scan
(GDR_FLAG_FORCE_GENERIC), the route actually taken, and the same scan cut
into segments (forced and automatic, dense and packed, with and without
states, in place)."""
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_GENERIC, GDR_FLAG_NO_SEGMENTS,
                                           gdr_device_check, gdr_flag_segments, gdr_forward,
                                           gdr_forward_varlen, gdr_trace_enable, gdr_trace_read)
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


# ------------------------------------------- the segmented scan on this route
def forward_seg(d, chunk, flags, inplace=False, store_ht=True):
    c = to_cuda(d)
    ht = c["h0"] if (inplace and c["h0"] is not None) else None
    gdr_trace_enable(True)
    try:
        out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], ht=ht,
                              chunk=chunk, flags=flags, store_ht=store_ht)
        gdr_device_check()
        tr = gdr_trace_read()
    finally:
        gdr_trace_enable(False)
    return out, ht, tr


def check_seg(d, chunk, segments, inplace=False):
    """Forced segments against the fp64 oracle at the float32 bound; the
    launches are the prep, the two scan waves, the set-up and (three or more
    segments) the combine."""
    ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d["h0"]))
    out, ht, tr = forward_seg(d, chunk, gdr_flag_segments(segments), inplace=inplace)
    assert tr["gdr_chunk_scan_tc"][0] == 2, tr
    eff = len(oracle.segment_bounds(d["q"].shape[1], chunk, segments))
    assert ("gdr_segment_combine" in tr) == (eff >= 3), tr
    assert_close("o", out, ref_o, d["q"].dtype)
    assert_close("ht", ht, ref_h, d["q"].dtype)
    return out, ht


@pytest.mark.parametrize("segments", [2, 3, 5])
@pytest.mark.parametrize("chunk", [16, 64])
def test_segmented_scan_forced(segments, chunk):
    check_seg(draw(2, 1000, 2, 4, 128, 128, dtype=torch.float32, seed=530 + segments + chunk),
              chunk, segments)


def test_segmented_scan_many_segments_ragged():
    """Eleven segments of one 32-token chunk and a ragged 8-token tail."""
    check_seg(draw(1, 328, 1, 2, 128, 128, dtype=torch.float32, seed=540), 32, 11)


def test_segmented_scan_conditioning_stress():
    """Slow decay and beta near 1 over 2048 tokens: the maps M of the middle
    segments carry the state almost undamped."""
    check_seg(draw(1, 2048, 2, 4, 128, 128, dtype=torch.float32, seed=541, g_mu=-3.0,
                   beta_mu=2.0, beta_sigma=0.5), 64, 6)


def test_segmented_scan_in_place_and_bf16_off_shape():
    """In place (ht = h0), and bf16 q/k/v on chunk 32 (the chunk-record route
    for the model's head shape)."""
    check_seg(draw(1, 900, 2, 4, 128, 128, dtype=torch.float32, seed=542), 64, 4, inplace=True)
    check_seg(draw(1, 900, 2, 4, 128, 128, dtype=torch.bfloat16, seed=543), 32, 3)


def test_segmented_scan_without_states():
    d = draw(2, 600, 1, 2, 128, 128, dtype=torch.float32, h0=False, seed=544)
    ref_o, _ = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")), None)
    out, ht, tr = forward_seg(d, 64, gdr_flag_segments(3), store_ht=False)
    assert ht is None and "gdr_segment_combine" in tr, tr
    assert_close("o", out, ref_o, torch.float32)


def test_segmented_scan_automatic():
    """One sequence of 2048 tokens on four value heads leaves most SMs idle:
    the automatic choice segments it; with GDR_FLAG_NO_SEGMENTS it walks
    whole; both within the bound."""
    d = draw(1, 2048, 2, 4, 128, 128, dtype=torch.float32, seed=545)
    ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d["h0"]))
    out, ht, tr = forward_seg(d, 64, 0)
    assert "gdr_segment_combine" in tr, tr
    assert_close("o", out, ref_o, torch.float32)
    assert_close("ht", ht, ref_h, torch.float32)
    out2, ht2, tr2 = forward_seg(d, 64, GDR_FLAG_NO_SEGMENTS)
    assert tr2["gdr_chunk_scan_tc"][0] == 1, tr2
    assert_close("o", out2, ref_o, torch.float32)


def test_segmented_scan_not_taken():
    """dk = 64 (the combine holds 128 x 128 states) and the CUDA-core scan
    walk whole whatever the flags."""
    for d, flags in [(draw(1, 700, 2, 4, 64, 64, dtype=torch.float32, seed=546), 0),
                     (draw(1, 700, 2, 4, 128, 128, dtype=torch.float32, seed=547),
                      GDR_FLAG_FORCE_GENERIC)]:
        _, _, tr = forward_seg(d, 64, gdr_flag_segments(3) | flags)
        assert tr.get("gdr_chunk_scan_tc", (1, 0.0))[0] <= 1 and "gdr_segment_combine" not in tr, tr


@pytest.mark.parametrize("segments", [2, 4])
def test_segmented_scan_packed(segments):
    """A packed f32 batch: the sequences over exactly `segments` segments are
    cut, a short one and a single token are not, and the slots are not in
    the order the longest-first plan runs them (per-sequence final states)."""
    gen = torch.Generator()
    gen.manual_seed(550 + segments)
    seqs = [draw(1, L, 2, 4, 128, 128, dtype=torch.float32, generator=gen)
            for L in (700, 1, 1000, 40)]
    packed, cu = pack(seqs)
    c = to_cuda(packed)
    gdr_trace_enable(True)
    try:
        out, ht = gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, h0=c["h0"],
                                     chunk=64, flags=gdr_flag_segments(segments))
        gdr_device_check()
        tr = gdr_trace_read()
    finally:
        gdr_trace_enable(False)
    assert tr["gdr_chunk_scan_tc"][0] == 3, tr
    for n, d in enumerate(seqs):
        ref_o, ref_h = oracle.recurrence(*(to_f64(d[x]) for x in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))
        assert_close("o[%d]" % n, out[:, cu[n]:cu[n + 1]], ref_o, torch.float32)
        assert_close("ht[%d]" % n, ht[n:n + 1], ref_h, torch.float32)


# ------------------------------------------ the chunk prep on the tensor cores
def test_prep_mixed_fast_and_exact_chunks():
    """f32, dk = dv = 128, chunk 64 (the tensor-core prep): the factored gram
    for most chunks, the exact pairwise decays for chunks 1 and 4, whose
    log-decay is scaled so that their half-chunk spans pass 60 nats, and a
    ragged last chunk; against the oracle, and the launches of the route."""
    d = draw(2, 64 * 6 + 17, 2, 4, 128, 128, dtype=torch.float32, seed=560)
    g = d["g"].clone()
    g[:, 64:128] *= 12.0
    g[:, 256:320] *= 12.0
    d["g"] = g
    ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d["h0"]))
    out, ht, tr = forward(d, 64)
    assert "gdr_chunk_prep_tc" in tr and "gdr_chunk_prep" not in tr, tr
    assert_close("o", out, ref_o, torch.float32)
    assert_close("ht", ht, ref_h, torch.float32)


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129])
def test_prep_lengths_around_the_chunk(T):
    """Chunk lengths 1 .. 64 through the tensor-core prep (T = 1 forced onto
    the chunked route), with and without h0."""
    from channelwise_gated_delta_gb300 import GDR_FLAG_FORCE_CHUNKED
    for h0 in (True, False):
        d = draw(1, T, 1, 2, 128, 128, dtype=torch.float32, h0=h0, seed=570 + T)
        ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))
        out, ht, tr = forward(d, 64, flags=GDR_FLAG_FORCE_CHUNKED)
        assert "gdr_chunk_prep_tc" in tr, tr
        assert_close("o", out, ref_o, torch.float32)
        assert_close("ht", ht, ref_h, torch.float32)


def test_prep_scalar_gate():
    """A scalar gate (one log-decay per token and value head) through the
    tensor-core prep."""
    d = draw(1, 300, 2, 4, 128, 128, dtype=torch.float32, seed=580, scalar_gate=True)
    ref_o, ref_h = oracle.scalar_gate_recurrence(
        *(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")), to_f64(d["h0"]))
    out, ht, tr = forward(d, 64)
    assert "gdr_chunk_prep_tc" in tr, tr
    assert_close("o", out, ref_o, torch.float32)
    assert_close("ht", ht, ref_h, torch.float32)


@pytest.mark.parametrize("HK,HV", [(2, 2), (1, 4), (4, 8)])
def test_prep_head_groupings(HK, HV):
    """Key heads shared by 1, 4 and 2 value heads through the tensor-core
    prep (each CTA reads its key head's k and q rows)."""
    d = draw(2, 200, HK, HV, 128, 128, dtype=torch.float32, seed=590 + 10 * HK + HV)
    ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d["h0"]))
    out, ht, tr = forward(d, 64)
    assert "gdr_chunk_prep_tc" in tr, tr
    assert_close("o", out, ref_o, torch.float32)
    assert_close("ht", ht, ref_h, torch.float32)


def test_segmented_scan_scalar_gate():
    """A scalar gate through the tensor-core prep and a segmented scan."""
    d = draw(1, 900, 2, 4, 128, 128, dtype=torch.float32, seed=600, scalar_gate=True)
    ref_o, ref_h = oracle.scalar_gate_recurrence(
        *(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")), to_f64(d["h0"]))
    out, ht, tr = forward_seg(d, 64, gdr_flag_segments(4))
    assert "gdr_segment_combine" in tr and "gdr_chunk_prep_tc" in tr, tr
    assert_close("o", out, ref_o, torch.float32)
    assert_close("ht", ht, ref_h, torch.float32)


def test_segmented_scan_packed_chunk32_bf16():
    """Packed bf16 q/k/v at chunk 32 (the CUDA-core prep, then the
    tensor-core scan in segments): the long sequences cut into 3, a decode
    token and a short sequence beside them."""
    gen = torch.Generator()
    gen.manual_seed(610)
    seqs = [draw(1, L, 2, 4, 128, 128, dtype=torch.bfloat16, generator=gen)
            for L in (500, 1, 333, 20)]
    packed, cu = pack(seqs)
    c = to_cuda(packed)
    gdr_trace_enable(True)
    try:
        out, ht = gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, h0=c["h0"],
                                     chunk=32, flags=gdr_flag_segments(3))
        gdr_device_check()
        tr = gdr_trace_read()
    finally:
        gdr_trace_enable(False)
    assert "gdr_segment_combine" in tr and "gdr_chunk_prep" in tr, tr
    for n, d in enumerate(seqs):
        ref_o, ref_h = oracle.recurrence(*(to_f64(d[x]) for x in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))
        assert_close("o[%d]" % n, out[:, cu[n]:cu[n + 1]], ref_o, torch.bfloat16)
        assert_close("ht[%d]" % n, ht[n:n + 1], ref_h, torch.bfloat16)


def test_segmented_scan_packed_in_place():
    """A packed f32 batch updated in place (ht = h0), cut into three
    segments: the h0 copies into the first segments' states come before any
    final state lands, and the sequence that walks whole keeps its own slot."""
    gen = torch.Generator()
    gen.manual_seed(620)
    seqs = [draw(1, L, 2, 4, 128, 128, dtype=torch.float32, generator=gen)
            for L in (40, 900, 650)]
    packed, cu = pack(seqs)
    c = to_cuda(packed)
    gdr_trace_enable(True)
    try:
        out, ht = gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, h0=c["h0"],
                                     ht=c["h0"], chunk=64, flags=gdr_flag_segments(3))
        gdr_device_check()
        tr = gdr_trace_read()
    finally:
        gdr_trace_enable(False)
    assert "gdr_segment_combine" in tr and tr["gdr_chunk_scan_tc"][0] == 3, tr
    assert ht.data_ptr() == c["h0"].data_ptr()
    for n, d in enumerate(seqs):
        ref_o, ref_h = oracle.recurrence(*(to_f64(d[x]) for x in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))
        assert_close("o[%d]" % n, out[:, cu[n]:cu[n + 1]], ref_o, torch.float32)
        assert_close("ht[%d]" % n, ht[n:n + 1], ref_h, torch.float32)
