"""The segmented state scan of the tensor-core route on the GPU: parity with
the fp64 oracle for forced segment counts (two to many, ragged last chunk,
with and without h0, in place, scalar gate, strong decays), the first
segment's rows bit for bit those of the unsegmented route, the automatic
choice on a small-batch long prefill, and packed batches whose long
sequences are cut (automatically and forced) beside ones that walk whole."""
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_NO_SEGMENTS, gdr_device_check, gdr_flag_segments,
                                           gdr_forward, gdr_forward_varlen, gdr_trace_enable,
                                           gdr_trace_read)
from channelwise_gated_delta_gb300.inputs import WORKLOADS, draw, draw_workload, pack, to_f64
from tests.parity_util import assert_close, to_cuda
from tests.test_parity_gpu import run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def waves(tr):
    """Launches of the tensor-core kernel: two waves when the scan is cut
    (plus one for the sequences that walk whole in a packed batch), one
    when it is not."""
    return tr.get("gdr_prefill_fused", (0, 0.0))[0]


def traced(fn):
    gdr_trace_enable(True)
    try:
        res = fn()
        gdr_device_check()
        return res, gdr_trace_read()
    finally:
        gdr_trace_enable(False)


def check_segmented(d, segments, inplace=False):
    dtype = d["q"].dtype
    ref_o, ref_h = run_oracle(d)
    (out, ht), tr = traced(lambda: run_gpu(d, 64, flags=gdr_flag_segments(segments),
                                           inplace=inplace))
    assert_close("o", out, ref_o, dtype)
    assert_close("ht", ht, ref_h, dtype)
    assert waves(tr) == 2, tr
    return out, ht


@pytest.mark.parametrize("segments", [2, 3, 4, 6])
@pytest.mark.parametrize("T", [129, 1000])
def test_forced_segments_match_oracle(segments, T):
    check_segmented(draw(1, T, 2, 4, 128, 128, dtype=torch.bfloat16, seed=400 + T + segments),
                    segments)


def test_batch_and_grouped_heads():
    check_segmented(draw(3, 700, 1, 4, 128, 128, dtype=torch.bfloat16, seed=410), 4)


def test_no_initial_state():
    check_segmented(draw(2, 500, 2, 2, 128, 128, dtype=torch.bfloat16, h0=False, seed=411), 3)


def test_in_place_state():
    check_segmented(draw(1, 640, 2, 4, 128, 128, dtype=torch.bfloat16, seed=412), 5, inplace=True)


def test_no_final_state():
    d = draw(1, 400, 2, 4, 128, 128, dtype=torch.bfloat16, seed=413)
    ref_o, _ = run_oracle(d)
    c = to_cuda(d)
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=64,
                          flags=gdr_flag_segments(3), store_ht=False)
    gdr_device_check()
    assert ht is None
    assert_close("o", out, ref_o, torch.bfloat16)


def test_one_chunk_per_segment():
    """More segments requested than chunks: every segment is one chunk."""
    check_segmented(draw(1, 300, 1, 2, 128, 128, dtype=torch.bfloat16, seed=414), 200)


def test_scalar_gate():
    d = draw(1, 900, 2, 4, 128, 128, dtype=torch.bfloat16, seed=415, scalar_gate=True)
    args = [to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")]
    ref_o, ref_h = oracle.scalar_gate_recurrence(*args, to_f64(d["h0"]))
    out, ht = run_gpu(d, 64, flags=gdr_flag_segments(4))
    assert_close("o", out, ref_o, torch.bfloat16)
    assert_close("ht", ht, ref_h, torch.bfloat16)


@pytest.mark.parametrize("g_mu,beta_mu", [(-3.0, 2.0), (2.0, 0.0), (6.0, 0.0)])
def test_decay_regimes(g_mu, beta_mu):
    """Weak decay with strong updates (the long-prefill distribution), strong
    decay, and decay strong enough for the kernel's exact pairwise path: the
    maps M_p run from the identity through the same range handling."""
    check_segmented(draw(1, 768, 2, 4, 128, 128, dtype=torch.bfloat16, seed=416, g_mu=g_mu,
                         beta_mu=beta_mu, beta_sigma=0.5), 4)


def test_first_segment_rows_are_the_unsegmented_bits():
    """Segment 0 runs from h0 through the same kernel code as the plain route:
    its rows (whole chunks) are bit for bit the plain route's."""
    d = draw(2, 1000, 2, 4, 128, 128, dtype=torch.bfloat16, seed=417)
    seg, _ = run_gpu(d, 64, flags=gdr_flag_segments(3))
    plain, _ = run_gpu(d, 64, flags=GDR_FLAG_NO_SEGMENTS)
    first = 64 * 6  # 16 chunks in 3 segments: 6 chunks each
    assert torch.equal(seg[:, :first], plain[:, :first])


def test_automatic_choice_on_a_small_batch_long_prefill():
    """B = 1, 32 value heads, T = 4096 (64 chunks): the automatic choice
    segments (32 CTAs would leave most SMs idle); oracle on a sample of heads."""
    w = WORKLOADS["prefill_t4k"]
    d = draw_workload(w)
    (out, ht), tr = traced(lambda: run_gpu(d, w.chunk))
    assert "gdr_segment_combine" in tr, tr
    ref = oracle.recurrence_heads(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                  to_f64(d["h0"]), [(0, 0), (0, 13), (0, 31)])
    for (b, hv), (ref_o, ref_h) in ref.items():
        assert_close("o[%d,%d]" % (b, hv), out[b, :, hv], ref_o, d["q"].dtype)
        assert_close("ht[%d,%d]" % (b, hv), ht[b, hv], ref_h, d["q"].dtype)
    # and it agrees with the unsegmented route to within the same bound
    plain_o, plain_h = run_gpu(d, w.chunk, flags=GDR_FLAG_NO_SEGMENTS)
    assert_close("o vs plain", out, to_f64(plain_o), d["q"].dtype)
    assert_close("ht vs plain", ht, to_f64(plain_h), d["q"].dtype)


def test_large_batch_is_not_segmented():
    """B x HV = 128 fills the device: the automatic choice keeps one walk."""
    d = draw(4, 1024, 16, 32, 128, 128, dtype=torch.bfloat16, seed=418)
    _, tr = traced(lambda: run_gpu(d, 64))
    assert waves(tr) == 1, tr


def mixed_decay(B, T, HK, HV, pattern, seed, scalar_gate=False):
    """A problem whose 64-row chunks follow `pattern`, one letter per chunk:
      f  weak decay (about 0.05 nats a step): the fast path;
      s  strong (about 6 nats a step): the exact path, its diagonal blocks
         factored about their middle row;
      x  steep (20 to 30 nats a step): diagonal blocks past the factor
         range, pairwise decays;
      c  weak, but one row drops by 100 nats in a few key channels (every
         channel with a scalar gate): a cliff inside one block."""
    d = draw(B, T, HK, HV, 128, 128, dtype=torch.bfloat16, seed=seed, g_mu=-3.0,
             scalar_gate=scalar_gate)
    gen = torch.Generator().manual_seed(seed + 1)
    g = d["g"]
    assert len(pattern) == (T + 63) // 64
    for c, kind in enumerate(pattern):
        rows = slice(64 * c, min(64 * c + 64, T))
        shape = g[:, rows].shape
        if kind == "s":
            g[:, rows] = -torch.nn.functional.softplus(torch.randn(shape, generator=gen) * 0.5 + 6.0)
        elif kind == "x":
            g[:, rows] = -(20.0 + 10.0 * torch.rand(shape, generator=gen))
        elif kind == "c":
            r = min(64 * c + 37, T - 1)
            if scalar_gate:
                g[:, r] = -100.0
            else:
                g[:, r, :, :5] = -100.0
        else:
            assert kind == "f"
    return d


def assert_close_by_chunk(got, ref):
    """The bf16 bound of each 64-row chunk of o on its own: a chunk of small
    outputs is not hidden behind another's large ones."""
    for t0 in range(0, ref.shape[1], 64):
        assert_close("o rows %d+" % t0, got[:, t0:t0 + 64], ref[:, t0:t0 + 64], torch.bfloat16)


MIXED = "fsfxsscfs" "fsxfcsx"  # 16 chunks, the last one 40 rows


@pytest.mark.parametrize("segments", [0, 4, 5])
def test_mixed_fast_and_exact_chunks_across_segments(segments):
    """Fast and exact-path chunks side by side, at segment starts and ends
    (4 segments: chunks 0-3 | 4-7 | 8-11 | 12-15; 5: a boundary inside the
    run of exact chunks), including a ragged exact last chunk; 0 = one
    unsegmented walk."""
    d = mixed_decay(2, 1000, 2, 4, MIXED, seed=430 + segments)
    ref_o, ref_h = run_oracle(d)
    flags = gdr_flag_segments(segments) if segments else GDR_FLAG_NO_SEGMENTS
    (out, ht), tr = traced(lambda: run_gpu(d, 64, flags=flags))
    assert_close_by_chunk(out, ref_o)
    assert_close("ht", ht, ref_h, torch.bfloat16)
    assert (waves(tr) == 2) == bool(segments), tr


def test_mixed_chunks_scalar_gate():
    d = mixed_decay(1, 1000, 2, 4, MIXED, seed=440, scalar_gate=True)
    args = [to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")]
    ref_o, ref_h = oracle.scalar_gate_recurrence(*args, to_f64(d["h0"]))
    for flags in (GDR_FLAG_NO_SEGMENTS, gdr_flag_segments(4)):
        out, ht = run_gpu(d, 64, flags=flags)
        assert_close_by_chunk(out, ref_o)
        assert_close("ht", ht, ref_h, torch.bfloat16)


# ---- packed variable-length batches: long sequences cut into segments


def run_packed(seqs, flags=0, inplace=False):
    packed, cu = pack(seqs)
    c = to_cuda(packed)
    ht = c["h0"] if (inplace and c["h0"] is not None) else None
    (out, ht), tr = traced(lambda: gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"],
                                                      cu, h0=c["h0"], ht=ht, chunk=64,
                                                      flags=flags))
    return out, ht, cu, tr


def check_packed(seqs, out, ht, cu):
    for n, d in enumerate(seqs):
        ref_o, ref_h = oracle.recurrence(*(to_f64(d[x]) for x in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))
        assert_close("o[%d]" % n, out[:, cu[n]:cu[n + 1]], ref_o, torch.bfloat16)
        assert_close("ht[%d]" % n, ht[n:n + 1], ref_h, torch.bfloat16)


def draw_packed(lengths, HK, HV, seed, **kw):
    gen = torch.Generator()
    gen.manual_seed(seed)
    return [draw(1, L, HK, HV, 128, 128, dtype=torch.bfloat16, generator=gen, **kw)
            for L in lengths]


def test_packed_long_sequence_segmented_automatically():
    """{4096, 1, 64} at the model's head shape: the 4096-token sequence is cut
    (32 value heads leave most SMs idle), the 64-token one walks whole and
    the single token decodes; every sequence against the oracle."""
    props = torch.cuda.get_device_properties(0)
    if props.multi_processor_count < 32 * 4:
        pytest.skip("too few SMs for a three-segment wave beside the other sequence")
    seqs = draw_packed((4096, 1, 64), 16, 32, seed=450)
    out, ht, cu, tr = run_packed(seqs)
    assert "gdr_segment_combine" in tr and "gdr_decode_kernel" in tr, tr
    check_packed(seqs, out, ht, cu)
    # the same batch with the scan unsegmented: the same results within the bound
    out2, ht2, _, tr2 = run_packed(seqs, flags=GDR_FLAG_NO_SEGMENTS)
    assert waves(tr2) == 1 and "gdr_segment_combine" not in tr2, tr2
    check_packed(seqs, out2, ht2, cu)


@pytest.mark.parametrize("segments", [2, 3, 5])
def test_packed_forced_segments_mixed_lengths(segments):
    """The sequences whose chunks spread over the forced count are cut, in an
    order their slots do not follow (longest first), beside ones that walk
    whole and a decode token."""
    lengths = (130, 1000, 40, 700, 1, 300)
    seqs = draw_packed(lengths, 2, 4, seed=460 + segments)
    out, ht, cu, tr = run_packed(seqs, flags=gdr_flag_segments(segments))
    assert waves(tr) >= 2, tr
    check_packed(seqs, out, ht, cu)


def test_packed_segments_in_place_and_without_h0():
    seqs = draw_packed((900, 64, 650), 2, 4, seed=470)
    out, ht, cu, tr = run_packed(seqs, flags=gdr_flag_segments(3), inplace=True)
    assert waves(tr) >= 2, tr
    check_packed(seqs, out, ht, cu)
    seqs = draw_packed((900, 650), 2, 4, seed=471, h0=False)
    out, ht, cu, tr = run_packed(seqs, flags=gdr_flag_segments(4))
    assert waves(tr) >= 2, tr
    check_packed(seqs, out, ht, cu)
