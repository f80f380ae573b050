"""GPU parity of the packed variable-length entry (gdr_forward_varlen): every
sequence of the packed batch against the fp64 oracle run on that sequence
alone, and bit for bit against one gdr_forward call per sequence (the same
kernels on the same rows)."""
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_CHUNKED, GDR_FLAG_FORCE_GENERIC,
                                           GDR_FLAG_NO_SEGMENTS,
                                           GdrError, gdr_device_check, gdr_forward, gdr_forward_varlen,
                                           gdr_varlen_workspace_bytes)
from channelwise_gated_delta_gb300.inputs import WORKLOADS, draw, draw_workload, pack, to_f64
from tests.parity_util import assert_close, to_cuda

pytestmark = pytest.mark.gpu


def draw_seqs(lengths, HK, HV, dk, dv, dtype, h0=True, seed=0, **kw):
    gen = torch.Generator()
    gen.manual_seed(seed)
    return [draw(1, L, HK, HV, dk, dv, dtype=dtype, h0=h0, generator=gen, **kw) for L in lengths]


def run_varlen(seqs, chunk, flags=0, inplace=False, store_ht=True):
    packed, cu = pack(seqs)
    c = to_cuda(packed)
    ht = c["h0"] if (inplace and c["h0"] is not None) else None
    out, ht = gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, h0=c["h0"],
                                 ht=ht, chunk=chunk, flags=flags, store_ht=store_ht)
    gdr_device_check()
    return out, ht, cu


def run_each(seqs, chunk, flags=0):
    """One gdr_forward call per sequence, the state scan unsegmented (as in
    the packed entry); returns (outs, hts) lists."""
    outs, hts = [], []
    for d in seqs:
        c = to_cuda(d)
        o, h = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=chunk,
                           flags=flags | GDR_FLAG_NO_SEGMENTS)
        outs.append(o)
        hts.append(h)
    gdr_device_check()
    return outs, hts


def check(seqs, chunk, flags=0, inplace=False, bitwise=True):
    dtype = seqs[0]["q"].dtype
    out, ht, cu = run_varlen(seqs, chunk, flags=flags, inplace=inplace)
    assert out.shape[:2] == (1, cu[-1])
    outs_1, hts_1 = run_each(seqs, chunk, flags=flags) if bitwise else (None, None)
    for n, d in enumerate(seqs):
        ref_o, ref_h = oracle.recurrence(*(to_f64(d[x]) for x in ("q", "k", "v", "g", "beta")),
                                         to_f64(d["h0"]))
        o_n = out[:, cu[n]:cu[n + 1]]
        assert_close("o[%d]" % n, o_n, ref_o, dtype)
        assert_close("ht[%d]" % n, ht[n:n + 1], ref_h, dtype)
        if bitwise:
            assert torch.equal(o_n, outs_1[n]), "o[%d] differs from the per-sequence call" % n
            assert torch.equal(ht[n:n + 1], hts_1[n]), "ht[%d] differs from the per-sequence call" % n


def test_ragged_b8_packed():
    """Eight sequences of lengths 1 .. 512 (float32: decode + CUDA-core prefill)."""
    w = WORKLOADS["ragged_b8"]
    check(draw_workload(w), w.chunk)


def test_ragged_b8_packed_bf16_tensor_core():
    """The same lengths in bf16 at dk = dv = 128, chunk 64: decode + tensor-core prefill."""
    w = WORKLOADS["ragged_b8"]
    check(draw_seqs(w.lengths, w.HK, w.HV, w.dk, w.dv, torch.bfloat16, seed=1), w.chunk)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mixed_lengths_with_empty(dtype):
    lengths = (1, 33, 0, 64, 65, 150, 2, 0, 200, 1)
    check(draw_seqs(lengths, 2, 4, 128, 128, dtype, seed=2), 64)


@pytest.mark.parametrize("dk,dv,chunk", [(32, 32, 16), (64, 128, 32), (128, 64, 64)])
def test_generic_shapes(dk, dv, chunk):
    lengths = (17, 1, 40, 3, 0, 96)
    check(draw_seqs(lengths, 1, 3, dk, dv, torch.float32, seed=3), chunk)


@pytest.mark.parametrize("flags", [GDR_FLAG_FORCE_GENERIC, GDR_FLAG_FORCE_CHUNKED,
                                   GDR_FLAG_FORCE_CHUNKED | GDR_FLAG_FORCE_GENERIC])
def test_flags(flags):
    lengths = (1, 70, 1, 129)
    check(draw_seqs(lengths, 2, 4, 128, 128, torch.bfloat16, seed=4), 64, flags=flags)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_no_initial_state(dtype):
    check(draw_seqs((5, 1, 64, 0, 77), 2, 4, 128, 128, dtype, h0=False, seed=5), 64)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_in_place_state(dtype):
    seqs = draw_seqs((1, 90, 0, 64), 2, 4, 128, 128, dtype, seed=6)
    check(seqs, 64, inplace=True, bitwise=False)


def test_no_final_state():
    seqs = draw_seqs((1, 90, 3), 2, 4, 128, 128, torch.bfloat16, seed=7)
    out, ht, cu = run_varlen(seqs, 64, store_ht=False)
    assert ht is None
    outs_1, _ = run_each(seqs, 64)
    for n in range(len(seqs)):
        assert torch.equal(out[:, cu[n]:cu[n + 1]], outs_1[n])


def test_all_empty_and_none():
    seqs = draw_seqs((0, 0, 0), 2, 4, 64, 64, torch.float32, seed=8)
    out, ht, cu = run_varlen(seqs, 64)
    assert out.shape == (1, 0, 4, 64)
    torch.testing.assert_close(ht.cpu(), pack(seqs)[0]["h0"], rtol=0, atol=0)
    # N = 0: nothing to do, nothing allocated
    assert gdr_varlen_workspace_bytes([0], 2, 4, 64, 64, 64, torch.float32) == 0


def test_long_and_short_mix():
    """A 4k sequence beside short ones: walked whole, the long one's CTAs run
    first (bit for bit the per-sequence calls); by default, with two value
    heads leaving the SMs idle, it is cut into segments (within the bound)."""
    lengths = (3, 4096, 1, 300, 64)
    seqs = draw_seqs(lengths, 1, 2, 128, 128, torch.bfloat16, seed=9, g_mu=-3.0, beta_mu=2.0,
                     beta_sigma=0.5)
    check(seqs, 64, flags=GDR_FLAG_NO_SEGMENTS)
    check(seqs, 64, bitwise=False)


def test_bad_cu_seqlens_rejected():
    seqs = draw_seqs((4, 4), 1, 1, 32, 32, torch.float32, seed=10)
    packed, _ = pack(seqs)
    c = to_cuda(packed)
    for cu in ([1, 4, 8], [0, 9, 8]):  # cu[0] != 0; decreasing
        with pytest.raises(GdrError) as e:
            gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, h0=c["h0"],
                               chunk=16)
        assert e.value.status == 2  # GDR_ERR_SHAPE
    with pytest.raises(ValueError):  # last offset != number of rows
        gdr_forward_varlen(c["q"], c["k"], c["v"], c["g"], c["beta"], [0, 4, 9], h0=c["h0"],
                           chunk=16)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64),
                                     (torch.float32, 128)])
def test_many_sequences_random_lengths(dtype, d):
    """257 sequences of random lengths 0..70 (tables of hundreds of entries,
    many single-token rows): bit for bit the per-sequence calls, and the
    oracle on a sample of sequences."""
    gen = torch.Generator()
    gen.manual_seed(20)
    lengths = [int(x) for x in torch.randint(0, 71, (257,), generator=gen)]
    lengths[3] = 1
    lengths[4] = 0
    seqs = draw_seqs(lengths, 1, 2, d, d, dtype, seed=21)
    out, ht, cu = run_varlen(seqs, 64)
    outs_1, hts_1 = run_each(seqs, 64)
    for n in range(len(seqs)):
        assert torch.equal(out[:, cu[n]:cu[n + 1]], outs_1[n]), n
        assert torch.equal(ht[n:n + 1], hts_1[n]), n
    for n in (0, 3, 4, 100, 256):
        d_ = seqs[n]
        ref_o, ref_h = oracle.recurrence(*(to_f64(d_[x]) for x in ("q", "k", "v", "g", "beta")),
                                         to_f64(d_["h0"]))
        assert_close("o[%d]" % n, out[:, cu[n]:cu[n + 1]], ref_o, dtype)
        assert_close("ht[%d]" % n, ht[n:n + 1], ref_h, dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_all_single_tokens_equal_dense_decode(dtype):
    """64 one-token sequences packed: the decode kernel through its row table
    gives the dense decode's bits."""
    d = draw(64, 1, 16, 32, 128, 128, dtype=dtype, seed=22)
    c = to_cuda(d)
    dense_o, dense_h = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"])
    flat = lambda x: x.reshape(1, 64, *x.shape[2:]).contiguous()
    out, ht = gdr_forward_varlen(flat(c["q"]), flat(c["k"]), flat(c["v"]), flat(c["g"]),
                                 flat(c["beta"]), list(range(65)), h0=c["h0"])
    gdr_device_check()
    assert torch.equal(out.reshape(dense_o.shape), dense_o)
    assert torch.equal(ht, dense_h)
