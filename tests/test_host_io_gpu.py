"""gdr_forward_host (host buffers in and out, batch elements pipelined
through two device slots): the same bits as the device entry on the same
values, on every route."""
import pytest
import torch

from channelwise_gated_delta_gb300 import (GDR_FLAG_NO_SEGMENTS, gdr_device_check, gdr_forward,
                                           gdr_forward_host)
from channelwise_gated_delta_gb300.inputs import draw

pytestmark = pytest.mark.gpu


def pinned(t):
    return None if t is None else t.contiguous().pin_memory()


def run_both(d, chunk, inplace=False, store_ht=True):
    host = {n: pinned(d[n]) for n in ("q", "k", "v", "g", "beta", "h0")}
    B, T, _, _ = d["q"].shape
    HV, dv, dk = d["v"].shape[2], d["v"].shape[3], d["q"].shape[3]
    out_h = torch.empty(B, T, HV, dv, dtype=d["q"].dtype).pin_memory()
    if inplace:
        ht_h = host["h0"]
    else:
        ht_h = torch.empty(B, HV, dk, dv).pin_memory() if store_ht else None
    gdr_forward_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["h0"], out_h,
                     ht_h, chunk=chunk)
    torch.cuda.current_stream().synchronize()
    gdr_device_check()
    c = {n: (None if t is None else t.cuda()) for n, t in d.items()}
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=chunk,
                          store_ht=store_ht)
    gdr_device_check()
    assert torch.equal(out_h, out.cpu())
    if store_ht:
        assert torch.equal(ht_h, ht.cpu())


@pytest.mark.parametrize("B,T,dtype,dk,dv", [
    (3, 200, torch.bfloat16, 128, 128),   # tensor-core route, odd batch through two slots
    (4, 70, torch.float32, 64, 64),       # CUDA-core route with its workspace in the slot
    (1, 33, torch.bfloat16, 128, 128),    # one slot
    (5, 1, torch.bfloat16, 128, 128),     # decode route
    (2, 0, torch.float32, 32, 32),        # empty sequences: ht = h0
])
def test_host_entry_matches_device_entry(B, T, dtype, dk, dv):
    run_both(draw(B, T, 2, 4, dk, dv, dtype=dtype, seed=B * 100 + T), 64)


def test_host_entry_no_initial_state_no_final_state():
    run_both(draw(3, 90, 1, 2, 128, 128, dtype=torch.bfloat16, h0=False, seed=7), 64,
             store_ht=False)


def test_host_entry_in_place_state():
    d = draw(3, 65, 1, 2, 128, 128, dtype=torch.bfloat16, seed=8)
    ref = {n: (None if t is None else t.clone()) for n, t in d.items()}
    run_both(d, 64, inplace=False)
    # in place: ht is h0 (host)
    host = {n: pinned(ref[n]) for n in ("q", "k", "v", "g", "beta", "h0")}
    out_h = torch.empty(3, 65, 2, 128, dtype=torch.bfloat16).pin_memory()
    gdr_forward_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["h0"],
                     out_h, host["h0"], chunk=64)
    torch.cuda.current_stream().synchronize()
    c = {n: t.cuda() for n, t in ref.items()}
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=64)
    assert torch.equal(out_h, out.cpu())
    assert torch.equal(host["h0"], ht.cpu())


def test_host_entry_back_to_back_calls():
    """Two calls in a row on one stream reuse the library's events and copy
    streams; the second's results are its own."""
    a = draw(3, 100, 1, 2, 128, 128, dtype=torch.bfloat16, seed=9)
    b = draw(3, 100, 1, 2, 128, 128, dtype=torch.bfloat16, seed=10)
    outs = []
    for d in (a, b):
        host = {n: pinned(d[n]) for n in ("q", "k", "v", "g", "beta", "h0")}
        o = torch.empty(3, 100, 2, 128, dtype=torch.bfloat16).pin_memory()
        h = torch.empty(3, 2, 128, 128).pin_memory()
        gdr_forward_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["h0"],
                         o, h, chunk=64)
        outs.append((o, h))
    torch.cuda.current_stream().synchronize()
    for d, (o, h) in zip((a, b), outs):
        c = {n: t.cuda() for n, t in d.items()}
        out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=64)
        assert torch.equal(o, out.cpu()) and torch.equal(h, ht.cpu())


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_host_entry_segments_long_sequences(dtype, d):
    """Sequences longer than two segments (4096 tokens) are streamed in
    segments that resume from the state the previous one left: the result is
    the recurrence's, to the route's tolerance, and within float32 rounding of
    the unsegmented device call."""
    import oracle
    from channelwise_gated_delta_gb300.inputs import to_f64
    from tests.parity_util import assert_close
    d_ = draw(2, 4500, 1, 2, d, d, dtype=dtype, seed=11)
    host = {n: pinned(d_[n]) for n in ("q", "k", "v", "g", "beta", "h0")}
    out_h = torch.empty(2, 4500, 2, d, dtype=dtype).pin_memory()
    ht_h = torch.empty(2, 2, d, d).pin_memory()
    gdr_forward_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["h0"], out_h,
                     ht_h, chunk=64)
    torch.cuda.current_stream().synchronize()
    gdr_device_check()
    ref_o, ref_h = oracle.recurrence(*(to_f64(d_[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d_["h0"]))
    assert_close("o", out_h, ref_o, dtype)
    assert_close("ht", ht_h, ref_h, dtype)
    c = {n: t.cuda() for n, t in d_.items()}
    # the host entry never segments the state scan; compare with the same walk
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=64,
                          flags=GDR_FLAG_NO_SEGMENTS)
    tol = 1e-2 if dtype == torch.bfloat16 else 1e-5
    assert (out_h.float() - out.cpu().float()).abs().max() <= tol * out.float().abs().max().cpu()
    assert (ht_h - ht.cpu()).abs().max() <= tol * ht.abs().max().cpu()
