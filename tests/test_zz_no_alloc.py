"""gdr_forward_chunked_noalloc: the chunked prefill with its scratch in a fixed
array inside the library, for callers that cannot allocate device memory
(a runtime whose memory planner owns all device memory, a serving loop that
must avoid cudaMalloc's synchronisation, a plugin bound to its host's
allocator).

It runs the same chunked kernels with the same flags as the regular entry
point, gdr_forward_ex with a workspace from torch's allocator, so its results
must equal that entry point's bit for bit; both are also checked against the
fp64 oracle.  The calls run a larger problem, then a smaller one, then the
larger one again: a stale read of the shared scratch inside the smaller
problem's footprint would see the larger problem's leftovers, not zeros.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_CHUNKED, GDR_FLAG_FORCE_GENERIC,
                                           gdr_device_check, gdr_forward, load_library)
from channelwise_gated_delta_gb300.inputs import draw, to_f64
from tests.parity_util import assert_close, to_cuda

SCRATCH_BYTES = 64 * 1024 * 1024  # GDR_NOALLOC_SCRATCH_BYTES in include/gdr.h


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def noalloc_call(lib, c, chunk):
    B, T, HK, dk = c["q"].shape
    HV, dv = c["v"].shape[2], c["v"].shape[3]
    out = torch.empty(B, T, HV, dv, dtype=c["q"].dtype, device="cuda")
    ht = torch.empty(B, HV, dk, dv, dtype=torch.float32, device="cuda")
    code = 1 if c["q"].dtype == torch.bfloat16 else 0
    stream = torch.cuda.current_stream()
    st = lib.gdr_forward_chunked_noalloc(
        _p(c["q"]), _p(c["k"]), _p(c["v"]), _p(c["g"]), _p(c["beta"]), _p(c["h0"]), _p(out),
        _p(ht), B, T, HK, HV, dk, dv, chunk, ctypes.c_void_p(stream.cuda_stream), code)
    assert st == 0, lib.gdr_status_string(st).decode()
    gdr_device_check()
    return out, ht


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_call_after_call():
    lib = load_library()
    large = (draw(1, 97, 16, 32, 128, 128, dtype=torch.bfloat16, seed=22), 64)
    small = (draw(2, 150, 2, 4, 64, 64, dtype=torch.float32, seed=21), 32)
    flags = GDR_FLAG_FORCE_CHUNKED | GDR_FLAG_FORCE_GENERIC
    for d, chunk in (large, small, large):
        c = to_cuda(d)
        ref_o, ref_h = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                                   chunk=chunk, flags=flags)
        gdr_device_check()
        out, ht = noalloc_call(lib, c, chunk)
        assert torch.equal(out, ref_o), "o differs from the regular entry point"
        assert torch.equal(ht, ref_h), "ht differs from the regular entry point"
        ro, rh = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                   to_f64(d["h0"]))
        assert_close("o (no-alloc vs oracle)", out, ro, d["q"].dtype)
        assert_close("ht (no-alloc vs oracle)", ht, rh, d["q"].dtype)


def test_noalloc_rejects_oversized_problem():
    """A problem whose scratch exceeds the fixed array is refused on the host,
    before anything is enqueued (fake, never-dereferenced pointers)."""
    lib = load_library()
    B, T, HK, HV, dk, dv, chunk = 4, 16384, 16, 32, 128, 128, 64
    need = lib.gdr_workspace_bytes(B, T, HK, HV, dk, dv, chunk, 1,
                                   GDR_FLAG_FORCE_CHUNKED | GDR_FLAG_FORCE_GENERIC)
    assert need > SCRATCH_BYTES
    base = 1 << 40
    ptrs = [ctypes.c_void_p(base + (i << 36)) for i in range(8)]
    st = lib.gdr_forward_chunked_noalloc(*ptrs, B, T, HK, HV, dk, dv, chunk, None, 1)
    assert st == 5  # GDR_ERR_WORKSPACE
