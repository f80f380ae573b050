"""gdr_forward_chunked_noalloc: the chunked prefill with its scratch in a fixed
array inside the library, for callers that cannot allocate device memory
(a runtime whose memory planner owns all device memory, a serving loop that
must avoid cudaMalloc's synchronisation, a plugin bound to its host's
allocator).

Its results must match the regular entry point, gdr_forward_ex, running the
same chunked kernels with a workspace from torch's allocator, within the
parity tolerance of the other tests.  Two calls in a row with different
problems check that the shared scratch carries nothing over between calls.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

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
def test_noalloc_matches_regular_entry_point_twice():
    lib = load_library()
    problems = [
        (draw(2, 150, 2, 4, 64, 64, dtype=torch.float32, seed=21), 32),
        (draw(1, 97, 16, 32, 128, 128, dtype=torch.bfloat16, seed=22), 64),
    ]
    flags = GDR_FLAG_FORCE_CHUNKED | GDR_FLAG_FORCE_GENERIC
    for d, chunk in problems:
        c = to_cuda(d)
        ref_o, ref_h = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                                   chunk=chunk, flags=flags)
        gdr_device_check()
        out, ht = noalloc_call(lib, c, chunk)
        dtype = d["q"].dtype
        assert_close("o (no-alloc vs regular)", out, to_f64(ref_o), dtype)
        assert_close("ht (no-alloc vs regular)", ht, to_f64(ref_h), dtype)


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
