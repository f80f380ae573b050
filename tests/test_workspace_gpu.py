"""The C entry gdr_forward and its workspace: the library's own (grown on
demand) or a caller-owned one registered with gdr_set_workspace, too small
ones refused before anything is enqueued, and the same bits as the
per-call-workspace entry either way."""
import ctypes

import pytest
import torch

from channelwise_gated_delta_gb300 import (gdr_device_check, gdr_forward, gdr_set_workspace,
                                           gdr_workspace_bytes, load_library)
from channelwise_gated_delta_gb300.inputs import draw
from tests.parity_util import to_cuda

pytestmark = pytest.mark.gpu


def c_forward(c, out, ht, chunk):
    lib = load_library()
    B, T, HK, dk = c["q"].shape
    HV, dv = c["v"].shape[2], c["v"].shape[3]
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    code = 1 if c["q"].dtype == torch.bfloat16 else 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gdr_forward(ptr(c["q"]), ptr(c["k"]), ptr(c["v"]), ptr(c["g"]), ptr(c["beta"]),
                           ptr(c["h0"]), ptr(out), ptr(ht), B, T, HK, HV, dk, dv, chunk, stream,
                           code)


CASES = [
    # CUDA-core route: chunk records
    (dict(B=2, T=100, HK=1, HV=2, dk=64, dv=64, dtype=torch.float32), 32),
    # tensor-core route, segmented automatically (B x HV = 32, 64 chunks)
    (dict(B=1, T=4096, HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16), 64),
]


@pytest.mark.parametrize("shape,chunk", CASES)
def test_library_and_registered_workspaces(shape, chunk):
    s = dict(shape)
    dtype = s.pop("dtype")
    d = draw(s["B"], s["T"], s["HK"], s["HV"], s["dk"], s["dv"], dtype=dtype, seed=600)
    c = to_cuda(d)
    ref_o, ref_h = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=chunk)
    need = gdr_workspace_bytes(s["B"], s["T"], s["HK"], s["HV"], s["dk"], s["dv"], chunk, dtype)
    assert need > 0
    out = torch.empty_like(ref_o)
    ht = torch.empty_like(ref_h)
    try:
        # the library's own workspace
        assert c_forward(c, out, ht, chunk) == 0
        gdr_device_check()
        assert torch.equal(out, ref_o) and torch.equal(ht, ref_h)
        # a caller-owned one of exactly the size asked for
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        gdr_set_workspace(ws)
        out.zero_()
        assert c_forward(c, out, ht, chunk) == 0
        gdr_device_check()
        assert torch.equal(out, ref_o) and torch.equal(ht, ref_h)
        # too small: refused, nothing written
        small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
        gdr_set_workspace(small)
        out.fill_(7.0)
        assert c_forward(c, out, ht, chunk) == 5  # GDR_ERR_WORKSPACE
        torch.cuda.synchronize()
        assert bool((out == 7.0).all())
    finally:
        gdr_set_workspace(None)
    # back to the library's own
    assert c_forward(c, out, ht, chunk) == 0
    gdr_device_check()
    assert torch.equal(out, ref_o) and torch.equal(ht, ref_h)


def test_unaligned_registration_refused():
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    lib = load_library()
    assert lib.gdr_set_workspace(ctypes.c_void_p(ws.data_ptr() + 16), 1024) == 4
