"""The failure path of the library's bounded waits, without a GPU fault:
the same bounded mbarrier wait the kernels use, run on a barrier that
nothing arrives on, gives up after its limit, reports it in its error word,
and leaves the kernel to finish and the context usable (a forward call right
after it runs and matches the oracle)."""
import pytest
import torch

import oracle
from channelwise_gated_delta_gb300 import gdr_device_check, gdr_forward
from channelwise_gated_delta_gb300.inputs import draw, to_f64
from tests.parity_util import assert_close, to_cuda
from tests.umma_diag import wait_limit

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [5, 50])
def test_bounded_wait_gives_up_and_context_survives(limit_ms):
    gave_up, ms = wait_limit(limit_ms * 1000000)
    assert gave_up == 32            # every waiting thread ran out
    assert ms >= 0.9 * limit_ms     # and only after its limit
    assert ms < limit_ms + 1000     # bounded: well inside a second past it
    d = draw(1, 100, 1, 2, 32, 32, dtype=torch.float32, seed=700 + limit_ms)
    c = to_cuda(d)
    out, ht = gdr_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], chunk=16)
    gdr_device_check()  # the library's own error word is untouched: GDR_OK
    ref_o, ref_h = oracle.recurrence(*(to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")),
                                     to_f64(d["h0"]))
    assert_close("o", out, ref_o, torch.float32)
    assert_close("ht", ht, ref_h, torch.float32)


def test_bad_limits_rejected():
    from tests.umma_diag import _load
    lib = _load()
    import ctypes
    buf = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.gdr_diag_wait_limit(10, ctypes.c_void_p(buf.data_ptr()), None) == -1
    assert lib.gdr_diag_wait_limit(2 * 10**9, ctypes.c_void_p(buf.data_ptr()), None) == -1
    assert lib.gdr_diag_wait_limit(10**7, None, None) == -1
