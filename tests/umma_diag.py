"""Loader of the test-only diagnostic library libgdr_diag.so (built next to
libgdr.so by build()): one tensor-core GEMM through a chosen pair of
shared-memory operand layouts, and the library's bounded mbarrier wait run
against a barrier that never completes."""
import ctypes
import os

import torch

_LIB = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "channelwise_gated_delta_gb300", "_lib", "libgdr_diag.so")
_lib = None

# operand layouts of the diagnostic GEMM
K_MAJOR, MN_MAJOR, K_MAJOR_OF_TRANSPOSE, MN_MAJOR_SW128, A_IN_TMEM, K_MAJOR_SW128 = range(6)


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise RuntimeError("libgdr_diag.so is not built (%s)" % _LIB)
        _lib = ctypes.CDLL(_LIB)
        vp, i = ctypes.c_void_p, ctypes.c_int
        _lib.gdr_diag_umma.argtypes = [i, i, i, vp, vp, vp, vp, vp]
        _lib.gdr_diag_umma.restype = i
        _lib.gdr_diag_wait_limit.argtypes = [ctypes.c_ulonglong, vp, vp]
        _lib.gdr_diag_wait_limit.restype = i
    return _lib


def umma_gemm(A, B, a_mode, b_mode):
    """A[128, 64] @ B[N, 64]^T (bf16 in, f32 out) computed by one tcgen05 GEMM
    with the given operand layouts; raises if a bounded wait timed out."""
    lib = _load()
    N = B.shape[0]
    D = torch.empty(A.shape[0], N, dtype=torch.float32, device=A.device)
    err = torch.zeros(1, dtype=torch.int32, device=A.device)
    stream = torch.cuda.current_stream(A.device)
    st = lib.gdr_diag_umma(int(a_mode), int(b_mode), N, ctypes.c_void_p(A.data_ptr()),
                           ctypes.c_void_p(B.data_ptr()), ctypes.c_void_p(D.data_ptr()),
                           ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise RuntimeError("gdr_diag_umma failed: %d" % st)
    torch.cuda.synchronize(A.device)
    if int(err.item()) != 0:
        raise RuntimeError("gdr_diag_umma: a bounded wait timed out")
    return D


def wait_limit(limit_ns, device="cuda"):
    """Runs the bounded wait on a barrier nothing arrives on (32 threads);
    returns (threads that gave up, elapsed milliseconds on the stream)."""
    lib = _load()
    gave_up = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    st = lib.gdr_diag_wait_limit(int(limit_ns), ctypes.c_void_p(gave_up.data_ptr()),
                                 ctypes.c_void_p(stream.cuda_stream))
    e1.record(stream)
    if st != 0:
        raise RuntimeError("gdr_diag_wait_limit failed: %d" % st)
    torch.cuda.synchronize(device)
    return int(gave_up.item()), e0.elapsed_time(e1)
