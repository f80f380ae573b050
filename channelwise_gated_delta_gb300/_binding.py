"""ctypes binding of libgdr.so (the C ABI in include/gdr.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their data pointers and the current CUDA stream are handed to the
library, and a non-OK status becomes an exception.  Every step of the forward
pass runs in the library's CUDA kernels; there is no fallback of any kind, and
the first call raises if the library has not been built.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgdr.so")

GDR_OK = 0
GDR_F32 = 0
GDR_BF16 = 1
GDR_FLAG_FORCE_CHUNKED = 1
GDR_FLAG_FORCE_GENERIC = 2
GDR_FLAG_SCALAR_GATE = 4
GDR_FLAG_NO_SEGMENTS = 8
GDR_FLAG_TREE_BLOCKED = 0x10000
GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD = 0x20000


def gdr_flag_segments(n):
    """Flag bits that make the tensor-core route cut the state scan into at
    most ``n`` segments (2 <= n <= 255), whatever the device."""
    if not 2 <= n <= 255:
        raise ValueError("segment count must be in 2 .. 255")
    return (n & 0xFF) << 8

STATUS_NAMES = {0: "GDR_OK", 1: "GDR_ERR_NULL", 2: "GDR_ERR_SHAPE", 3: "GDR_ERR_UNSUPPORTED",
                4: "GDR_ERR_ALIGN", 5: "GDR_ERR_WORKSPACE", 6: "GDR_ERR_CUDA",
                7: "GDR_ERR_TIMEOUT", 8: "GDR_ERR_ALIAS"}

EXPORTED = ("gdr_workspace_bytes", "gdr_set_workspace", "gdr_forward_ex", "gdr_forward",
            "gdr_forward_chunked_noalloc",
            "gdr_varlen_workspace_bytes", "gdr_forward_varlen", "gdr_tree_workspace_bytes",
            "gdr_forward_tree", "gdr_host_staging_bytes", "gdr_forward_host", "gdr_device_check",
            "gdr_trace_enable", "gdr_trace_read", "gdr_status_string",
            "gdr_last_cuda_error", "gdr_version")

_lib = None


class GdrError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(msg)
        self.status = status


def load_library(path=LIB_PATH):
    """Loads libgdr.so and declares its signatures.  Raises if it is missing."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            "libgdr.so is not built (%s). Build it with `python -c \"import __graft_entry__ as g; "
            "g.build()\"` or `python channelwise_gated_delta_gb300/build.py`." % path)
    lib = ctypes.CDLL(path)
    vp, sz, i, u = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint
    fwd = [vp] * 8 + [i] * 7 + [vp, i]
    lib.gdr_set_workspace.argtypes = [vp, sz]
    lib.gdr_set_workspace.restype = i
    lib.gdr_workspace_bytes.argtypes = [i] * 8 + [u]
    lib.gdr_workspace_bytes.restype = sz
    lib.gdr_forward_ex.argtypes = fwd + [vp, sz, u]
    lib.gdr_forward_ex.restype = i
    lib.gdr_forward.argtypes = fwd
    lib.gdr_forward.restype = i
    lib.gdr_forward_chunked_noalloc.argtypes = fwd
    lib.gdr_forward_chunked_noalloc.restype = i
    ip = ctypes.POINTER(i)
    lib.gdr_varlen_workspace_bytes.argtypes = [ip, i, i, i, i, i, i, i, u]
    lib.gdr_varlen_workspace_bytes.restype = sz
    lib.gdr_forward_varlen.argtypes = [vp] * 8 + [ip] + [i] * 6 + [vp, i, vp, sz, u]
    lib.gdr_forward_varlen.restype = i
    lib.gdr_tree_workspace_bytes.argtypes = [i] * 7 + [u]
    lib.gdr_tree_workspace_bytes.restype = sz
    lib.gdr_forward_tree.argtypes = [vp] * 7 + [ip] + [i] * 6 + [vp, i, vp, sz, u]
    lib.gdr_forward_tree.restype = i
    lib.gdr_host_staging_bytes.argtypes = [i] * 8
    lib.gdr_host_staging_bytes.restype = sz
    lib.gdr_forward_host.argtypes = fwd + [vp, sz]
    lib.gdr_forward_host.restype = i
    lib.gdr_device_check.argtypes = [vp]
    lib.gdr_device_check.restype = i
    lib.gdr_status_string.argtypes = [i]
    lib.gdr_status_string.restype = ctypes.c_char_p
    lib.gdr_last_cuda_error.argtypes = []
    lib.gdr_last_cuda_error.restype = i
    lib.gdr_version.argtypes = []
    lib.gdr_version.restype = ctypes.c_char_p
    lib.gdr_trace_enable.argtypes = [i]
    lib.gdr_trace_enable.restype = i
    lib.gdr_trace_read.argtypes = [i, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i),
                                   ctypes.POINTER(ctypes.c_double)]
    lib.gdr_trace_read.restype = i
    if path == LIB_PATH:
        _lib = lib
    return lib


def _check(lib, st):
    if st != GDR_OK:
        msg = lib.gdr_status_string(st).decode()
        if st == 6:
            msg += " (cudaError %d)" % lib.gdr_last_cuda_error()
        raise GdrError(st, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return GDR_BF16
    if dt == torch.float32:
        return GDR_F32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % dt)


def gdr_workspace_bytes(B, T, HK, HV, dk, dv, chunk=64, dtype=torch.bfloat16, flags=0):
    lib = load_library()
    return int(lib.gdr_workspace_bytes(B, T, HK, HV, dk, dv, chunk, _dtype_code(dtype), flags))


def gdr_forward(q, k, v, g, beta, h0=None, out=None, ht=None, chunk=64, stream=None,
                workspace=None, flags=0, store_ht=True):
    """Channelwise gated delta rule forward on the GPU.

    q, k [B, T, HK, dk]; v [B, T, HV, dv] (bf16 or f32, all the same dtype);
    g [B, T, HV, dk] f32; beta [B, T, HV] f32; h0 [B, HV, dk, dv] f32 or None.
    ``out`` / ``ht`` are allocated when not given (``ht=h0`` updates in place;
    ``store_ht=False`` skips the final state).  The workspace, if the route
    needs one, is allocated from torch's allocator unless passed in.
    Enqueued on ``stream`` (default: torch's current stream).  Returns (out, ht).
    """
    lib = load_library()
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    dev = q.device
    code = _dtype_code(q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0),
                    ("out", out), ("ht", ht)):
        if t is None:
            continue
        if t.device != dev or dev.type != "cuda":
            raise ValueError("%s must be a CUDA tensor on %s" % (name, dev))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if k.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k must match q in shape and dtype; v must match q in dtype")
    if tuple(g.shape) == (B, T, HV):   # a scalar gate: one log-decay per token and head
        flags |= GDR_FLAG_SCALAR_GATE
    elif tuple(g.shape) != (B, T, HV, dk):
        raise ValueError("g must be [B, T, HV, dk] (channelwise) or [B, T, HV] (scalar gate)")
    if tuple(v.shape[:2]) != (B, T) or tuple(beta.shape) != (B, T, HV):
        raise ValueError("inconsistent shapes")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if h0 is not None and (tuple(h0.shape) != (B, HV, dk, dv) or h0.dtype != torch.float32):
        raise ValueError("h0 must be float32 [B, HV, dk, dv]")
    if out is None:
        out = torch.empty(B, T, HV, dv, dtype=q.dtype, device=dev)
    if ht is None and store_ht:
        ht = torch.empty(B, HV, dk, dv, dtype=torch.float32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    need = int(lib.gdr_workspace_bytes(B, T, HK, HV, dk, dv, chunk, code, flags))
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if need > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if need > 0 else 0
    st = lib.gdr_forward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(out),
                            _ptr(ht), B, T, HK, HV, dk, dv, chunk,
                            ctypes.c_void_p(stream.cuda_stream), code, ws_ptr, ws_bytes, flags)
    _check(lib, st)
    return out, ht


_registered_ws = {}


def gdr_set_workspace(workspace, device=None):
    """Registers ``workspace`` (a CUDA uint8 tensor, 256-byte aligned, or None
    to go back to the library's own) as the workspace of the C entry
    ``gdr_forward`` on its device.  A reference is kept while registered."""
    lib = load_library()
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        with torch.cuda.device(dev):
            _check(lib, lib.gdr_set_workspace(None, 0))
        _registered_ws.pop(dev.index, None)
        return
    if workspace.device.type != "cuda":
        raise ValueError("the workspace must be a CUDA tensor")
    with torch.cuda.device(workspace.device):
        _check(lib, lib.gdr_set_workspace(_ptr(workspace),
                                          workspace.numel() * workspace.element_size()))
    _registered_ws[workspace.device.index] = workspace


def _cu_array(cu_seqlens):
    """cu_seqlens (a sequence of ints or a CPU integer tensor) as a ctypes int32 array."""
    if isinstance(cu_seqlens, torch.Tensor):
        if cu_seqlens.device.type != "cpu":
            raise ValueError("cu_seqlens must be host memory (a CPU tensor or a list)")
        cu_seqlens = cu_seqlens.tolist()
    vals = [int(x) for x in cu_seqlens]
    if not vals:
        raise ValueError("cu_seqlens needs at least one entry")
    return (ctypes.c_int * len(vals))(*vals), len(vals) - 1


def gdr_varlen_workspace_bytes(cu_seqlens, HK, HV, dk, dv, chunk=64, dtype=torch.bfloat16, flags=0):
    lib = load_library()
    cu, n = _cu_array(cu_seqlens)
    return int(lib.gdr_varlen_workspace_bytes(cu, n, HK, HV, dk, dv, chunk, _dtype_code(dtype),
                                              flags))


def gdr_forward_varlen(q, k, v, g, beta, cu_seqlens, h0=None, out=None, ht=None, chunk=64,
                       stream=None, workspace=None, flags=0, store_ht=True):
    """Packed variable-length batch: N sequences stored back to back.

    q, k [total, HK, dk]; v [total, HV, dv]; g [total, HV, dk] f32; beta [total, HV]
    f32 (a leading batch dim of 1 is accepted and kept on ``out``); cu_seqlens
    host ints [N + 1]; h0 / ht [N, HV, dk, dv] f32.  Returns (out, ht).
    """
    lib = load_library()
    cu, n = _cu_array(cu_seqlens)
    lead = q.dim() == 4
    if lead:
        if q.shape[0] != 1:
            raise ValueError("a packed batch has a leading dim of 1")
        q, k, v, g, beta = q[0], k[0], v[0], g[0], beta[0]
    total, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    dev = q.device
    code = _dtype_code(q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0),
                    ("out", out), ("ht", ht)):
        if t is None:
            continue
        if t.device != dev or dev.type != "cuda":
            raise ValueError("%s must be a CUDA tensor on %s" % (name, dev))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if cu[n] != total:
        raise ValueError("cu_seqlens[-1] (%d) != number of token rows (%d)" % (cu[n], total))
    if k.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k must match q in shape and dtype; v must match q in dtype")
    if tuple(g.shape) == (total, HV):   # a scalar gate
        flags |= GDR_FLAG_SCALAR_GATE
    elif tuple(g.shape) != (total, HV, dk):
        raise ValueError("g must be [total, HV, dk] (channelwise) or [total, HV] (scalar gate)")
    if v.shape[0] != total or tuple(beta.shape) != (total, HV):
        raise ValueError("inconsistent shapes")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if h0 is not None and (tuple(h0.shape) != (n, HV, dk, dv) or h0.dtype != torch.float32):
        raise ValueError("h0 must be float32 [N, HV, dk, dv]")
    if out is None:
        out = torch.empty(total, HV, dv, dtype=q.dtype, device=dev)
    elif out.dim() == 4:
        out = out[0]
    if ht is None and store_ht:
        ht = torch.empty(n, HV, dk, dv, dtype=torch.float32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    need = int(lib.gdr_varlen_workspace_bytes(cu, n, HK, HV, dk, dv, chunk, code, flags))
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if need > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if need > 0 else 0
    st = lib.gdr_forward_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                _ptr(out), _ptr(ht), cu, n, HK, HV, dk, dv, chunk,
                                ctypes.c_void_p(stream.cuda_stream), code, ws_ptr, ws_bytes, flags)
    _check(lib, st)
    return (out.unsqueeze(0) if lead else out), ht


def gdr_tree_workspace_bytes(B, T, HK, HV, dk, dv, dtype=torch.bfloat16, flags=0):
    lib = load_library()
    return int(lib.gdr_tree_workspace_bytes(B, T, HK, HV, dk, dv, _dtype_code(dtype), flags))


def gdr_forward_tree(q, k, v, g, beta, parent, h0=None, out=None, stream=None, workspace=None,
                     flags=0):
    """Tree verification: each batch element's T <= 512 tokens form a draft
    tree given by ``parent`` (host ints [B, T], parent[b, t] in [-1, t-1]);
    every token's output is that of the recurrence run along its root path
    from h0[b].  Tensors as in gdr_forward.  Returns out [B, T, HV, dv]."""
    lib = load_library()
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    dev = q.device
    code = _dtype_code(q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0),
                    ("out", out)):
        if t is None:
            continue
        if t.device != dev or dev.type != "cuda":
            raise ValueError("%s must be a CUDA tensor on %s" % (name, dev))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if k.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k must match q in shape and dtype; v must match q in dtype")
    if tuple(g.shape) == (B, T, HV):   # a scalar gate
        flags |= GDR_FLAG_SCALAR_GATE
    elif tuple(g.shape) != (B, T, HV, dk):
        raise ValueError("g must be [B, T, HV, dk] (channelwise) or [B, T, HV] (scalar gate)")
    if tuple(v.shape[:2]) != (B, T) or tuple(beta.shape) != (B, T, HV):
        raise ValueError("inconsistent shapes")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if h0 is not None and (tuple(h0.shape) != (B, HV, dk, dv) or h0.dtype != torch.float32):
        raise ValueError("h0 must be float32 [B, HV, dk, dv]")
    par = torch.as_tensor(parent, dtype=torch.int32, device="cpu").contiguous()
    if tuple(par.shape) != (B, T):
        raise ValueError("parent must be [B, T]")
    par_c = par.numpy().ctypes.data_as(ctypes.POINTER(ctypes.c_int))
    if out is None:
        out = torch.empty(B, T, HV, dv, dtype=q.dtype, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    need = int(lib.gdr_tree_workspace_bytes(B, T, HK, HV, dk, dv, code, flags))
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if need > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if need > 0 else 0
    st = lib.gdr_forward_tree(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(out),
                              par_c, B, T, HK, HV, dk, dv, ctypes.c_void_p(stream.cuda_stream), code,
                              ws_ptr, ws_bytes, flags)
    _check(lib, st)
    return out


def gdr_host_staging_bytes(B, T, HK, HV, dk, dv, chunk=64, dtype=torch.bfloat16):
    lib = load_library()
    return int(lib.gdr_host_staging_bytes(B, T, HK, HV, dk, dv, chunk, _dtype_code(dtype)))


def gdr_forward_host(q, k, v, g, beta, h0, out, ht, chunk=64, stream=None, staging=None,
                     device=None):
    """The forward pass on HOST tensors (CPU, pinned for overlap): copies in,
    computes and copies out through the library, batch elements pipelined
    through two device slots.  Shapes as in gdr_forward; ``out`` and ``ht``
    (may be None, or ``ht is h0``) are host tensors written by the call,
    complete once ``stream`` (default: the current stream of ``device``)
    reaches the call's end.  Returns (out, ht)."""
    lib = load_library()
    B, T, HK, dk = q.shape
    HV, dv = v.shape[2], v.shape[3]
    code = _dtype_code(q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0),
                    ("out", out), ("ht", ht)):
        if t is None:
            continue
        if t.device.type != "cpu":
            raise ValueError("%s must be a host tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if k.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype or out.dtype != q.dtype:
        raise ValueError("k, v and out must match q in dtype (and k in shape)")
    if tuple(v.shape[:2]) != (B, T) or tuple(g.shape) != (B, T, HV, dk) or \
            tuple(beta.shape) != (B, T, HV) or tuple(out.shape) != (B, T, HV, dv):
        raise ValueError("inconsistent shapes")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    for name, t in (("h0", h0), ("ht", ht)):
        if t is not None and (tuple(t.shape) != (B, HV, dk, dv) or t.dtype != torch.float32):
            raise ValueError("%s must be float32 [B, HV, dk, dv]" % name)
    dev = torch.device("cuda") if device is None else torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    need = int(lib.gdr_host_staging_bytes(B, T, HK, HV, dk, dv, chunk, code))
    if need > 0 and (staging is None or staging.numel() * staging.element_size() < need):
        staging = torch.empty(need, dtype=torch.uint8, device=dev)
    st_ptr = _ptr(staging) if need > 0 else None
    st_bytes = staging.numel() * staging.element_size() if need > 0 else 0
    st = lib.gdr_forward_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                              _ptr(out), _ptr(ht), B, T, HK, HV, dk, dv, chunk,
                              ctypes.c_void_p(stream.cuda_stream), code, st_ptr, st_bytes)
    _check(lib, st)
    return out, ht


def gdr_device_check(stream=None):
    """Waits for the stream and raises if a kernel reported a bounded-wait timeout."""
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream()
    _check(lib, lib.gdr_device_check(ctypes.c_void_p(stream.cuda_stream)))


def gdr_trace_enable(on=True):
    """Starts (or stops) recording CUDA events around every launch of the library."""
    load_library().gdr_trace_enable(1 if on else 0)


def gdr_trace_read():
    """Waits for the traced launches and returns {kernel name: (launches, total ms)}
    for every kernel kind launched since tracing was enabled (records are cleared)."""
    lib = load_library()
    n = 32
    names = (ctypes.c_char_p * n)()
    launches = (ctypes.c_int * n)()
    total = (ctypes.c_double * n)()
    got = lib.gdr_trace_read(n, names, launches, total)
    if got < 0:
        raise GdrError(6, "gdr_trace_read: a CUDA event query failed")
    return {names[i].decode(): (launches[i], total[i]) for i in range(got) if launches[i] > 0}


def gdr_version():
    return load_library().gdr_version().decode()
