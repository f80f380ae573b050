"""The C ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU (CPU only: no compute call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


@pytest.fixture(scope="module")
def lib():
    from channelwise_gated_delta_gb300 import _binding
    from channelwise_gated_delta_gb300 import build as cbuild
    cbuild.build()
    return _binding.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDR_API\s+[\w\s\*]+?\b(gdr_\w+)\s*\(", text)))


def test_header_declares_the_api():
    syms = declared_symbols()
    for s in ("gdr_forward", "gdr_forward_ex", "gdr_workspace_bytes", "gdr_device_check",
              "gdr_status_string", "gdr_last_cuda_error", "gdr_version"):
        assert s in syms


def test_every_declared_symbol_is_exported(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), "libgdr.so does not export %s" % s


def test_internal_symbols_are_hidden(lib):
    # only the C ABI is visible; kernels and launchers are not
    assert not hasattr(lib, "_ZN3gdr13launch_decodeERKNS_7ProblemEP11CUstream_st")


def test_status_strings_and_version(lib):
    for st in range(9):
        assert lib.gdr_status_string(st).decode().startswith("GDR_")
    assert lib.gdr_version().decode().count(".") == 2


FAKE = 1 << 40  # 16-byte aligned host address that is never dereferenced


def call(lib, B=1, T=4, HK=1, HV=2, dk=32, dv=32, chunk=16, dtype=1, ptrs=None, ws=None,
         ws_bytes=0, flags=0):
    step = 1 << 30
    p = dict(q=FAKE, k=FAKE + step, v=FAKE + 2 * step, g=FAKE + 3 * step, beta=FAKE + 4 * step,
             h0=FAKE + 5 * step, out=FAKE + 6 * step, ht=FAKE + 7 * step)
    if ptrs:
        p.update(ptrs)
    args = [ctypes.c_void_p(p[n]) if p[n] is not None else None
            for n in ("q", "k", "v", "g", "beta", "h0", "out", "ht")]
    return lib.gdr_forward_ex(*args, B, T, HK, HV, dk, dv, chunk, None, dtype,
                              None if ws is None else ctypes.c_void_p(ws), ws_bytes, flags)


@pytest.mark.parametrize("kw,status", [
    (dict(HK=2, HV=3), 2),                 # HV % HK != 0
    (dict(B=-1), 2),
    (dict(T=-3), 2),
    (dict(HK=0), 2),
    (dict(dk=48), 3),                      # unsupported head dim
    (dict(dv=256), 3),
    (dict(chunk=128), 3),
    (dict(dtype=7), 3),
    (dict(ptrs=dict(q=None)), 1),
    (dict(ptrs=dict(out=None)), 1),
    (dict(ptrs=dict(g=FAKE + (3 << 30) + 4)), 4),     # misaligned
    (dict(ptrs=dict(beta=FAKE + (4 << 30) + 2)), 4),  # beta needs 4-byte alignment
    (dict(ptrs=dict(out=FAKE + 16)), 8),               # out overlaps q
    (dict(ptrs=dict(ht=FAKE + (1 << 30))), 8),         # ht overlaps k
    (dict(ptrs=dict(ht=FAKE + (5 << 30) + 16)), 8),    # ht partially overlaps h0
    (dict(T=40), 5),                                   # prefill needs a workspace, none given
])
def test_bad_arguments_rejected_before_launch(lib, kw, status):
    assert call(lib, **kw) == status


def test_workspace_sizes(lib):
    # decode needs none; the CUDA-core prefill needs one record per chunk
    assert lib.gdr_workspace_bytes(64, 1, 16, 32, 128, 128, 64, 1, 0) == 0
    small = lib.gdr_workspace_bytes(1, 40, 1, 2, 32, 32, 16, 0, 0)
    assert small > 0
    assert lib.gdr_workspace_bytes(1, 1, 1, 2, 32, 32, 16, 0, 1) > 0   # forced chunked at T=1
    assert lib.gdr_workspace_bytes(1, 40, 2, 3, 32, 32, 16, 0, 0) == 0  # invalid shape
    # a workspace one byte short is rejected
    assert call(lib, T=40, dtype=0, ws=FAKE + (9 << 30), ws_bytes=small - 1) == 5
    # misaligned workspace
    assert call(lib, T=40, dtype=0, ws=FAKE + (9 << 30) + 16, ws_bytes=small) == 4


def test_segmented_scan_workspace(lib):
    """Forced segments on the tensor-core route: 2P - 3 f32 states per
    (batch, value head) plus small tables; none when segments are off, the
    route is the CUDA-core one, or the sequence has fewer than two chunks."""
    from channelwise_gated_delta_gb300 import GDR_FLAG_NO_SEGMENTS, gdr_flag_segments
    state = 128 * 128 * 4
    for B, T, HV, P, P_eff in [(1, 4096, 32, 3, 3), (2, 1000, 4, 5, 4), (1, 200, 2, 2, 2),
                               (1, 4096, 2, 255, 64)]:
        need = lib.gdr_workspace_bytes(B, T, HV // 2, HV, 128, 128, 64, 1, gdr_flag_segments(P))
        states = B * (2 * P_eff - 3) * HV * state
        assert states <= need < states + 64 * 1024 + B * (3 * P_eff) * 1024, (B, T, HV, P)
    seg3 = gdr_flag_segments(3)
    assert lib.gdr_workspace_bytes(1, 4096, 16, 32, 128, 128, 64, 1,
                                   seg3 | GDR_FLAG_NO_SEGMENTS) == 0
    assert lib.gdr_workspace_bytes(1, 64, 1, 2, 128, 128, 64, 1, seg3) == 0   # one chunk
    # no device here, so the automatic choice never segments
    assert lib.gdr_workspace_bytes(1, 4096, 16, 32, 128, 128, 64, 1, 0) == 0
    # missing or short workspace: rejected before any launch
    need = lib.gdr_workspace_bytes(1, 4096, 16, 32, 128, 128, 64, 1, seg3)
    kw = dict(T=4096, HK=16, HV=32, dk=128, dv=128, chunk=64, dtype=1, flags=seg3)
    assert call(lib, **kw) == 5
    assert call(lib, ws=FAKE + (9 << 30), ws_bytes=need - 1, **kw) == 5
    with pytest.raises(ValueError):
        gdr_flag_segments(1)


def test_scan_route_segmented_workspace(lib):
    """The chunk-record route (f32 q/k/v, or chunk 32): forced segments add
    2P - 3 f32 states per (batch, value head) and small run tables after the
    records; none with GDR_FLAG_NO_SEGMENTS, on the CUDA-core scan
    (GDR_FLAG_FORCE_GENERIC), for dk != 128, or with one chunk."""
    from channelwise_gated_delta_gb300 import (GDR_FLAG_FORCE_GENERIC, GDR_FLAG_NO_SEGMENTS,
                                               gdr_flag_segments)
    state = 128 * 128 * 4
    for B, T, HV, chunk, dt, P, P_eff in [(1, 4096, 32, 32, 1, 3, 3), (1, 4096, 32, 64, 0, 3, 3),
                                          (2, 1000, 4, 64, 0, 5, 4), (1, 300, 2, 16, 0, 7, 7),
                                          (1, 200, 2, 64, 0, 2, 2)]:
        ws = lambda f: lib.gdr_workspace_bytes(B, T, HV // 2, HV, 128, 128, chunk, dt, f)
        rec = ws(0 if P_eff < 3 else GDR_FLAG_NO_SEGMENTS)
        assert rec > 0
        extra = ws(gdr_flag_segments(P)) - ((rec + 255) // 256 * 256)
        states = B * (2 * P_eff - 3) * HV * state
        assert states < extra <= states + 3 * 256 + B * 3 * P_eff * 32, (B, T, HV, chunk, P)
        assert ws(gdr_flag_segments(P) | GDR_FLAG_FORCE_GENERIC) == ws(GDR_FLAG_FORCE_GENERIC)
    seg3 = gdr_flag_segments(3)
    f32 = lambda dk, T, f: lib.gdr_workspace_bytes(1, T, 1, 2, dk, dk, 64, 0, f)
    assert f32(64, 4096, seg3) == f32(64, 4096, 0)       # dk = 64: not segmented
    assert f32(128, 64, seg3) == f32(128, 64, 0)         # one chunk
    assert f32(128, 4096, seg3 | GDR_FLAG_NO_SEGMENTS) == f32(128, 4096, GDR_FLAG_NO_SEGMENTS)
    # no device here, so the automatic choice never segments
    assert f32(128, 4096, 0) == f32(128, 4096, GDR_FLAG_NO_SEGMENTS)


def test_varlen_scan_route_segmented_workspace(lib):
    """Packed f32 batches: the forced count cuts every chunk-record
    sequence spread over exactly P segments, each with 2P - 3 states per value
    head; decode tokens and shorter sequences are not cut."""
    from channelwise_gated_delta_gb300 import GDR_FLAG_NO_SEGMENTS, gdr_flag_segments
    HV, state = 4, 128 * 128 * 4
    ws = lambda cu, f: lib.gdr_varlen_workspace_bytes(cu_array(cu), len(cu) - 1, 2, HV, 128,
                                                      128, 64, 0, f)
    cu = [0, 1000, 1001, 1701, 1741]   # 16 chunks, one token, 11 chunks, 1 chunk
    base = ws(cu, GDR_FLAG_NO_SEGMENTS)
    assert ws(cu, 0) == base
    assert ws(cu, gdr_flag_segments(5)) == base   # 16 and 11 chunks both spread over 4
    for P, cut in [(3, 2), (2, 2), (4, 2), (16, 1), (11, 1)]:
        extra = ws(cu, gdr_flag_segments(P)) - (base + 255) // 256 * 256
        states = cut * (2 * P - 3) * HV * state
        assert states < extra <= states + 3 * 256 + cut * 3 * P * 32, (P, extra)
    assert ws([0, 40, 80], gdr_flag_segments(3)) == ws([0, 40, 80], 0)


@pytest.mark.parametrize("T", [65, 128, 129, 300, 1000, 4096, 4097])
@pytest.mark.parametrize("P", [2, 3, 4, 5, 7, 16, 100])
def test_segment_count_matches_oracle_bounds(lib, T, P):
    """The library's segment plan (read back from its state slots: 2P-3 per
    batch element and head) cuts a sequence into as many pieces as the
    oracle's segment_bounds, which are written independently."""
    import oracle
    from channelwise_gated_delta_gb300 import gdr_flag_segments
    B, HV = 2, 4
    need = lib.gdr_workspace_bytes(B, T, 2, HV, 128, 128, 64, 1, gdr_flag_segments(P))
    want = len(oracle.segment_bounds(T, 64, P))
    if want < 2:
        assert need == 0
        return
    state = B * HV * 128 * 128 * 4
    slots = need // state              # the tables and two rows stay under one slot
    assert slots == 2 * want - 3, (T, P, slots, want)


def test_set_workspace_argument_checks(lib):
    """gdr_set_workspace checks its arguments before it looks for a device."""
    assert lib.gdr_set_workspace(None, 4096) == 1                  # GDR_ERR_NULL
    assert lib.gdr_set_workspace(ctypes.c_void_p(FAKE + 16), 4096) == 4  # GDR_ERR_ALIGN


def test_binding_fails_loudly_without_library(tmp_path):
    from channelwise_gated_delta_gb300 import _binding
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load_library(str(tmp_path / "missing.so"))


def cu_array(vals):
    return (ctypes.c_int * len(vals))(*vals)


def call_varlen(lib, cu, N=None, HK=1, HV=2, dk=32, dv=32, chunk=16, dtype=0, ptrs=None, ws=None,
                ws_bytes=0, flags=0):
    step = 1 << 30
    p = dict(q=FAKE, k=FAKE + step, v=FAKE + 2 * step, g=FAKE + 3 * step, beta=FAKE + 4 * step,
             h0=FAKE + 5 * step, out=FAKE + 6 * step, ht=FAKE + 7 * step)
    if ptrs:
        p.update(ptrs)
    args = [ctypes.c_void_p(p[n]) if p[n] is not None else None
            for n in ("q", "k", "v", "g", "beta", "h0", "out", "ht")]
    n = len(cu) - 1 if N is None else N
    arr = None if cu is None else cu_array(cu)
    return lib.gdr_forward_varlen(*args, arr, n, HK, HV, dk, dv, chunk, None, dtype,
                                  None if ws is None else ctypes.c_void_p(ws), ws_bytes, flags)


@pytest.mark.parametrize("cu,kw,status", [
    ([1, 4, 8], {}, 2),             # cu_seqlens[0] != 0
    ([0, 5, 4], {}, 2),             # decreasing offsets
    ([0, 4], dict(N=-1), 2),        # negative count
    (None, dict(N=2), 1),           # no offsets
    ([0, 4, 8], dict(HK=2, HV=3), 2),
    ([0, 4, 8], dict(dk=48), 3),
    ([0, 4, 8], dict(ptrs=dict(q=None)), 1),
    ([0, 4, 8], dict(ptrs=dict(out=FAKE + 16)), 8),     # out overlaps q
    ([0, 4, 8], dict(ptrs=dict(ht=FAKE + (5 << 30) + 16)), 8),
    ([0, 4, 8], {}, 5),             # needs a workspace, none given
])
def test_varlen_bad_arguments_rejected_before_launch(lib, cu, kw, status):
    assert call_varlen(lib, cu, **kw) == status


def test_varlen_segmented_workspace(lib):
    """A packed batch with forced segments: the sequences whose chunks spread
    over the count get 2P - 3 f32 states per value head in the workspace (the
    rest of the batch as before); on this machine (no device) the automatic
    choice cuts nothing."""
    from channelwise_gated_delta_gb300 import GDR_FLAG_NO_SEGMENTS, gdr_flag_segments
    state = 128 * 128 * 4
    ws = lambda cu, flags: lib.gdr_varlen_workspace_bytes(cu_array(cu), len(cu) - 1, 2, 4, 128,
                                                          128, 64, 1, flags)
    cu = [0, 1000, 1001, 1701, 1741]       # 1000 and 700 tokens cut, 1 decodes, 40 walks
    base = ws(cu, 0)
    assert base == ws(cu, GDR_FLAG_NO_SEGMENTS)
    for P, ncut in [(3, 2), (2, 2)]:
        extra = ws(cu, gdr_flag_segments(P)) - base
        states = ncut * (2 * P - 3) * 4 * state
        assert states <= extra < states + 64 * 1024, (P, extra)
    assert ws(cu, gdr_flag_segments(5) | GDR_FLAG_NO_SEGMENTS) == base
    assert ws([0, 40, 80], gdr_flag_segments(3)) == ws([0, 40, 80], 0)  # nothing spreads that far


def test_varlen_workspace_sizes(lib):
    ws = lambda cu, **kw: lib.gdr_varlen_workspace_bytes(
        cu_array(cu), len(cu) - 1, kw.get("HK", 1), kw.get("HV", 2), kw.get("dk", 32),
        kw.get("dv", 32), kw.get("chunk", 16), kw.get("dtype", 0), kw.get("flags", 0))
    assert ws([0]) == 0                     # no sequences
    assert ws([0, 0, 0]) == 0               # only empty ones: nothing to stage
    one = ws([0, 1])                        # one single-token sequence: its table row
    assert 0 < one <= 512
    small = ws([0, 40])
    more = ws([0, 40, 80])                  # twice the chunk records
    assert small > one and more > small
    assert ws([0, 40, 80], HK=2, HV=3) == 0  # invalid shape
    assert ws([1, 40]) == 0                  # invalid offsets
    # a workspace one byte short, or misaligned, is rejected
    assert call_varlen(lib, [0, 40], ws=FAKE + (9 << 30), ws_bytes=small - 1) == 5
    assert call_varlen(lib, [0, 40], ws=FAKE + (9 << 30) + 16, ws_bytes=small) == 4


def call_tree(lib, parent, B=1, T=4, HK=1, HV=2, dk=32, dv=32, dtype=0, ws=None, ws_bytes=0):
    step = 1 << 30
    args = [ctypes.c_void_p(FAKE + n * step) for n in range(7)]
    arr = None if parent is None else cu_array(parent)
    return lib.gdr_forward_tree(*args, arr, B, T, HK, HV, dk, dv, None, dtype,
                                None if ws is None else ctypes.c_void_p(ws), ws_bytes, 0)


@pytest.mark.parametrize("parent,kw,status", [
    ([-1, 0, 0, 1], dict(T=513), 3),        # more than 512 tokens
    ([-1, 0, 3, 1], {}, 2),                  # parent after its child
    ([-1, -2, 0, 1], {}, 2),                 # parent below -1
    (None, {}, 1),                           # no parents
    ([-1, 0, 0, 1], dict(dk=48), 3),
    ([-1, 0, 0, 1], {}, 5),                  # needs a workspace
])
def test_tree_bad_arguments_rejected_before_launch(lib, parent, kw, status):
    assert call_tree(lib, parent, **kw) == status


def test_tree_workspace_sizes(lib):
    assert lib.gdr_tree_workspace_bytes(1, 0, 1, 2, 32, 32, 0, 0) == 0
    assert lib.gdr_tree_workspace_bytes(1, 513, 1, 2, 32, 32, 0, 0) == 0
    # past 64 tokens (or forced): the blocked solve -- parents, ancestor masks,
    # path sums, block references, spread flags and column operands
    # (channelwise gates), the block-pair fragments (bf16 pairs hi + lo for
    # f32), their flags and the f32 diagonal blocks
    def up(x):
        return (x + 255) // 256 * 256

    def blocked(B, T, HV, dk, m, scalar=False):
        Tp = 32 if T <= 32 else (T + 31) // 32 * 32
        NB = (T + 15) // 16
        NTRI = NB * (NB + 1) // 2
        trees = B * HV
        refs = 0 if scalar else (up(trees * NB * dk * 4) + up(trees * NB * (dk // 8) * 4)
                                 + up(trees * Tp * (dk // 2) * m * 4))
        return (up(B * T * 4) + up(B * Tp * (Tp // 32) * 4) + up(trees * Tp * (1 if scalar else dk) * 4)
                + refs + up(trees * NTRI * 2 * m * 128 * 4) + up(trees * NTRI * 4)
                + up(trees * NB * 256 * 4))
    assert lib.gdr_tree_workspace_bytes(1, 65, 1, 2, 32, 32, 0, 0) == blocked(1, 65, 2, 32, 2)
    assert lib.gdr_tree_workspace_bytes(3, 512, 2, 4, 128, 64, 1, 0) == blocked(3, 512, 4, 128, 1)
    assert lib.gdr_tree_workspace_bytes(2, 64, 1, 2, 128, 128, 1, 0x10000) == blocked(2, 64, 2, 128, 1)
    assert lib.gdr_tree_workspace_bytes(2, 300, 1, 2, 64, 64, 1, 4) == blocked(2, 300, 2, 64, 1, True)
    small = lib.gdr_tree_workspace_bytes(1, 16, 1, 2, 32, 32, 0, 0)
    assert 0 < small < lib.gdr_tree_workspace_bytes(1, 17, 1, 2, 32, 32, 0, 0)
    # tensor-core route (bf16, d = 128): the parents only
    assert lib.gdr_tree_workspace_bytes(2, 64, 1, 2, 128, 128, 1, 0) == 512
    assert lib.gdr_tree_workspace_bytes(2, 64, 1, 2, 128, 128, 1, 2) > 512  # forced CUDA cores
    assert call_tree(lib, [-1, 0, 0, 1], ws=FAKE + (9 << 30), ws_bytes=small - 1) == 5


def test_host_entry_rejections(lib):
    assert lib.gdr_host_staging_bytes(0, 10, 1, 2, 32, 32, 16, 0) == 0
    assert lib.gdr_host_staging_bytes(2, 10, 2, 3, 32, 32, 16, 0) == 0
    one = lib.gdr_host_staging_bytes(1, 10, 1, 2, 32, 32, 16, 0)
    assert 0 < one and lib.gdr_host_staging_bytes(5, 10, 1, 2, 32, 32, 16, 0) == 2 * one
    step = 1 << 30
    ptrs = [ctypes.c_void_p(FAKE + n * step) for n in range(8)]
    args = lambda **kw: [kw.get("B", 2), 10, 1, 2, kw.get("dk", 32), 32, 16, None, 0]
    assert lib.gdr_forward_host(*ptrs, *args(), None, 0) == 5             # no staging
    assert lib.gdr_forward_host(*ptrs, *args(dk=48), None, 0) == 3
    assert lib.gdr_forward_host(*ptrs, *args(B=-1), None, 0) == 2
    assert lib.gdr_forward_host(*ptrs, *args(), ctypes.c_void_p(FAKE + (9 << 30) + 16),
                                2 * one) == 4                              # misaligned
