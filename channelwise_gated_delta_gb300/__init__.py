"""GB300 (sm_103a) channelwise gated delta rule forward.

The compute lives in libgdr.so (C ABI: include/gdr.h); this package is its
thin Python binding plus the seeded synthetic input generator.
"""
from ._binding import (GDR_BF16, GDR_F32, GDR_FLAG_FORCE_CHUNKED, GDR_FLAG_FORCE_GENERIC,
                       GDR_FLAG_NO_SEGMENTS, GDR_FLAG_SCALAR_GATE, GDR_FLAG_TREE_BLOCKED,
                       GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD,
                       gdr_flag_segments,
                       GdrError, gdr_device_check, gdr_forward, gdr_forward_host,
                       gdr_forward_tree, gdr_host_staging_bytes,
                       gdr_forward_varlen, gdr_tree_workspace_bytes,
                       gdr_set_workspace,
                       gdr_trace_enable,
                       gdr_trace_read, gdr_version,
                       gdr_varlen_workspace_bytes, gdr_workspace_bytes, load_library)

__all__ = ["gdr_forward", "gdr_workspace_bytes", "gdr_forward_varlen", "gdr_varlen_workspace_bytes",
           "gdr_forward_tree", "gdr_tree_workspace_bytes", "gdr_forward_host",
           "gdr_host_staging_bytes", "gdr_device_check", "gdr_version", "gdr_set_workspace",
           "gdr_trace_enable", "gdr_trace_read",
           "load_library", "GdrError", "GDR_F32", "GDR_BF16", "GDR_FLAG_FORCE_CHUNKED",
           "GDR_FLAG_FORCE_GENERIC", "GDR_FLAG_SCALAR_GATE", "GDR_FLAG_NO_SEGMENTS",
           "GDR_FLAG_TREE_BLOCKED", "GDR_FLAG_TREE_GRAM_PER_VALUE_HEAD",
           "gdr_flag_segments"]
