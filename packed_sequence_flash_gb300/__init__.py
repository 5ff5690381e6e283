"""Packed-sequence flash attention for GB300 (sm_103a).

Exact softmax attention over packed variable-length sequences: forward with an
fp32 log-sum-exp, backward from caller-supplied out/lse with dK/dV reduced to
the KV heads, and the doc-ids -> varlen-segment builder. The compute runs in
hand-written tcgen05/TMA kernels inside libpsf.so (C ABI in include/psf.h);
this package only marshals arguments.
"""
from .attention import (NO_WINDOW, attn_dense_bwd, attn_dense_fwd, attn_varlen_bwd, attn_varlen_fwd,
                        build_cross_segments, build_doc_segments, bwd_workspace_size, check_device_status,
                        check_pipeline_wait, chunk_attention, chunk_attention_backward, chunk_dense_eligible,
                        device_status, document_causal_attention, document_causal_attention_backward,
                        fwd_workspace_size, grad_add_live_rows, lse_merge, lse_merge_live_rows, pad_fixup,
                        set_wait_limit_ns)
from ._lib import PSFError

__all__ = [
    "NO_WINDOW", "PSFError", "attn_dense_bwd", "attn_dense_fwd", "attn_varlen_bwd", "attn_varlen_fwd",
    "build_cross_segments", "build_doc_segments", "bwd_workspace_size", "check_device_status",
    "check_pipeline_wait", "chunk_attention", "chunk_attention_backward", "chunk_dense_eligible", "device_status",
    "document_causal_attention", "document_causal_attention_backward", "fwd_workspace_size",
    "grad_add_live_rows", "lse_merge", "lse_merge_live_rows", "pad_fixup", "set_wait_limit_ns",
]
