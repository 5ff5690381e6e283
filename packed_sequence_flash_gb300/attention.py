"""Python binding of libpsf.so: argument marshalling only.

Every function allocates its outputs and workspace with torch (device memory
and the current stream are all torch provides) and calls the C ABI; every step
of the computation runs in the library's CUDA kernels. Non-zero return codes
raise ``PSFError`` (a ``ValueError``).

Layouts follow the pages:
  * varlen: packed ``[T, H, D]`` with ``lse [H, T]``
    [ffpa_attention page, ``_ffpa_varlen_fwd``];
  * dense: ``[B, H, N, D]`` with ``lse [B, H, N]``
    [ffpa_attention page, ``_ffpa_dense_fwd``];
  * document-causal: ``[B, H, S, D]`` (or packed ``[S, H, D]`` for one row)
    [fa4 page, ``document_causal_fa4_attention``].
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (PSF_BWD_PACK_GQA, PSF_DTYPE_BF16, PSF_DTYPE_F16, PSF_FWD_PACK_GQA, PSF_LAYOUT_BHSD, PSF_LAYOUT_THD,
                   PSF_SEGMENTS_SKIP_PAD, check)

NO_WINDOW = -(2 ** 31)  # the pages' "no window" sentinel


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _window(window) -> int:
    if window is None:
        return NO_WINDOW
    return int(window)


_DTYPES = {torch.bfloat16: PSF_DTYPE_BF16, torch.float16: PSF_DTYPE_F16}


def _dtype_code(tensors, strided=False):
    """PSF_DTYPE_* of a call's 16-bit tensors ((tensor, name) pairs), which must share one type.
    strided: the call takes strides (else every tensor must be contiguous)."""
    t0, n0 = tensors[0]
    if t0.dtype not in _DTYPES:
        raise ValueError(f"{n0} must be bfloat16 or float16, got {t0.dtype}")
    for t, n in tensors:
        (_need_view if strided else _need)(t, n, t0.dtype)
    return _DTYPES[t0.dtype]


def _grads_like(q, k, v):
    """Gradient buffers with their inputs' strides where those are non-overlapping
    and dense, else in a dense layout (torch.empty_like's rule)."""
    return tuple(torch.empty_like(t) for t in (q, k, v))


def _need(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _i32(t, name):
    _need(t, name, torch.int32)
    return t


def _need_view(t, name, dtype=None):
    """A strided CUDA tensor whose head dim is contiguous and whose data starts on a 16-byte boundary
    (the kernels read every tensor through TMA views built from its strides)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name}: the last (head) dim must be contiguous")
    if t.data_ptr() % 16:
        raise ValueError(f"{name}: data must start on a 16-byte boundary")


def _strides(tensors, layout):
    """The C ABI's strides argument: NULL when every tensor is contiguous, else
    int64 (batch, head, row) element strides per tensor ([T, H, D] tensors have
    no batch dim: its stride is ignored)."""
    if all(t.is_contiguous() for t in tensors):
        return None
    vals = []
    for t in tensors:
        if layout == PSF_LAYOUT_THD:
            vals += [0, t.stride(1), t.stride(0)]
        else:
            vals += [t.stride(0), t.stride(1), t.stride(2)]
    return (ctypes.c_int64 * len(vals))(*vals)


def device_status(clear: bool = True) -> int:
    """Synchronise and return the kernel-side status (0, PSF_EDEVICE_ARGS or PSF_ETIMEOUT)."""
    return _lib.load().psf_device_status(1 if clear else 0)


def check_device_status() -> None:
    rc = device_status(True)
    check(rc)


def set_wait_limit_ns(ns: int) -> None:
    _lib.load().psf_set_wait_limit_ns(int(ns))


def check_pipeline_wait(arrive: bool) -> None:
    """Launch the bounded-wait check on the current stream: with arrive=False
    its wait runs out after the wait limit and records PSF_ETIMEOUT, which
    device_status() then returns; with arrive=True it records nothing."""
    check(_lib.load().psf_check_pipeline_wait(1 if arrive else 0, _stream()))


def fwd_workspace_size(total_q_rows: int, nseg: int) -> int:
    return int(_lib.load().psf_attn_fwd_workspace_size(int(total_q_rows), int(nseg)))


def bwd_workspace_size(total_q_rows: int, total_k_rows: int, nseg: int, Hq: int, Hkv: int, Dqk: int,
                       Dv: int) -> int:
    return int(_lib.load().psf_attn_bwd_workspace_size(int(total_q_rows), int(total_k_rows), int(nseg), int(Hq),
                                                       int(Hkv), int(Dqk), int(Dv)))


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# varlen (packed THD, or BHSD rows when layout="bhsd")

def _varlen_dims(q, k, v, layout):
    if layout == "thd":
        Tq, Hq, Dqk = q.shape
        Tk, Hkv, _ = k.shape
        return PSF_LAYOUT_THD, 1, Tq, Tk, Hq, Hkv, Dqk, v.shape[2]
    B, Hq, Sq, Dqk = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    return PSF_LAYOUT_BHSD, B, Sq, Sk, Hq, Hkv, Dqk, v.shape[3]


def _cap(softcap):
    return float(softcap) if softcap else 0.0


def attn_varlen_fwd(q, k, v, cu_q, cu_k, max_q, max_k, scale, causal, window=None, dev_meta=None,
                    layout="thd", out=None, lse=None, workspace=None, pack_gqa=False, softcap=None):
    """Packed varlen forward -> (out, lse). cu_q/cu_k int32 [nseg+1] on the device.
    q, k, v: bf16 or fp16 (one type); out has their type, lse is fp32.
    pack_gqa: the query heads of a KV head share one tile (same results; for
    short segments). softcap > 0 caps each logit as softcap * tanh(logit / softcap)."""
    dt = _dtype_code([(q, "q"), (k, "k"), (v, "v")], strided=True)
    _i32(cu_q, "cu_q")
    _i32(cu_k, "cu_k")
    lay, B, Sq, Sk, Hq, Hkv, Dqk, Dv = _varlen_dims(q, k, v, layout)
    nseg = cu_q.numel() - 1
    if out is None:
        out = torch.empty(*q.shape[:-1], Dv, dtype=q.dtype, device=q.device)
    else:
        _need_view(out, "out", q.dtype)
    if lse is None:
        lse = torch.empty((Hq, Sq) if lay == PSF_LAYOUT_THD else (B, Hq, Sq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(fwd_workspace_size(B * Sq, nseg), q.device)
    rc = _lib.load().psf_attn_varlen_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_q), _ptr(cu_k), _ptr(dev_meta), nseg,
        int(max_q), int(max_k), lay, dt, B, Sq, Sk, Hq, Hkv, Dqk, Dv, _strides((q, k, v, out), lay), float(scale),
        int(bool(causal)),
        _window(window), _cap(softcap), PSF_FWD_PACK_GQA if pack_gqa else 0, _ptr(workspace), workspace.numel(),
        _stream())
    check(rc)
    return out, lse


def attn_varlen_bwd(dout, q, k, v, out, lse, cu_q, cu_k, max_q, max_k, scale, causal, window=None,
                    dev_meta=None, layout="thd", workspace=None, softcap=None, pack_gqa=False):
    """Packed varlen backward from caller-supplied out/lse -> (dq, dk, dv) in the inputs' type.
    pack_gqa: each step takes a KV head's query heads together (same results)."""
    dt = _dtype_code([(dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")], strided=True)
    _need(lse, "lse", torch.float32)
    _i32(cu_q, "cu_q")
    _i32(cu_k, "cu_k")
    lay, B, Sq, Sk, Hq, Hkv, Dqk, Dv = _varlen_dims(q, k, v, layout)
    nseg = cu_q.numel() - 1
    dq, dk, dv = _grads_like(q, k, v)
    if workspace is None:
        workspace = _workspace(bwd_workspace_size(B * Sq, B * Sk, nseg, Hq, Hkv, Dqk, Dv), q.device)
    rc = _lib.load().psf_attn_varlen_bwd(
        _ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_q),
        _ptr(cu_k), _ptr(dev_meta), nseg, int(max_q), int(max_k), lay, dt, B, Sq, Sk, Hq, Hkv, Dqk, Dv,
        _strides((q, k, v, out, dout, dq, dk, dv), lay), float(scale), int(bool(causal)), _window(window), _cap(softcap), PSF_BWD_PACK_GQA if pack_gqa else 0, _ptr(workspace),
        workspace.numel(), _stream())
    check(rc)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# dense [B, H, N, D]

def attn_dense_fwd(q, k, v, scale, causal, window=None, workspace=None, pack_gqa=False, softcap=None):
    """Dense forward -> (out [B,Hq,Nq,Dv] in the inputs' type, lse [B,Hq,Nq] fp32).
    q, k, v may be strided views (for example ``x.transpose(1, 2)`` of a [B, N, H, D]
    tensor) whose head dim is contiguous; they are read in place."""
    dt = _dtype_code([(q, "q"), (k, "k"), (v, "v")], strided=True)
    B, Hq, Nq, Dqk = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    out = torch.empty(B, Hq, Nq, Dv, dtype=q.dtype, device=q.device)
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(fwd_workspace_size(B * Nq, B), q.device)
    rc = _lib.load().psf_attn_dense_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, Dqk,
                                        Dv, _strides((q, k, v, out), PSF_LAYOUT_BHSD), dt, float(scale), int(bool(causal)), _window(window), _cap(softcap),
                                        PSF_FWD_PACK_GQA if pack_gqa else 0, _ptr(workspace), workspace.numel(),
                                        _stream())
    check(rc)
    return out, lse


def attn_dense_bwd(dout, q, k, v, out, lse, scale, causal, window=None, workspace=None, softcap=None,
                   pack_gqa=False):
    """Dense backward -> (dq, dk, dv) in [B,H,N,D], dk/dv at Hkv heads; each
    gradient has its input's strides (strided inputs are read in place)."""
    dt = _dtype_code([(dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")], strided=True)
    _need(lse, "lse", torch.float32)
    B, Hq, Nq, Dqk = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    dq, dk, dv = _grads_like(q, k, v)
    if workspace is None:
        workspace = _workspace(bwd_workspace_size(B * Nq, B * Nk, B, Hq, Hkv, Dqk, Dv), q.device)
    rc = _lib.load().psf_attn_dense_bwd(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dq),
                                        _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nk, Dqk, Dv,
                                        _strides((q, k, v, out, dout, dq, dk, dv), PSF_LAYOUT_BHSD), dt, float(scale),
                                        int(bool(causal)), _window(window), _cap(softcap),
                                        PSF_BWD_PACK_GQA if pack_gqa else 0, _ptr(workspace), workspace.numel(),
                                        _stream())
    check(rc)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# segment builder, pad fixup, merge

def build_doc_segments(kv_doc_ids, q_length, q_global_start, capacity=None, want_pad_flags=False, skip_pad=False):
    """Doc ids [B, Sk] int32 (device) -> (cu_q, cu_k, dev_meta, seg_is_pad).

    dev_meta = int32 [nseg, max_q, max_k] on the device; cu arrays hold
    capacity + 1 entries of which the first nseg + 1 are meaningful.
    skip_pad: padding pieces become (their queries, no keys) + (no queries,
    their keys), so the attention itself zeroes padding queries.
    """
    _i32(kv_doc_ids, "kv_doc_ids")
    if kv_doc_ids.dim() == 1:
        kv_doc_ids = kv_doc_ids[None]
    B, Sk = kv_doc_ids.shape
    if capacity is None:
        capacity = (B * Sk + B) * (2 if skip_pad else 1)
    dev = kv_doc_ids.device
    cu_q = torch.empty(capacity + 1, dtype=torch.int32, device=dev)
    cu_k = torch.empty(capacity + 1, dtype=torch.int32, device=dev)
    meta = torch.empty(3, dtype=torch.int32, device=dev)
    pad = torch.empty(max(capacity, 1), dtype=torch.uint8, device=dev) if want_pad_flags else None
    rc = _lib.load().psf_build_doc_segments(_ptr(kv_doc_ids), B, Sk, int(q_length), int(q_global_start),
                                            _ptr(cu_q), _ptr(cu_k), int(capacity), _ptr(meta), _ptr(pad),
                                            PSF_SEGMENTS_SKIP_PAD if skip_pad else 0, _stream())
    check(rc)
    return cu_q, cu_k, meta, pad


def chunk_dense_eligible(kv_doc_ids, q_start, q_length, k_start, k_length):
    """(local, cross) dense-kernel eligibility of the key chunk
    [k_start, k_start + k_length) for the query shard [q_start, q_start + q_length)
    of every row of kv_doc_ids [B, S] (device int32): see psf_chunk_dense_flags.
    Reads the two flags back to the host (one synchronisation)."""
    _i32(kv_doc_ids, "kv_doc_ids")
    if kv_doc_ids.dim() == 1:
        kv_doc_ids = kv_doc_ids[None]
    B, S = kv_doc_ids.shape
    flags = torch.empty(2, dtype=torch.int32, device=kv_doc_ids.device)
    check(_lib.load().psf_chunk_dense_flags(_ptr(kv_doc_ids), B, S, int(q_start), int(q_length), int(k_start),
                                            int(k_length), _ptr(flags), _stream()))
    f = flags.tolist()
    return bool(f[0]), bool(f[1])


def chunk_attention(q, k, v, kv_doc_ids, q_start, k_start, scale, causal, window=None, dense=None, softcap=None):
    """One chunk of the ring decomposition on one device: the query shard
    [q_start, q_start + Lq) of every row, q [B, Hq, Lq, Dqk], against the key
    chunk [k_start, k_start + Lk), k [B, Hkv, Lk, Dqk] / v [B, Hkv, Lk, Dv], with
    kv_doc_ids [B, S] the whole rows' ids.

    causal=True is the local role (the chunk ends where the shard ends; the
    document-causal mask, optional left window); causal=False the cross role
    (the chunk before the shard, no mask inside the shared document).
    dense=None routes by chunk_dense_eligible (one host read); True / False
    force the dense kernels (then pad_fixup) or the segment path. softcap > 0
    caps the logits (the backward takes it from the plan).
    Returns (out, lse, plan); plan feeds chunk_attention_backward.
    """
    if not causal and window is not None:
        raise ValueError("a cross chunk runs without a window")
    B, Hq, Lq, _ = q.shape
    Lk = k.shape[2]
    if dense is None:
        local, cross = chunk_dense_eligible(kv_doc_ids, q_start, Lq, k_start, Lk)
        dense = local if causal else cross
    if dense:
        out, lse = attn_dense_fwd(q, k, v, scale, causal, window, softcap=softcap)
        pad_fixup(out, lse, kv_doc_ids[:, q_start:q_start + Lq].contiguous(), "bhsd")
        return out, lse, ("dense", causal, window, softcap)
    if causal:
        ids_chunk = kv_doc_ids[:, k_start:k_start + Lk].contiguous()
        cu_q, cu_k, meta, _ = build_doc_segments(ids_chunk, Lq, q_start - k_start, skip_pad=True)
    else:
        cu_q, cu_k, meta = build_cross_segments(kv_doc_ids, q_start, Lq, k_start, Lk)
    out, lse = attn_varlen_fwd(q, k, v, cu_q, cu_k, -1, -1, scale, causal, window, dev_meta=meta, layout="bhsd",
                               softcap=softcap)
    return out, lse, ("segments", causal, window, softcap, cu_q, cu_k, meta)


def chunk_attention_backward(dout, q, k, v, out, lse, plan, scale):
    """Backward of chunk_attention from the (possibly merged) out/lse -> (dq, dk, dv)."""
    if plan[0] == "dense":
        return attn_dense_bwd(dout, q, k, v, out, lse, scale, plan[1], plan[2], softcap=plan[3])
    _, causal, window, softcap, cu_q, cu_k, meta = plan
    return attn_varlen_bwd(dout, q, k, v, out, lse, cu_q, cu_k, -1, -1, scale, causal, window, dev_meta=meta,
                           layout="bhsd", softcap=softcap)


def pad_fixup(out, lse, q_doc_ids, layout="thd"):
    """In place: rows with query doc id 0 get out = 0 and lse = -inf."""
    _dtype_code([(out, "out")])
    _need(lse, "lse", torch.float32)
    _i32(q_doc_ids, "q_doc_ids")
    if layout == "thd":
        Lq, Hq, Dv = out.shape
        B, lay = 1, PSF_LAYOUT_THD
    else:
        B, Hq, Lq, Dv = out.shape
        lay = PSF_LAYOUT_BHSD
    rc = _lib.load().psf_pad_fixup(_ptr(out), _ptr(lse), _ptr(q_doc_ids), lay, B, Lq, Hq, Dv, _stream())
    check(rc)
    return out, lse


def lse_merge(o1, l1, o2, l2, want_f32=True, want_bf16=False):
    """Merge two partial results over disjoint keys: o [T,H,D] bf16, l [H,T] fp32."""
    dt = _dtype_code([(o1, "o1"), (o2, "o2")])
    for t, n in ((l1, "l1"), (l2, "l2")):
        _need(t, n, torch.float32)
    T, H, D = o1.shape
    of = torch.empty(T, H, D, dtype=torch.float32, device=o1.device) if want_f32 else None
    ob = torch.empty(T, H, D, dtype=o1.dtype, device=o1.device) if want_bf16 else None
    l = torch.empty(H, T, dtype=torch.float32, device=o1.device)
    rc = _lib.load().psf_lse_merge(_ptr(o1), _ptr(l1), _ptr(o2), _ptr(l2), _ptr(of), _ptr(ob), _ptr(l), T, H, D,
                                   dt, _stream())
    check(rc)
    return of, ob, l


def build_cross_segments(kv_doc_ids, q_start, q_length, k_start, k_length):
    """Segments of the shard [q_start, q_start + q_length) against the earlier
    key chunk [k_start, k_start + k_length) of every row of kv_doc_ids [B, S]
    (device int32) -> (cu_q, cu_k, dev_meta), 3 segments per row; run the chunk
    with causal=False."""
    _i32(kv_doc_ids, "kv_doc_ids")
    if kv_doc_ids.dim() == 1:
        kv_doc_ids = kv_doc_ids[None]
    B, S = kv_doc_ids.shape
    dev = kv_doc_ids.device
    cu_q = torch.empty(3 * B + 1, dtype=torch.int32, device=dev)
    cu_k = torch.empty(3 * B + 1, dtype=torch.int32, device=dev)
    meta = torch.empty(3, dtype=torch.int32, device=dev)
    rc = _lib.load().psf_build_cross_segments(_ptr(kv_doc_ids), B, S, int(q_start), int(q_length), int(k_start),
                                              int(k_length), _ptr(cu_q), _ptr(cu_k), _ptr(meta), _stream())
    check(rc)
    return cu_q, cu_k, meta


def lse_merge_live_rows(o_run, l_acc, o_new, l_new, cu_q, cu_k, dev_meta=None, o_acc=None):
    """In place: merge (o_new, l_new) into the running (o_run / o_acc, l_acc) on
    the query rows of the segments that have keys. o_run bf16 [T,H,D] (may be
    None when o_acc, fp32 [T,H,D], holds the running output), l_acc fp32 [H,T]."""
    dt = _dtype_code([(o_new, "o_new")] + ([(o_run, "o_run")] if o_run is not None else []))
    for t, n in ((l_acc, "l_acc"), (l_new, "l_new")):
        _need(t, n, torch.float32)
    if o_acc is not None:
        _need(o_acc, "o_acc", torch.float32)
    T, H, D = o_new.shape
    rc = _lib.load().psf_lse_merge_live_rows(_ptr(o_acc), _ptr(o_run), _ptr(l_acc), _ptr(o_new), _ptr(l_new),
                                             _ptr(cu_q), _ptr(cu_k), _ptr(dev_meta), cu_q.numel() - 1, T, H, D, dt,
                                             _stream())
    check(rc)


def grad_add_live_rows(dst, src, cu_q, cu_k, dev_meta=None):
    """In place: dst += src (bf16 [T,H,D]) on the query rows of the segments that have keys."""
    dt = _dtype_code([(dst, "dst"), (src, "src")])
    T, H, D = dst.shape
    rc = _lib.load().psf_grad_add_live_rows(_ptr(dst), _ptr(src), _ptr(cu_q), _ptr(cu_k), _ptr(dev_meta),
                                            cu_q.numel() - 1, T, H, D, dt, _stream())
    check(rc)


# ---------------------------------------------------------------------------
# document-causal composition [fa4 page, document_causal_fa4_attention]

def document_causal_attention(q, k, v, q_doc_ids, kv_doc_ids, q_global_start, scale, window=None, skip_pad=True,
                              pack_gqa=True, softcap=None):
    """Causal per-document attention of a local query shard against global keys.

    q [B, Hq, Lq, Dqk], k [B, Hkv, Sk, Dqk], v [B, Hkv, Sk, Dv] (or packed
    [Lq, Hq, Dqk] / [Sk, Hkv, D] for a single row); doc ids [B, Lq] / [B, Sk]
    int32, 1-based, 0 = padding. Returns (out, lse, segments) where padding
    queries are zero with lse -inf, and segments = (cu_q, cu_k, dev_meta) for
    the backward. No host synchronisation: the segment count stays on the device.
    skip_pad (default): padding runs get segments without keys for their
    queries, so the attention writes their zero rows itself and computes no
    padding pairs; False runs padding runs as ordinary segments and zeroes
    the padding queries afterwards with pad_fixup (q_doc_ids is read only then).
    pack_gqa (default): the forward packs a KV head's query heads into one
    tile where the shape allows it (head dims 64 and 128); the results are the
    same and packed documents run faster; False takes one head per tile.
    softcap > 0 caps the logits (pass the same value to the backward).
    """
    layout = "thd" if q.dim() == 3 else "bhsd"
    if kv_doc_ids.dim() == 1:
        kv_doc_ids = kv_doc_ids[None]
    if q_doc_ids.dim() == 1:
        q_doc_ids = q_doc_ids[None]
    Lq = q.shape[0] if layout == "thd" else q.shape[2]
    cu_q, cu_k, meta, _ = build_doc_segments(kv_doc_ids, Lq, q_global_start, skip_pad=skip_pad)
    out, lse = attn_varlen_fwd(q, k, v, cu_q, cu_k, -1, -1, scale, True, window, dev_meta=meta, layout=layout,
                               pack_gqa=pack_gqa, softcap=softcap)
    if not skip_pad:
        pad_fixup(out, lse, q_doc_ids, layout)
    return out, lse, (cu_q, cu_k, meta)


def document_causal_attention_backward(dout, q, k, v, out, lse, segments, scale, window=None, softcap=None,
                                       pack_gqa=True):
    """Backward of document_causal_attention from its out/lse -> (dq, dk, dv).
    pack_gqa (default): a step takes the query heads of a KV head together where
    the shape allows it (head dims up to 128, 2 or 4 query heads per KV head, no
    softcap); same results."""
    layout = "thd" if q.dim() == 3 else "bhsd"
    cu_q, cu_k, meta = segments
    return attn_varlen_bwd(dout, q, k, v, out, lse, cu_q, cu_k, -1, -1, scale, True, window, dev_meta=meta,
                           layout=layout, softcap=softcap, pack_gqa=pack_gqa)
