"""fp64 CPU oracle for packed-sequence softmax attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product path never
imports this package, and this package imports nothing from the product.

The arithmetic lives in ``psf_oracle.c`` (plain C, double precision); this
module marshals numpy arrays to it. Inputs arrive as whatever dtype the caller
has and are converted exactly to float64 (bf16 and fp32 values are exactly
representable in fp64).

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: library routines on special cases, closed forms, central
finite differences, invariants and hand-derived segment lists.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "psf_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

MODE_SEGMENTS = 0
MODE_DOCUMENT = 1


def build(force: bool = False) -> str:
    """Compile psf_oracle.c into liboracle.so next to it (gcc, a second or two)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [I, I, I, P, P, I, P, I, I, I, I,
                                            P, P, P, I, I, I, I, I, I, D, D, P, I, P, P, I]
            lib.oracle_attn_fwd.restype = I
            lib.oracle_attn_bwd.argtypes = [I, I, I, P, P, I, P, I, I, I, I,
                                            P, P, P, P, P, P, I, I, I, I, I, I, D, D,
                                            P, I, P, I, P, P, P, I]
            lib.oracle_attn_bwd.restype = I
            lib.oracle_build_segments.argtypes = [P, I, I, I, I, P, P, I, P, P, I]
            lib.oracle_build_segments.restype = I
            lib.oracle_lse_merge.argtypes = [P, P, P, P, P, P, I, I, I]
            lib.oracle_build_cross_segments.argtypes = [P, I, I, I, I, I, I, P, P, P, P]
            lib.oracle_build_cross_segments.restype = I
            lib.oracle_lse_merge.restype = None
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu")
        import torch

        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray | None:
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _window(window) -> int:
    if window is None:
        return 0
    w = int(window)
    return w if w > 0 else 0


def _mask_args(mode, causal, window, cu_q, cu_k, doc_ids, B, Sk, Lq, q0):
    nseg = 0 if cu_q is None else len(cu_q) - 1
    return [mode, int(bool(causal)), _window(window), _ptr(cu_q), _ptr(cu_k), nseg,
            _ptr(doc_ids), B, Sk, Lq, q0]


# ---------------------------------------------------------------------------
# forward

def _softcap(softcap) -> float:
    return float(softcap) if softcap is not None and softcap > 0 else 0.0


def _fwd(mode, q, k, v, scale, causal, window, cu_q=None, cu_k=None, doc_ids=None, B=0, Sk=0,
         Lq=0, q0=0, rows=None, nthreads=None, softcap=None):
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, Dqk = q.shape
    Tk, Hkv, _ = k.shape
    Dv = v.shape[2]
    out = np.zeros((Tq, Hq, Dv), dtype=np.float64)
    lse = np.full((Hq, Tq), -np.inf, dtype=np.float64)
    rows = _i32(rows)
    rc = lib.oracle_attn_fwd(*_mask_args(mode, causal, window, cu_q, cu_k, doc_ids, B, Sk, Lq, q0),
                             _ptr(q), _ptr(k), _ptr(v), Tq, Tk, Hq, Hkv, Dqk, Dv, float(scale),
                             _softcap(softcap), _ptr(rows), 0 if rows is None else len(rows), _ptr(out), _ptr(lse),
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd failed ({rc})")
    return out, lse


def attn_fwd_segments(q, k, v, cu_q, cu_k, scale, causal, window=None, rows=None, nthreads=None, softcap=None):
    """Packed forward: q [Tq,Hq,Dqk], k [Tk,Hkv,Dqk], v [Tk,Hkv,Dv] -> out [Tq,Hq,Dv], lse [Hq,Tq].
    softcap > 0 caps each logit as softcap * tanh(logit / softcap)."""
    return _fwd(MODE_SEGMENTS, q, k, v, scale, causal, window, cu_q=_i32(cu_q), cu_k=_i32(cu_k),
                rows=rows, nthreads=nthreads, softcap=softcap)


def attn_fwd_document(q, k, v, doc_ids, q_global_start, scale, window=None, rows=None,
                      nthreads=None, softcap=None):
    """Document-causal forward with the mask materialised from doc ids.

    q [B*Lq, Hq, Dqk] (batch-major rows), k/v [B*Sk, Hkv, D]; doc_ids [B, Sk].
    """
    doc_ids = _i32(doc_ids)
    B, Sk = doc_ids.shape
    Lq = q.shape[0] // B
    return _fwd(MODE_DOCUMENT, q, k, v, scale, True, window, doc_ids=doc_ids, B=B, Sk=Sk, Lq=Lq,
                q0=int(q_global_start), rows=rows, nthreads=nthreads, softcap=softcap)


def attn_fwd_dense(q, k, v, scale, causal, window=None, nthreads=None, softcap=None):
    """Dense forward on [B,H,N,D]: out [B,Hq,Nq,Dv], lse [B,Hq,Nq]; causal is bottom-right."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, Dqk = q.shape
    Nk = k.shape[2]
    qp = q.transpose(0, 2, 1, 3).reshape(B * Nq, Hq, Dqk)
    kp = k.transpose(0, 2, 1, 3).reshape(B * Nk, k.shape[1], Dqk)
    vp = v.transpose(0, 2, 1, 3).reshape(B * Nk, v.shape[1], v.shape[3])
    cu_q = np.arange(B + 1, dtype=np.int32) * Nq
    cu_k = np.arange(B + 1, dtype=np.int32) * Nk
    out, lse = attn_fwd_segments(qp, kp, vp, cu_q, cu_k, scale, causal, window, nthreads=nthreads,
                                 softcap=softcap)
    out = out.reshape(B, Nq, Hq, -1).transpose(0, 2, 1, 3)
    lse = lse.reshape(Hq, B, Nq).transpose(1, 0, 2)
    return np.ascontiguousarray(out), np.ascontiguousarray(lse)


# ---------------------------------------------------------------------------
# backward

def _bwd(mode, dout, q, k, v, out, lse, scale, causal, window, cu_q=None, cu_k=None, doc_ids=None,
         B=0, Sk=0, Lq=0, q0=0, q_rows=None, k_rows=None, want_dq=True, want_dkdv=True,
         nthreads=None, softcap=None):
    lib = _load()
    dout, q, k, v, out, lse = (_f64(x) for x in (dout, q, k, v, out, lse))
    Tq, Hq, Dqk = q.shape
    Tk, Hkv, _ = k.shape
    Dv = v.shape[2]
    dq = np.zeros((Tq, Hq, Dqk)) if want_dq else None
    dk = np.zeros((Tk, Hkv, Dqk)) if want_dkdv else None
    dv = np.zeros((Tk, Hkv, Dv)) if want_dkdv else None
    q_rows, k_rows = _i32(q_rows), _i32(k_rows)
    rc = lib.oracle_attn_bwd(*_mask_args(mode, causal, window, cu_q, cu_k, doc_ids, B, Sk, Lq, q0),
                             _ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), Tq, Tk,
                             Hq, Hkv, Dqk, Dv, float(scale), _softcap(softcap), _ptr(q_rows),
                             0 if q_rows is None else len(q_rows), _ptr(k_rows),
                             0 if k_rows is None else len(k_rows), _ptr(dq), _ptr(dk), _ptr(dv),
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd failed ({rc})")
    return dq, dk, dv


def attn_bwd_segments(dout, q, k, v, out, lse, cu_q, cu_k, scale, causal, window=None, q_rows=None,
                      k_rows=None, want_dq=True, want_dkdv=True, nthreads=None, softcap=None):
    """Packed backward from caller-supplied out [Tq,Hq,Dv] / lse [Hq,Tq] -> dq, dk, dv."""
    return _bwd(MODE_SEGMENTS, dout, q, k, v, out, lse, scale, causal, window, cu_q=_i32(cu_q),
                cu_k=_i32(cu_k), q_rows=q_rows, k_rows=k_rows, want_dq=want_dq,
                want_dkdv=want_dkdv, nthreads=nthreads, softcap=softcap)


def attn_bwd_document(dout, q, k, v, out, lse, doc_ids, q_global_start, scale, window=None,
                      q_rows=None, k_rows=None, want_dq=True, want_dkdv=True, nthreads=None, softcap=None):
    doc_ids = _i32(doc_ids)
    B, Sk = doc_ids.shape
    Lq = q.shape[0] // B
    return _bwd(MODE_DOCUMENT, dout, q, k, v, out, lse, scale, True, window, doc_ids=doc_ids, B=B,
                Sk=Sk, Lq=Lq, q0=int(q_global_start), q_rows=q_rows, k_rows=k_rows,
                want_dq=want_dq, want_dkdv=want_dkdv, nthreads=nthreads, softcap=softcap)


def attn_bwd_dense(dout, q, k, v, out, lse, scale, causal, window=None, nthreads=None, softcap=None):
    """Dense backward on [B,H,N,D] with lse [B,Hq,Nq]; returns dq, dk, dv in [B,H,N,D]."""
    dout, q, k, v, out, lse = (_f64(x) for x in (dout, q, k, v, out, lse))
    B, Hq, Nq, Dqk = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    Dv = v.shape[3]

    def pack(x):
        return x.transpose(0, 2, 1, 3).reshape(B * x.shape[2], x.shape[1], x.shape[3])

    lse_p = lse.transpose(1, 0, 2).reshape(Hq, B * Nq)
    cu_q = np.arange(B + 1, dtype=np.int32) * Nq
    cu_k = np.arange(B + 1, dtype=np.int32) * Nk
    dq, dk, dv = attn_bwd_segments(pack(dout), pack(q), pack(k), pack(v), pack(out), lse_p, cu_q,
                                   cu_k, scale, causal, window, nthreads=nthreads, softcap=softcap)

    def unpack(x, N, H, D):
        return np.ascontiguousarray(x.reshape(B, N, H, D).transpose(0, 2, 1, 3))

    return unpack(dq, Nq, Hq, Dqk), unpack(dk, Nk, Hkv, Dqk), unpack(dv, Nk, Hkv, Dv)


# ---------------------------------------------------------------------------
# segment builder and merge

def build_segments(doc_ids, q_length, q_global_start, skip_pad=False):
    """Doc ids [B, Sk] -> (cu_q, cu_k, max_q, max_k) as numpy int32 arrays and ints.
    skip_pad: every padding piece becomes (its queries, no keys) then (no
    queries, its keys)."""
    lib = _load()
    doc_ids = _i32(doc_ids)
    if doc_ids.ndim == 1:
        doc_ids = doc_ids[None, :]
    B, Sk = doc_ids.shape
    cap = 2 * B * (Sk + 1) + 2
    cu_q = np.zeros(cap + 1, dtype=np.int32)
    cu_k = np.zeros(cap + 1, dtype=np.int32)
    mq = np.zeros(1, dtype=np.int32)
    mk = np.zeros(1, dtype=np.int32)
    n = lib.oracle_build_segments(_ptr(doc_ids), B, Sk, int(q_length), int(q_global_start),
                                  _ptr(cu_q), _ptr(cu_k), cap, _ptr(mq), _ptr(mk), 1 if skip_pad else 0)
    if n < 0:
        raise ValueError("oracle_build_segments: capacity exceeded")
    return cu_q[: n + 1].copy(), cu_k[: n + 1].copy(), int(mq[0]), int(mk[0])


def build_cross_segments(doc_ids, q_start, q_length, k_start, k_length):
    """Cross-chunk segments of the shard [q_start, q_start + q_length) against
    the earlier key chunk [k_start, k_start + k_length) of every row of
    doc_ids [B, S] -> (cu_q, cu_k, max_q, max_k)."""
    lib = _load()
    doc_ids = _i32(doc_ids)
    if doc_ids.ndim == 1:
        doc_ids = doc_ids[None, :]
    B, S = doc_ids.shape
    cu_q = np.zeros(3 * B + 1, dtype=np.int32)
    cu_k = np.zeros(3 * B + 1, dtype=np.int32)
    mq = np.zeros(1, dtype=np.int32)
    mk = np.zeros(1, dtype=np.int32)
    n = lib.oracle_build_cross_segments(_ptr(doc_ids), B, S, int(q_start), int(q_length), int(k_start),
                                        int(k_length), _ptr(cu_q), _ptr(cu_k), _ptr(mq), _ptr(mk))
    if n < 0:
        raise ValueError("oracle_build_cross_segments: the key chunk must lie before the query shard")
    return cu_q, cu_k, int(mq[0]), int(mk[0])


def row_is_single_document(ids_row):
    """Exactly one document with no padding: every position holds the same id > 0.
    [cp_attention page, the row predicate behind the dense_cross flag of
    `_build_packed_ring_segments`]"""
    ids_row = [int(x) for x in np.asarray(ids_row).reshape(-1)]
    return len(ids_row) > 0 and ids_row[0] > 0 and all(x == ids_row[0] for x in ids_row)


def row_is_document_prefix(ids_row):
    """The real (> 0) tokens are one document forming a contiguous prefix and the
    padding, if any, is a trailing suffix (an all-padding row qualifies).
    [cp_attention page, the row predicate behind the dense_local flag]"""
    ids_row = [int(x) for x in np.asarray(ids_row).reshape(-1)]
    k = 0
    while k < len(ids_row) and ids_row[k] != 0:
        k += 1
    return len(set(ids_row[:k])) <= 1 and all(x == 0 for x in ids_row[k:])


def chunk_dense_flags(doc_ids, q_start, q_length, k_start, k_length):
    """(local, cross): whether the key chunk [k_start, k_start + k_length) may run
    through the dense kernel for the query shard [q_start, q_start + q_length)
    of every row of doc_ids [B, S], in the local role (causal; the chunk ends
    where the shard ends and contains it; every row's chunk a document prefix)
    or the cross role (non-causal; the chunk before the shard; every row's
    [k_start, q_start) one document without padding that the shard starts with
    and holds alone, padding only as its suffix).
    [cp_attention page, `_build_packed_ring_segments` dense flags,
    `_chunk_dense_eligible`]"""
    ids = np.asarray(doc_ids)
    if ids.ndim == 1:
        ids = ids[None]
    q_end, k_end = q_start + q_length, k_start + k_length
    local = q_length > 0 and k_start <= q_start and k_end == q_end and all(
        row_is_document_prefix(row[k_start:k_end]) for row in ids)
    cross = q_length > 0 and k_length > 0 and k_end <= q_start and all(
        row_is_single_document(row[k_start:q_start]) and row[q_start] == row[k_start]
        and row_is_document_prefix(row[q_start:q_end]) for row in ids)
    return bool(local), bool(cross)


def live_rows(cu_q, cu_k):
    """Query rows of the segments that have at least one key (numpy int array)."""
    cu_q, cu_k = np.asarray(cu_q), np.asarray(cu_k)
    rows = [np.arange(cu_q[s], cu_q[s + 1]) for s in range(len(cu_q) - 1) if cu_k[s + 1] > cu_k[s]]
    return np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)


def lse_merge_live_rows(o_acc, l_acc, o_new, l_new, cu_q, cu_k):
    """Running result (o_acc [T,H,D], l_acc [H,T]) merged with one chunk's
    (o_new, l_new) on the query rows of the chunk's segments with keys; the
    other rows keep the running values. Returns new fp64 arrays.
    [cp_attention page, the in-place live-row merge]"""
    o = _f64(o_acc).copy()
    l = _f64(l_acc).copy()
    rows = live_rows(cu_q, cu_k)
    if rows.size:
        om, lm = lse_merge(o[rows], l[:, rows], _f64(o_new)[rows], _f64(l_new)[:, rows])
        o[rows] = om
        l[:, rows] = lm
    return o, l


def grad_add_live_rows(dst, src, cu_q, cu_k):
    """dst + src on the query rows of the segments with keys, dst elsewhere
    (fp64). [cp_attention page, the in-place grad scatter-add]"""
    out = _f64(dst).copy()
    rows = live_rows(cu_q, cu_k)
    out[rows] += _f64(src)[rows]
    return out


def lse_merge(o1, l1, o2, l2):
    """Merge two partial results o [T,H,D], l [H,T] -> (o, l)."""
    lib = _load()
    o1, l1, o2, l2 = (_f64(x) for x in (o1, l1, o2, l2))
    T, H, D = o1.shape
    o = np.zeros_like(o1)
    l = np.zeros_like(l1)
    lib.oracle_lse_merge(_ptr(o1), _ptr(l1), _ptr(o2), _ptr(l2), _ptr(o), _ptr(l), T, H, D)
    return o, l
