"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare with the stated tolerances.

Tolerances (fp32 lse, bf16 outputs and gradients):
  out   max |err| <= 2e-2 (absolute, against the fp64 oracle)
  lse   max |err| <= 1e-3 (absolute); -inf rows must agree exactly
  dQ/dK/dV  relative Frobenius error <= 3e-2 against the fp64 oracle
  segment builder: bit-exact
"""
import numpy as np
import torch

import oracle
import packed_sequence_flash_gb300 as psf

OUT_TOL = 2e-2
LSE_TOL = 1e-3
GRAD_TOL = 3e-2


def cuda(t):
    return t.to("cuda")


def np64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_fwd(out, lse, out_ref, lse_ref, rows=None, lse_rows_axis=-1):
    o, l = np64(out), np64(lse)
    if rows is not None:
        o, out_ref = o[rows], out_ref[rows]
        l = np.take(l, rows, axis=lse_rows_axis)
        lse_ref = np.take(lse_ref, rows, axis=lse_rows_axis)
    assert not np.isnan(o).any() and not np.isnan(l).any()
    err = np.max(np.abs(o - out_ref)) if o.size else 0.0
    assert err <= OUT_TOL, f"out max|err| {err:.3e}"
    assert np.array_equal(np.isneginf(l), np.isneginf(lse_ref)), "-inf lse rows differ"
    fin = np.isfinite(lse_ref)
    if fin.any():
        lerr = np.max(np.abs(l[fin] - lse_ref[fin]))
        assert lerr <= LSE_TOL, f"lse max|err| {lerr:.3e}"
    return err


def rel_fro(a, ref):
    den = np.linalg.norm(ref)
    num = np.linalg.norm(a - ref)
    if den == 0:
        return num
    return num / den


def assert_grads(got, ref, names=("dq", "dk", "dv"), rows=None):
    errs = {}
    for g, r, n in zip(got, ref, names):
        a = np64(g)
        if rows is not None and n in rows:
            a, r = a[rows[n]], r[rows[n]]
        assert not np.isnan(a).any(), n
        e = rel_fro(a, r)
        errs[n] = e
        assert e <= GRAD_TOL, f"{n} relative Frobenius error {e:.3e}"
    return errs


def doc_case(w, window=None, check_bwd=True, skip_pad=True):
    """Run a packed single-row document workload through both paths."""
    q, k, v, do = (cuda(t) for t in (w.q, w.k, w.v, w.dout))
    ids = torch.from_numpy(w.doc_ids).to("cuda")
    Lq = w.q.shape[0]
    qids = ids[:, w.q_global_start:w.q_global_start + Lq].contiguous()
    out, lse, seg = psf.document_causal_attention(q, k, v, qids, ids, w.q_global_start, w.scale, window,
                                                  skip_pad=skip_pad)
    out_o, lse_o = oracle.attn_fwd_document(w.q, w.k, w.v, w.doc_ids, w.q_global_start, w.scale, window)
    assert_fwd(out, lse, out_o, lse_o)
    res = {}
    if check_bwd:
        grads = psf.document_causal_attention_backward(do, q, k, v, out, lse, seg, w.scale, window)
        ref = oracle.attn_bwd_document(w.dout, w.q, w.k, w.v, out_o, lse_o, w.doc_ids, w.q_global_start,
                                       w.scale, window)
        res = assert_grads(grads, ref)
    assert psf.device_status() == 0
    return res
