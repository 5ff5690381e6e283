"""Full-size parity: the five workloads at their stated sizes (and the
short-document workload with packed query heads), run through the same calls
the benchmark times, checked against the oracle on every row where the oracle
takes seconds (workloads 2 and 4; workload 1 is checked whole in the parity
tests) and on sampled rows elsewhere (the oracle evaluates forward rows and dQ
rows one query at a time and dK/dV rows one key at a time).

Workload 5 also runs the cross-chunk decomposition of the cp_attention page on
one GPU: the query shard 32768..65535 attends its own key chunk causally
(through the builder) and the earlier key chunk non-causally (through the
cross-chunk builder: the document that straddles the chunk edge, as one segment
between zero-query and zero-key segments); the cross result is merged into the
local one on its live rows, each chunk's backward is fed the merged out/lse, and
the cross chunk's dQ is added on its live rows. The result is compared with the
oracle's unsplit document-causal result for that shard.
"""
import numpy as np
import pytest
import torch

import oracle
import packed_sequence_flash_gb300 as psf
from packed_sequence_flash_gb300 import inputs
from gpu_helpers import GRAD_TOL, LSE_TOL, OUT_TOL, np64, rel_fro

pytestmark = pytest.mark.gpu


def _rows(n_total, n_sample, seed, must=()):
    r = np.random.default_rng(seed)
    rows = set(int(x) for x in r.choice(n_total, size=min(n_sample, n_total), replace=False))
    rows.update(int(m) for m in must if 0 <= m < n_total)
    return np.array(sorted(rows), dtype=np.int32)


def _check_fwd_rows(out, lse, out_o, lse_o, rows):
    o = np64(out)[rows]
    l = np64(lse)[:, rows]
    ro, rl = out_o[rows], lse_o[:, rows]
    assert not np.isnan(o).any() and not np.isnan(l).any()
    err = np.max(np.abs(o - ro))
    assert err <= OUT_TOL, f"out max|err| {err:.3e}"
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    if fin.any():
        assert np.max(np.abs(l[fin] - rl[fin])) <= LSE_TOL


def _check_grad_rows(g, ref, rows, name):
    a = np64(g)[rows]
    e = rel_fro(a, ref[rows])
    assert e <= GRAD_TOL, f"{name} relative Frobenius error {e:.3e} on sampled rows"


def _doc_full(cfg, n_rows=192, softcap=None, pack_gqa=False, seed=0, every_row=False):
    """Workload `cfg` through the document path against the oracle: on sampled
    rows, or on every query and key row (every_row) where the oracle is cheap."""
    w = inputs.config(cfg, seed=seed)
    dev = "cuda"
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    ids = torch.from_numpy(w.doc_ids).to(dev)
    Lq = w.q.shape[0]
    qids = ids[:, w.q_global_start:w.q_global_start + Lq].contiguous()
    out, lse, seg = psf.document_causal_attention(q, k, v, qids, ids, w.q_global_start, w.scale, w.window,
                                                  softcap=softcap, pack_gqa=pack_gqa)
    grads = psf.document_causal_attention_backward(do, q, k, v, out, lse, seg, w.scale, w.window, softcap=softcap,
                                                   pack_gqa=pack_gqa)
    assert psf.device_status() == 0
    # sample rows, always including document edges and the shard edges
    starts = np.cumsum([0] + w.extra["lengths"])
    if every_row:
        q_rows = np.arange(Lq, dtype=np.int32)
        k_rows = np.arange(w.k.shape[0], dtype=np.int32)
    else:
        q_rows = _rows(Lq, n_rows, 1, must=[0, Lq - 1] + [s - w.q_global_start for s in starts])
        k_rows = _rows(w.k.shape[0], n_rows, 2,
                       must=[0, w.k.shape[0] - 1] + list(starts[:-1]) + list(starts[1:] - 1))
    out_o, lse_o = oracle.attn_fwd_document(w.q, w.k, w.v, w.doc_ids, w.q_global_start, w.scale, w.window,
                                            rows=q_rows, softcap=softcap)
    _check_fwd_rows(out, lse, out_o, lse_o, q_rows)
    # the oracle backward needs the oracle's out/lse on every query row a sampled key sees
    out_all, lse_all = oracle.attn_fwd_document(w.q, w.k, w.v, w.doc_ids, w.q_global_start, w.scale, w.window,
                                                softcap=softcap)
    dq_o, dk_o, dv_o = oracle.attn_bwd_document(w.dout, w.q, w.k, w.v, out_all, lse_all, w.doc_ids,
                                                w.q_global_start, w.scale, w.window, q_rows=q_rows, k_rows=k_rows,
                                                softcap=softcap)
    _check_grad_rows(grads[0], dq_o, q_rows, "dq")
    _check_grad_rows(grads[1], dk_o, k_rows, "dk")
    _check_grad_rows(grads[2], dv_o, k_rows, "dv")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_workload2_full_size_every_row(seed):
    _doc_full(2, seed=seed, every_row=True)


def test_workload2_full_size_every_row_packed_heads():
    # the document path's default: a KV head's query heads share a tile
    _doc_full(2, every_row=True, pack_gqa=True)


def test_workload4_full_size_shard_unequal_dims_every_row():
    _doc_full(4, every_row=True)


def test_workload2_full_size_softcap():
    _doc_full(2, softcap=30.0)


def test_short_documents_full_size_pack_gqa():
    # 65536 tokens of 16-64 token documents, the query heads of each KV head
    # packed into one tile in the forward and one step in the backward
    _doc_full(6, n_rows=256, pack_gqa=True)


def test_workload3_dense_d512_full_size():
    w = inputs.config(3, seed=0)
    q, k, v, do = (t.to("cuda") for t in (w.q, w.k, w.v, w.dout))
    out, lse = psf.attn_dense_fwd(q, k, v, w.scale, True)
    grads = psf.attn_dense_bwd(do, q, k, v, out, lse, w.scale, True)
    assert psf.device_status() == 0
    B, Hq, N, D = w.q.shape
    q_rows = _rows(N, 24, 3, must=[0, 1, 127, 128, N - 1])
    k_rows = np.arange(N - 24, N, dtype=np.int32)  # keys seen by few queries (causal)
    need = np.union1d(q_rows, np.arange(N - 24, N)).astype(np.int32)
    cu = np.array([0, N], np.int32)
    for b in range(B):
        qp, kp, vp, dp = (x[b].permute(1, 0, 2).contiguous() for x in (w.q, w.k, w.v, w.dout))
        out_o, lse_o = oracle.attn_fwd_segments(qp, kp, vp, cu, cu, w.scale, True, rows=need)
        _check_fwd_rows(out[b].permute(1, 0, 2), lse[b], out_o, lse_o, q_rows)
        dq_o, dk_o, dv_o = oracle.attn_bwd_segments(dp, qp, kp, vp, out_o, lse_o, cu, cu, w.scale, True,
                                                    q_rows=q_rows, k_rows=k_rows)
        _check_grad_rows(grads[0][b].permute(1, 0, 2), dq_o, q_rows, "dq")
        _check_grad_rows(grads[1][b].permute(1, 0, 2), dk_o, k_rows, "dk")
        _check_grad_rows(grads[2][b].permute(1, 0, 2), dv_o, k_rows, "dv")


def _cheap_key_rows(lengths, offset=0, per_doc=2):
    """Keys whose visible query sets are short (the last tokens of every
    document, all tokens of the shortest one), so the oracle's per-key dK/dV
    needs few full query rows."""
    starts = np.cumsum([0] + list(lengths))
    rows = []
    for a, n in zip(starts[:-1], lengths):
        rows.extend(range(a + n - per_doc, a + n))
    i = int(np.argmin(lengths))
    rows.extend(range(starts[i], starts[i] + min(lengths[i], 64)))
    return np.array(sorted(set(int(r) + offset for r in rows)), dtype=np.int32)


def _queries_seeing(ids_row, keys, q0, Lq, window):
    """Query rows (shard-relative) that see any of `keys` (document-causal)."""
    need = set()
    for j in keys:
        doc = ids_row[j]
        if doc == 0:
            continue
        p = j
        while p < q0 + Lq and ids_row[p] == doc and (not window or p - j < window):
            if p >= q0:
                need.add(p - q0)
            p += 1
    return np.array(sorted(need), dtype=np.int32)


def test_workload5_full_size_window():
    w = inputs.config(5, seed=0)
    dev = "cuda"
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    ids = torch.from_numpy(w.doc_ids).to(dev)
    out, lse, seg = psf.document_causal_attention(q, k, v, ids, ids, 0, w.scale, w.window)
    grads = psf.document_causal_attention_backward(do, q, k, v, out, lse, seg, w.scale, w.window)
    assert psf.device_status() == 0
    S = w.k.shape[0]
    starts = np.cumsum([0] + w.extra["lengths"])
    q_rows = _rows(S, 64, 7, must=[0, S - 1] + list(starts[:-1]) + [s + w.window for s in starts[:-1]])
    k_rows = _cheap_key_rows(w.extra["lengths"])
    need = np.union1d(q_rows, _queries_seeing(w.doc_ids[0], k_rows, 0, S, w.window)).astype(np.int32)
    out_n, lse_n = oracle.attn_fwd_document(w.q, w.k, w.v, w.doc_ids, 0, w.scale, w.window, rows=need)
    _check_fwd_rows(out, lse, out_n, lse_n, q_rows)
    dq_o, dk_o, dv_o = oracle.attn_bwd_document(w.dout, w.q, w.k, w.v, out_n, lse_n, w.doc_ids, 0, w.scale,
                                                w.window, q_rows=q_rows, k_rows=k_rows)
    _check_grad_rows(grads[0], dq_o, q_rows, "dq")
    _check_grad_rows(grads[1], dk_o, k_rows, "dk")
    _check_grad_rows(grads[2], dv_o, k_rows, "dv")


def test_workload5_cross_chunk_merge():
    w = inputs.config(5, seed=0)
    dev = "cuda"
    S = w.k.shape[0]
    split = S // 2
    Lq = S - split
    ids_row = w.doc_ids[0]
    q_sh, do_sh = w.q[split:], w.dout[split:]
    q, k, v, do = (t.to(dev) for t in (q_sh, w.k, w.v, do_sh))
    # local chunk: keys split..S, causal, through the builder
    ids_local = torch.from_numpy(np.ascontiguousarray(w.doc_ids[:, split:])).to(dev)
    out1, lse1, seg1 = psf.document_causal_attention(q, k[split:], v[split:], ids_local, ids_local, 0, w.scale)
    # cross chunk: keys 0..split, non-causal, through the cross-chunk builder
    ids = torch.from_numpy(w.doc_ids).to(dev)
    cq2, ck2, meta2 = psf.build_cross_segments(ids, split, Lq, 0, split)
    cu_q2, cu_k2, mq2, mk2 = oracle.build_cross_segments(w.doc_ids, split, Lq, 0, split)
    np.testing.assert_array_equal(cq2.cpu().numpy(), cu_q2)
    np.testing.assert_array_equal(ck2.cpu().numpy(), cu_k2)
    out2, lse2 = psf.attn_varlen_fwd(q, k[:split], v[:split], cq2, ck2, -1, -1, w.scale, False, dev_meta=meta2)
    # the local result is the running one; merge the cross chunk in on its live rows
    out_m, lse_m = out1.clone(), lse1.clone()
    psf.lse_merge_live_rows(out_m, lse_m, out2, lse2, cq2, ck2, dev_meta=meta2)
    # each chunk's backward is fed the merged out/lse
    dq1, dk1, dv1 = psf.document_causal_attention_backward(do, q, k[split:], v[split:], out_m, lse_m, seg1,
                                                           w.scale)
    dq2, dk2, dv2 = psf.attn_varlen_bwd(do, q, k[:split], v[:split], out_m, lse_m, cq2, ck2, -1, -1, w.scale,
                                        False, dev_meta=meta2)
    dq = dq1.clone()
    psf.grad_add_live_rows(dq, dq2, cq2, ck2, dev_meta=meta2)
    assert psf.device_status() == 0
    dk = torch.cat([dk2, dk1])
    dv = torch.cat([dv2, dv1])
    # against the oracle's unsplit result for the shard, on sampled query rows
    # and on keys with short query sets
    strad = int(cu_q2[2])
    q_rows = _rows(Lq, 64, 5, must=[0, Lq - 1, strad - 1, strad])
    out_o, lse_o = oracle.attn_fwd_document(q_sh, w.k, w.v, w.doc_ids, split, w.scale, None, rows=q_rows)
    _check_fwd_rows(out_m, lse_m, out_o, lse_o, q_rows)
    ends = np.cumsum(w.extra["lengths"])
    k_rows = np.array(sorted({int(e) - d for e in ends if e > split + strad for d in (1, 2)}), dtype=np.int32)
    need = np.union1d(q_rows, _queries_seeing(ids_row, k_rows, split, Lq, None)).astype(np.int32)
    out_n, lse_n = oracle.attn_fwd_document(q_sh, w.k, w.v, w.doc_ids, split, w.scale, None, rows=need)
    dq_o, dk_o, dv_o = oracle.attn_bwd_document(do_sh, q_sh, w.k, w.v, out_n, lse_n, w.doc_ids, split, w.scale,
                                                None, q_rows=q_rows, k_rows=k_rows)
    _check_grad_rows(dq, dq_o, q_rows, "dq")
    _check_grad_rows(dk, dk_o, k_rows, "dk")
    _check_grad_rows(dv, dv_o, k_rows, "dv")
    # the decomposition as a whole against the unsplit path on every row
    qids = ids[:, split:].contiguous()
    out_u, lse_u, seg_u = psf.document_causal_attention(q, k, v, qids, ids, split, w.scale)
    gu = psf.document_causal_attention_backward(do, q, k, v, out_u, lse_u, seg_u, w.scale)
    assert float((out_m.float() - out_u.float()).abs().max()) <= OUT_TOL
    for a, b, n in ((dq, gu[0], "dq"), (dk, gu[1], "dk"), (dv, gu[2], "dv")):
        e = float(torch.linalg.norm(a.float() - b.float()) / torch.linalg.norm(b.float()))
        assert e <= GRAD_TOL, f"{n}: chunked vs unsplit relative Frobenius {e:.3e}"


def test_workload5_full_shard_lse_merge_and_pad_fixup():
    # The plain two-result merge over the whole query shard of workload 5 (the
    # local chunk's and the cross chunk's results, every row), against the
    # oracle's merge of the same inputs on sampled rows and against the
    # live-row merge on every row; then the literal pad fixup over the local
    # result, which must leave it unchanged (padding rows are already zero).
    w = inputs.config(5, seed=0)
    dev = "cuda"
    S = w.k.shape[0]
    split = S // 2
    Lq = S - split
    q, k, v = (t.to(dev) for t in (w.q[split:], w.k, w.v))
    ids_local = torch.from_numpy(np.ascontiguousarray(w.doc_ids[:, split:])).to(dev)
    out1, lse1, _ = psf.document_causal_attention(q, k[split:], v[split:], ids_local, ids_local, 0, w.scale)
    ids = torch.from_numpy(w.doc_ids).to(dev)
    cq2, ck2, meta2 = psf.build_cross_segments(ids, split, Lq, 0, split)
    out2, lse2 = psf.attn_varlen_fwd(q, k[:split], v[:split], cq2, ck2, -1, -1, w.scale, False, dev_meta=meta2)
    of, ob, lm = psf.lse_merge(out1, lse1, out2, lse2, want_f32=True, want_bf16=True)
    out_m, lse_m = out1.clone(), lse1.clone()
    psf.lse_merge_live_rows(out_m, lse_m, out2, lse2, cq2, ck2, dev_meta=meta2)
    assert psf.device_status() == 0
    rows = _rows(Lq, 256, 11, must=[0, Lq - 1, int(cq2[2].item()) - 1, int(cq2[2].item())])
    o_ref, l_ref = oracle.lse_merge(np64(out1)[rows], np64(lse1)[:, rows], np64(out2)[rows], np64(lse2)[:, rows])
    assert np.max(np.abs(np64(of)[rows] - o_ref)) <= 1e-5
    assert np.array_equal(np.isneginf(np64(lm)[:, rows]), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.max(np.abs(np64(lm)[:, rows][fin] - l_ref[fin])) <= 1e-5
    assert float((ob.float() - of).abs().max()) <= 2.0 ** -7 * max(1.0, float(of.abs().max()))
    assert float((out_m.float() - ob.float()).abs().max()) <= 2.0 ** -7 * max(1.0, float(of.abs().max()))
    assert torch.equal(torch.isneginf(lse_m), torch.isneginf(lm))
    fin_t = torch.isfinite(lm)
    assert float((lse_m[fin_t] - lm[fin_t]).abs().max()) <= 1e-5
    before_o, before_l = out1.clone(), lse1.clone()
    psf.pad_fixup(out1, lse1, ids_local[0].contiguous())
    assert psf.device_status() == 0
    assert torch.equal(out1, before_o) and torch.equal(lse1, before_l)
