"""Pins for the fp64 oracle: each check ties it to something other than itself.

Sources of truth used here (never the oracle's own formula retyped):
  * library routines on special cases: torch's fp64 ``scaled_dot_product_attention``
    with boolean masks built by ``torch.tril``/``torch.triu``, ``torch.logsumexp``,
    and torch autograd;
  * closed forms (window of one token, zero keys, constant values, window wider
    than the segment);
  * central finite differences of the oracle's own forward for the gradients;
  * invariants (GQA = repeated-KV MHA, chunked results merged by lse = full result,
    document mode = segment mode over the builder's segments, zero-query segments
    contribute nothing, pad rows zero);
  * hand-derived segment lists and brute-force pair visibility for the builders
    (doc ids -> segments, and the cross-chunk builder of a query shard against an
    earlier key chunk), and the cross-chunk decomposition (live-row merge, live-row
    gradient add) against document mode on the unsplit problem.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def rnd(*shape, s=1.0):
    return rng.standard_normal(shape) * s


def sdpa64(q, k, v, mask, scale):
    """torch fp64 SDPA on [Tq,H,D] single-segment inputs with a [Tq,Tk] bool mask."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    Hq, Hkv = qt.shape[1], kt.shape[1]
    kt = kt.repeat_interleave(Hq // Hkv, dim=1)
    vt = vt.repeat_interleave(Hq // Hkv, dim=1)
    m = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def torch_lse(q, k, mask, scale):
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(q.shape[1] // k.shape[1], dim=0)
    z = scale * qt @ kt.transpose(1, 2)
    if mask is not None:
        z = z.masked_fill(~torch.from_numpy(mask), -math.inf)
    return torch.logsumexp(z, dim=-1).numpy()  # [H, Tq]


def band_mask(m, n, causal, window):
    """Bottom-right aligned causal band from torch.tril/triu diagonals."""
    full = torch.ones(m, n, dtype=torch.bool)
    mask = full.clone()
    delta = n - m
    if causal:
        mask &= torch.tril(full, diagonal=delta)
    if window:
        mask &= torch.triu(full, diagonal=delta - window + 1)
    return mask.numpy()


def one_seg(m, n):
    return np.array([0, m], np.int32), np.array([0, n], np.int32)


# ---------------------------------------------------------------------------
# forward pins

@pytest.mark.parametrize("causal,window,m,n", [
    (False, None, 9, 13), (True, None, 9, 13), (True, None, 13, 13), (True, 4, 9, 13),
    (False, 3, 11, 11), (True, 1, 6, 6), (True, None, 5, 20),
])
def test_fwd_matches_torch_sdpa_single_segment(causal, window, m, n):
    q, k, v = rnd(m, 4, 16), rnd(n, 2, 16), rnd(n, 2, 8)
    cu_q, cu_k = one_seg(m, n)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.3, causal, window)
    mask = band_mask(m, n, causal, window)
    ref = sdpa64(q, k, v, mask, 0.3)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch_lse(q, k, mask, 0.3), rtol=1e-12, atol=1e-12)


def test_fwd_rows_without_keys_are_zero_and_neg_inf():
    # more queries than keys: bottom-right alignment leaves the first m - n rows empty
    m, n = 10, 4
    q, k, v = rnd(m, 2, 8), rnd(n, 1, 8), rnd(n, 1, 8)
    cu_q, cu_k = one_seg(m, n)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.5, True)
    assert np.all(out[: m - n] == 0) and np.all(np.isneginf(lse[:, : m - n]))
    mask = band_mask(m, n, True, None)
    np.testing.assert_allclose(out[m - n:], sdpa64(q, k, v, mask, 0.5)[m - n:], rtol=1e-12, atol=1e-12)
    # uncovered rows past the last segment and zero-key segments behave the same
    out2, lse2 = oracle.attn_fwd_segments(rnd(6, 2, 8), k, v, np.array([0, 2, 4], np.int32),
                                          np.array([0, 0, 4], np.int32), 0.5, False)
    assert np.all(out2[:2] == 0) and np.all(np.isneginf(lse2[:, :2]))
    assert np.all(out2[4:] == 0) and np.all(np.isneginf(lse2[:, 4:]))


def test_fwd_closed_form_window_one():
    # W = 1: each query sees only the key on its bottom-right diagonal
    m, n = 7, 11
    q, k, v = rnd(m, 2, 8), rnd(n, 2, 8), rnd(n, 2, 4)
    cu_q, cu_k = one_seg(m, n)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.7, True, 1)
    for i in range(m):
        j = i + n - m
        np.testing.assert_allclose(out[i], v[j], rtol=1e-13)
        for h in range(2):
            assert lse[h, i] == pytest.approx(0.7 * float(q[i, h] @ k[j, h]), rel=1e-13)


def test_fwd_closed_form_zero_keys_gives_mean_and_log_count():
    m, n, W = 6, 9, 4
    q, k, v = rnd(m, 1, 8), np.zeros((n, 1, 8)), rnd(n, 1, 5)
    cu_q, cu_k = one_seg(m, n)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 1.0, True, W)
    d = n - m
    for i in range(m):
        lo, hi = max(0, i + d - W + 1), i + d
        np.testing.assert_allclose(out[i, 0], v[lo:hi + 1, 0].mean(axis=0), rtol=1e-12)
        assert lse[0, i] == pytest.approx(math.log(hi - lo + 1), rel=1e-13)


def test_fwd_closed_form_constant_values():
    q, k = rnd(12, 2, 8), rnd(12, 1, 8)
    u = rnd(6)
    v = np.broadcast_to(u, (12, 1, 6)).copy()
    out, _ = oracle.attn_fwd_segments(q, k, v, *one_seg(12, 12), 0.4, True, 5)
    np.testing.assert_allclose(out, np.broadcast_to(u, out.shape), rtol=1e-12)


def test_fwd_window_wider_than_segment_equals_no_window():
    q, k, v = rnd(9, 2, 8), rnd(14, 2, 8), rnd(14, 2, 8)
    a = oracle.attn_fwd_segments(q, k, v, *one_seg(9, 14), 0.3, True, 14)
    b = oracle.attn_fwd_segments(q, k, v, *one_seg(9, 14), 0.3, True, None)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_fwd_gqa_equals_repeated_kv():
    q, k, v = rnd(10, 6, 8), rnd(10, 2, 8), rnd(10, 2, 8)
    cu = np.array([0, 4, 10], np.int32)
    a_out, a_lse = oracle.attn_fwd_segments(q, k, v, cu, cu, 0.3, True, 3)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    b_out, b_lse = oracle.attn_fwd_segments(q, kr, vr, cu, cu, 0.3, True, 3)
    np.testing.assert_array_equal(a_out, b_out)
    np.testing.assert_array_equal(a_lse, b_lse)


def test_fwd_merge_of_two_key_chunks_equals_full():
    # non-causal segment; keys split in two chunks; merge by lse reproduces the whole
    m, n, n1 = 8, 15, 6
    q, k, v = rnd(m, 2, 8), rnd(n, 1, 8), rnd(n, 1, 8)
    full = oracle.attn_fwd_segments(q, k, v, *one_seg(m, n), 0.5, False)
    c1 = oracle.attn_fwd_segments(q, k[:n1], v[:n1], *one_seg(m, n1), 0.5, False)
    c2 = oracle.attn_fwd_segments(q, k[n1:], v[n1:], *one_seg(m, n - n1), 0.5, False)
    o, l = oracle.lse_merge(c1[0], c1[1], c2[0], c2[1])
    np.testing.assert_allclose(o, full[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l, full[1], rtol=1e-13)


def test_merge_neg_inf_rows():
    o1, o2 = rnd(3, 1, 4), rnd(3, 1, 4)
    l1 = np.array([[-np.inf, 0.5, -np.inf]])
    l2 = np.array([[-np.inf, -np.inf, 1.5]])
    o, l = oracle.lse_merge(o1 * 0, l1, o2 * 0, l2)
    assert np.all(o[0] == 0) and np.isneginf(l[0, 0])
    o, l = oracle.lse_merge(o1, l1, o2, l2)
    np.testing.assert_allclose(o[1], o1[1])
    np.testing.assert_allclose(o[2], o2[2])
    assert l[0, 1] == 0.5 and l[0, 2] == 1.5
    assert not np.isnan(o).any()


def test_dense_batches_are_independent():
    q, k, v = rnd(2, 4, 16, 8), rnd(2, 2, 16, 8), rnd(2, 2, 16, 8)
    out, lse = oracle.attn_fwd_dense(q, k, v, 0.3, True)
    for b in range(2):
        ob, lb = oracle.attn_fwd_dense(q[b:b + 1], k[b:b + 1], v[b:b + 1], 0.3, True)
        np.testing.assert_array_equal(out[b], ob[0])
        np.testing.assert_array_equal(lse[b], lb[0])
    # and a single batch equals torch SDPA with a causal mask
    qp = q[0].transpose(1, 0, 2)
    ref = sdpa64(qp, k[0].transpose(1, 0, 2), v[0].transpose(1, 0, 2), band_mask(16, 16, True, None), 0.3)
    np.testing.assert_allclose(out[0].transpose(1, 0, 2), ref, rtol=1e-12, atol=1e-13)


def _random_doc_ids(B, S, seed, pad_prob=0.3):
    r = np.random.default_rng(seed)
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        pos, d = 0, 1
        while pos < S:
            n = int(r.integers(1, 6))
            ids[b, pos:pos + n] = 0 if r.random() < pad_prob else d
            d += 1
            pos += n
    return ids


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("window", [None, 3])
def test_document_mode_equals_segments_over_builder(seed, window):
    B, S = 2, 24
    ids = _random_doc_ids(B, S, seed)
    q0, Lq = [(0, 24), (8, 16), (5, 7)][seed % 3]
    q, k, v = rnd(B * Lq, 4, 8), rnd(B * S, 2, 8), rnd(B * S, 2, 8)
    doc = oracle.attn_fwd_document(q, k, v, ids, q0, 0.4, window)
    cu_q, cu_k, mq, mk = oracle.build_segments(ids, Lq, q0)
    seg = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.4, True, window)
    qid = ids[:, q0:q0 + Lq].reshape(-1)
    pad = qid == 0
    assert np.all(doc[0][pad] == 0) and np.all(np.isneginf(doc[1][:, pad]))
    np.testing.assert_allclose(doc[0][~pad], seg[0][~pad], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(doc[1][:, ~pad], seg[1][:, ~pad], rtol=1e-13)


def test_zero_query_segments_contribute_nothing():
    q, k, v = rnd(6, 2, 8), rnd(14, 2, 8), rnd(14, 2, 8)
    a = oracle.attn_fwd_segments(q, k[:10], v[:10], np.array([0, 4, 6], np.int32),
                                 np.array([0, 5, 10], np.int32), 0.3, True)
    # insert zero-query segments (extra keys) before, between and after
    k2 = np.concatenate([k[10:12], k[:5], k[12:13], k[5:10], k[13:14]])
    v2 = np.concatenate([v[10:12], v[:5], v[12:13], v[5:10], v[13:14]])
    b = oracle.attn_fwd_segments(q, k2, v2, np.array([0, 0, 4, 4, 6, 6], np.int32),
                                 np.array([0, 2, 7, 8, 13, 14], np.int32), 0.3, True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------------------
# backward pins

def _loss_and_grads(mode_kwargs, q, k, v, g, scale, causal, window):
    if "doc_ids" in mode_kwargs:
        f = lambda q_, k_, v_: oracle.attn_fwd_document(q_, k_, v_, mode_kwargs["doc_ids"],
                                                        mode_kwargs["q0"], scale, window)
        out, lse = f(q, k, v)
        grads = oracle.attn_bwd_document(g, q, k, v, out, lse, mode_kwargs["doc_ids"],
                                         mode_kwargs["q0"], scale, window)
    else:
        cu_q, cu_k = mode_kwargs["cu_q"], mode_kwargs["cu_k"]
        f = lambda q_, k_, v_: oracle.attn_fwd_segments(q_, k_, v_, cu_q, cu_k, scale, causal, window)
        out, lse = f(q, k, v)
        grads = oracle.attn_bwd_segments(g, q, k, v, out, lse, cu_q, cu_k, scale, causal, window)
    return f, grads


def _fd_check(f, grads, q, k, v, g, h=1e-6):
    loss = lambda q_, k_, v_: float(np.sum(f(q_, k_, v_)[0] * g))
    for t_idx, (x, gx) in enumerate(zip((q, k, v), grads)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            args = [q, k, v]
            xp = x.copy(); xp[i] += h
            xm = x.copy(); xm[i] -= h
            args[t_idx] = xp; lp = loss(*args)
            args[t_idx] = xm; lm = loss(*args)
            num[i] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - gx) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-6, (t_idx, err)


@pytest.mark.parametrize("causal,window", [(True, None), (True, 3), (False, None), (False, 2)])
def test_bwd_matches_central_finite_differences_segments(causal, window):
    cu_q = np.array([0, 3, 3, 7], np.int32)   # includes a zero-query segment
    cu_k = np.array([0, 4, 6, 11], np.int32)
    q, k, v, g = rnd(7, 2, 3), rnd(11, 1, 3), rnd(11, 1, 2), rnd(7, 2, 2)
    f, grads = _loss_and_grads(dict(cu_q=cu_q, cu_k=cu_k), q, k, v, g, 0.6, causal, window)
    _fd_check(f, grads, q, k, v, g)


def test_bwd_matches_central_finite_differences_document():
    ids = np.array([[1, 1, 1, 0, 2, 2, 2, 2, 3, 0, 0]], np.int32)
    q0, Lq = 2, 7
    q, k, v, g = rnd(Lq, 2, 3), rnd(11, 2, 3), rnd(11, 2, 2), rnd(Lq, 2, 2)
    f, grads = _loss_and_grads(dict(doc_ids=ids, q0=q0), q, k, v, g, 0.8, True, 3)
    _fd_check(f, grads, q, k, v, g)


def test_bwd_matches_torch_autograd_sdpa():
    m, n = 9, 12
    q, k, v, g = rnd(m, 4, 8), rnd(n, 2, 8), rnd(n, 2, 6), rnd(m, 4, 6)
    cu_q, cu_k = one_seg(m, n)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.3, True, 5)
    dq, dk, dv = oracle.attn_bwd_segments(g, q, k, v, out, lse, cu_q, cu_k, 0.3, True, 5)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None].requires_grad_()
    kt = torch.from_numpy(k).permute(1, 0, 2)[None].requires_grad_()
    vt = torch.from_numpy(v).permute(1, 0, 2)[None].requires_grad_()
    mask = torch.from_numpy(band_mask(m, n, True, 5))
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(2, 1), vt.repeat_interleave(2, 1), attn_mask=mask, scale=0.3)
    o.backward(torch.from_numpy(g).permute(1, 0, 2)[None])
    np.testing.assert_allclose(dq, qt.grad[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_bwd_gqa_sums_repeated_kv_grads():
    cu = np.array([0, 5, 12], np.int32)
    q, k, v, g = rnd(12, 6, 8), rnd(12, 2, 8), rnd(12, 2, 4), rnd(12, 6, 4)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu, cu, 0.3, True)
    dq, dk, dv = oracle.attn_bwd_segments(g, q, k, v, out, lse, cu, cu, 0.3, True)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    dq2, dk2, dv2 = oracle.attn_bwd_segments(g, q, kr, vr, out, lse, cu, cu, 0.3, True)
    np.testing.assert_allclose(dq, dq2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dk, dk2.reshape(12, 2, 3, 8).sum(2), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dv, dv2.reshape(12, 2, 3, 4).sum(2), rtol=1e-12, atol=1e-14)


def test_bwd_chunked_with_merged_out_lse_sums_to_full():
    # the ring decomposition: each key chunk's backward fed the merged out/lse
    m, n, n1 = 8, 14, 5
    q, k, v, g = rnd(m, 2, 8), rnd(n, 1, 8), rnd(n, 1, 8), rnd(m, 2, 8)
    cu_q, cu_k = one_seg(m, n)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.5, False)
    full = oracle.attn_bwd_segments(g, q, k, v, out, lse, cu_q, cu_k, 0.5, False)
    a = oracle.attn_bwd_segments(g, q, k[:n1], v[:n1], out, lse, *one_seg(m, n1), 0.5, False)
    b = oracle.attn_bwd_segments(g, q, k[n1:], v[n1:], out, lse, *one_seg(m, n - n1), 0.5, False)
    np.testing.assert_allclose(a[0] + b[0], full[0], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(np.concatenate([a[1], b[1]]), full[1], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(np.concatenate([a[2], b[2]]), full[2], rtol=1e-11, atol=1e-13)


def test_bwd_row_samples_match_full():
    cu = np.array([0, 7, 19], np.int32)
    q, k, v, g = rnd(19, 4, 8), rnd(19, 2, 8), rnd(19, 2, 8), rnd(19, 4, 8)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu, cu, 0.3, True, 6)
    full = oracle.attn_bwd_segments(g, q, k, v, out, lse, cu, cu, 0.3, True, 6)
    rows = np.array([0, 6, 7, 18], np.int32)
    part = oracle.attn_bwd_segments(g, q, k, v, out, lse, cu, cu, 0.3, True, 6, q_rows=rows,
                                    k_rows=rows)
    for t, u in zip(part, full):
        np.testing.assert_array_equal(t[rows], u[rows])
    o2, l2 = oracle.attn_fwd_segments(q, k, v, cu, cu, 0.3, True, 6, rows=rows)
    np.testing.assert_array_equal(o2[rows], out[rows])


def test_bwd_neg_inf_lse_rows_give_zero_grads():
    # pad rows are fed lse = -inf and contribute nothing
    cu = np.array([0, 6], np.int32)
    q, k, v, g = rnd(6, 1, 4), rnd(6, 1, 4), rnd(6, 1, 4), rnd(6, 1, 4)
    out, lse = oracle.attn_fwd_segments(q, k, v, cu, cu, 0.5, True)
    lse2 = lse.copy(); lse2[0, 3:] = -np.inf
    out2 = out.copy(); out2[3:] = 0
    dq, dk, dv = oracle.attn_bwd_segments(g, q, k, v, out2, lse2, cu, cu, 0.5, True)
    assert np.all(dq[3:] == 0)
    # keys 3..5 are seen only by rows 3..5, so they receive nothing
    assert np.all(dk[3:] == 0) and np.all(dv[3:] == 0)
    assert not np.isnan(dq).any()


# ---------------------------------------------------------------------------
# builder pins

def test_builder_golden_examples():
    with open(os.path.join(GOLDEN, "builder_examples.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        cu_q, cu_k, mq, mk = oracle.build_segments(c["doc_ids"], c["q_length"], c["q_global_start"])
        assert cu_q.tolist() == c["cu_q"], c
        assert cu_k.tolist() == c["cu_k"], c
        assert (mq, mk) == (c["max_q"], c["max_k"]), c


@pytest.mark.parametrize("seed", range(25))
def test_builder_brute_force_visibility_and_tiling(seed):
    r = np.random.default_rng(seed)
    B, S = int(r.integers(1, 4)), int(r.integers(1, 20))
    ids = _random_doc_ids(B, S, 100 + seed, pad_prob=0.25)
    q0 = int(r.integers(0, S))
    Lq = int(r.integers(0, S - q0 + 1))
    cu_q, cu_k, mq, mk = oracle.build_segments(ids, Lq, q0)
    nq, nk = np.diff(cu_q), np.diff(cu_k)
    # tiling of the flattened query and key tensors
    assert cu_q[0] == 0 and cu_k[0] == 0 and cu_q[-1] == B * Lq and cu_k[-1] == B * S
    assert np.all(nq >= 0) and np.all(nk >= 1)
    assert mq == (nq.max() if len(nq) else 0) and mk == (nk.max() if len(nk) else 0)
    # causal bottom-right visibility from (cu, delta) equals the doc-id predicate
    seg_vis = np.zeros((B * Lq, B * S), bool)
    for s in range(len(nq)):
        d = nk[s] - nq[s]
        for i in range(nq[s]):
            for j in range(nk[s]):
                if j <= i + d:
                    seg_vis[cu_q[s] + i, cu_k[s] + j] = True
    doc_vis = np.zeros_like(seg_vis)
    for b in range(B):
        for i in range(Lq):
            p = q0 + i
            for j in range(S):
                same_run = len(set(ids[b, min(j, p):max(j, p) + 1].tolist())) == 1
                if same_run and j <= p:
                    doc_vis[b * Lq + i, b * S + j] = True
    np.testing.assert_array_equal(seg_vis, doc_vis)


def test_builder_skip_pad_golden_examples():
    with open(os.path.join(GOLDEN, "builder_skip_pad_examples.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        cu_q, cu_k, mq, mk = oracle.build_segments(c["doc_ids"], c["q_length"], c["q_global_start"], skip_pad=True)
        assert cu_q.tolist() == c["cu_q"], c
        assert cu_k.tolist() == c["cu_k"], c
        assert (mq, mk) == (c["max_q"], c["max_k"]), c


@pytest.mark.parametrize("seed", range(25))
def test_builder_skip_pad_brute_force(seed):
    # padding queries sit in segments without keys, padding keys in segments
    # without queries, and every other pair is the doc-id predicate
    r = np.random.default_rng(seed)
    B, S = int(r.integers(1, 4)), int(r.integers(1, 20))
    ids = _random_doc_ids(B, S, 700 + seed, pad_prob=0.35)
    q0 = int(r.integers(0, S))
    Lq = int(r.integers(0, S - q0 + 1))
    cu_q, cu_k, mq, mk = oracle.build_segments(ids, Lq, q0, skip_pad=True)
    nq, nk = np.diff(cu_q), np.diff(cu_k)
    assert cu_q[0] == 0 and cu_k[0] == 0 and cu_q[-1] == B * Lq and cu_k[-1] == B * S
    assert np.all(nq >= 0) and np.all(nk >= 0)
    assert mq == (nq.max() if len(nq) else 0) and mk == (nk.max() if len(nk) else 0)
    qid = ids[:, q0:q0 + Lq].reshape(-1)
    kid = ids.reshape(-1)
    for s in range(len(nq)):
        if (qid[cu_q[s]:cu_q[s + 1]] == 0).any():
            assert nk[s] == 0 and (qid[cu_q[s]:cu_q[s + 1]] == 0).all()
        if (kid[cu_k[s]:cu_k[s + 1]] == 0).any():
            assert nq[s] == 0 and (kid[cu_k[s]:cu_k[s + 1]] == 0).all()
    seg_vis = np.zeros((B * Lq, B * S), bool)
    for s in range(len(nq)):
        d = nk[s] - nq[s]
        for i in range(nq[s]):
            for j in range(nk[s]):
                if j <= i + d:
                    seg_vis[cu_q[s] + i, cu_k[s] + j] = True
    doc_vis = np.zeros_like(seg_vis)
    for b in range(B):
        for i in range(Lq):
            p = q0 + i
            if ids[b, p] == 0:
                continue
            for j in range(p + 1):
                if np.all(ids[b, j:p + 1] == ids[b, p]):
                    doc_vis[b * Lq + i, b * S + j] = True
    np.testing.assert_array_equal(seg_vis, doc_vis)


@pytest.mark.parametrize("seed,window", [(0, None), (1, None), (2, 3), (3, 5)])
def test_skip_pad_segments_equal_document_mode(seed, window):
    # the skip-pad segments run through the plain segment oracle, with no pad
    # fixup afterwards, reproduce the document-mode result (forward and
    # backward) including the padding rows' zero output and -inf lse
    r = np.random.default_rng(seed)
    B, S, Hq, Hkv, D = 2, 24, 2, 1, 8
    ids = _random_doc_ids(B, S, 900 + seed, pad_prob=0.3)
    q0 = int(r.integers(0, 12))
    Lq = int(r.integers(1, S - q0 + 1))
    q, do = rnd(B * Lq, Hq, D), rnd(B * Lq, Hq, D)
    k, v = rnd(B * S, Hkv, D), rnd(B * S, Hkv, D)
    scale = 0.35
    cu_q, cu_k, _, _ = oracle.build_segments(ids, Lq, q0, skip_pad=True)
    o, l = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, True, window)
    ro, rl = oracle.attn_fwd_document(q, k, v, ids, q0, scale, window)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(l[fin], rl[fin], atol=1e-12)
    assert (ids[:, q0:q0 + Lq].reshape(-1) == 0).sum() == 0 or np.isneginf(rl).any()
    g = oracle.attn_bwd_segments(do, q, k, v, o, l, cu_q, cu_k, scale, True, window)
    rg = oracle.attn_bwd_document(do, q, k, v, ro, rl, ids, q0, scale, window)
    for a, b in zip(g, rg):
        np.testing.assert_allclose(a, b, atol=1e-10)


# ---------------------------------------------------------------------------
# dense-kernel eligibility of a ring chunk (routing)

def test_dense_route_golden_examples():
    with open(os.path.join(GOLDEN, "dense_route_examples.json")) as fh:
        g = json.load(fh)
    for r in g["rows"]:
        assert oracle.row_is_single_document(r["ids"]) == r["single"], r
        assert oracle.row_is_document_prefix(r["ids"]) == r["prefix"], r
    for c in g["chunks"]:
        got = oracle.chunk_dense_flags(c["doc_ids"], c["q_start"], c["q_length"], c["k_start"], c["k_length"])
        assert got == (c["local"], c["cross"]), c


def _bhsd(x, B, N):
    # packed [B*N, H, D] -> [B, H, N, D]
    return x.reshape(B, N, x.shape[1], x.shape[2]).transpose(0, 2, 1, 3)


def _packed(x):
    # [B, H, N, D] -> packed [B*N, H, D]
    B, H, N, D = x.shape
    return x.transpose(0, 2, 1, 3).reshape(B * N, H, D)


def _dense_route(q, k, v, do, qids, scale, causal, window=None):
    """Dense oracle on [B,H,N,D], padding query rows zeroed after, backward fed the fixed out/lse."""
    o, l = oracle.attn_fwd_dense(q, k, v, scale, causal, window)
    pad = np.asarray(qids) == 0  # [B, Lq]
    o = o.copy()
    l = l.copy()
    o[pad[:, None, :, None].repeat(o.shape[1], 1).repeat(o.shape[3], 3)] = 0.0
    l[pad[:, None, :].repeat(l.shape[1], 1)] = -np.inf
    g = oracle.attn_bwd_dense(do, q, k, v, o, l, scale, causal, window)
    return o, l, g


@pytest.mark.parametrize("seed,window", [(0, None), (1, None), (2, 4)])
def test_dense_local_route_equals_document_mode(seed, window):
    r = np.random.default_rng(seed)
    B, S, Hq, Hkv, D = 3, 20, 2, 1, 8
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        ids[b, :int(r.integers(0, S + 1))] = b + 1  # one document prefix, padding suffix
    q0 = int(r.integers(0, S))
    Lq = S - q0
    k0 = int(r.integers(0, q0 + 1))
    Lk = S - k0
    assert oracle.chunk_dense_flags(ids, q0, Lq, k0, Lk)[0]
    q, do = rnd(B, Hq, Lq, D), rnd(B, Hq, Lq, D)
    k, v = rnd(B, Hkv, Lk, D), rnd(B, Hkv, Lk, D)
    scale = 0.4
    o, l, g = _dense_route(q, k, v, do, ids[:, q0:], scale, True, window)
    ids_chunk = ids[:, k0:]
    ro, rl = oracle.attn_fwd_document(_packed(q), _packed(k), _packed(v), ids_chunk, q0 - k0, scale, window)
    np.testing.assert_allclose(_packed(o), ro, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(l.transpose(1, 0, 2).reshape(Hq, -1)), np.isneginf(rl))
    rg = oracle.attn_bwd_document(_packed(do), _packed(q), _packed(k), _packed(v), ro, rl, ids_chunk, q0 - k0,
                                  scale, window)
    for a, b in zip(g, rg):
        np.testing.assert_allclose(_packed(a), b, atol=1e-10)


@pytest.mark.parametrize("seed", range(3))
def test_dense_cross_route_equals_cross_segments(seed):
    r = np.random.default_rng(20 + seed)
    B, S, Hq, Hkv, D = 2, 24, 2, 1, 8
    q0 = int(r.integers(4, 16))
    Lq = S - q0
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        ids[b, :q0 + int(r.integers(1, Lq + 1))] = b + 3  # the document crosses into the shard, then padding
    k0 = int(r.integers(0, q0))
    Lk = int(r.integers(1, q0 - k0 + 1))
    assert oracle.chunk_dense_flags(ids, q0, Lq, k0, Lk)[1]
    q, do = rnd(B, Hq, Lq, D), rnd(B, Hq, Lq, D)
    k, v = rnd(B, Hkv, Lk, D), rnd(B, Hkv, Lk, D)
    scale = 0.4
    o, l, g = _dense_route(q, k, v, do, ids[:, q0:], scale, False)
    cu_q, cu_k, _, _ = oracle.build_cross_segments(ids, q0, Lq, k0, Lk)
    ro, rl = oracle.attn_fwd_segments(_packed(q), _packed(k), _packed(v), cu_q, cu_k, scale, False)
    np.testing.assert_allclose(_packed(o), ro, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(l.transpose(1, 0, 2).reshape(Hq, -1)), np.isneginf(rl))
    rg = oracle.attn_bwd_segments(_packed(do), _packed(q), _packed(k), _packed(v), ro, rl, cu_q, cu_k, scale, False)
    for a, b in zip(g, rg):
        np.testing.assert_allclose(_packed(a), b, atol=1e-10)


def test_dense_route_flags_off_for_two_documents():
    ids = np.array([[1, 1, 1, 2, 2, 2, 2, 2]], np.int32)
    assert oracle.chunk_dense_flags(ids, 4, 4, 4, 4) == (True, False)    # chunk = shard = document 2 alone
    assert oracle.chunk_dense_flags(ids, 2, 6, 2, 6) == (False, False)   # the chunk holds 1 and 2
    assert oracle.chunk_dense_flags(ids, 4, 4, 0, 2) == (False, False)   # cross: [0, 4) holds 1 and 2


# ---------------------------------------------------------------------------
# cross-chunk pins (the one-device core of the ring decomposition)

def test_cross_builder_golden_examples():
    with open(os.path.join(GOLDEN, "cross_examples.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        cu_q, cu_k, mq, mk = oracle.build_cross_segments(c["doc_ids"], c["q_start"], c["q_length"], c["k_start"],
                                                         c["k_length"])
        assert cu_q.tolist() == c["cu_q"], c
        assert cu_k.tolist() == c["cu_k"], c
        assert (mq, mk) == (c["max_q"], c["max_k"]), c


def test_cross_builder_rejects_chunk_after_shard_start():
    with pytest.raises(ValueError):
        oracle.build_cross_segments([[1, 1, 1, 1]], 2, 2, 1, 2)


@pytest.mark.parametrize("seed", range(25))
def test_cross_builder_brute_force_pairs_and_tiling(seed):
    r = np.random.default_rng(seed)
    B, S = int(r.integers(1, 4)), int(r.integers(2, 24))
    ids = _random_doc_ids(B, S, 300 + seed, pad_prob=0.25)
    q0 = int(r.integers(1, S))
    Lq = int(r.integers(0, S - q0 + 1))
    k0 = int(r.integers(0, q0))
    Lk = int(r.integers(0, q0 - k0 + 1))
    cu_q, cu_k, mq, mk = oracle.build_cross_segments(ids, q0, Lq, k0, Lk)
    nq, nk = np.diff(cu_q), np.diff(cu_k)
    assert len(nq) == 3 * B and cu_q[-1] == B * Lq and cu_k[-1] == B * Lk
    assert np.all(nq >= 0) and np.all(nk >= 0)
    assert mq == nq.max() and mk == nk.max()
    # every segment lies inside its own batch row of the shard and the chunk
    for s in range(3 * B):
        b = s // 3
        assert b * Lq <= cu_q[s] <= cu_q[s + 1] <= (b + 1) * Lq
        assert b * Lk <= cu_k[s] <= cu_k[s + 1] <= (b + 1) * Lk
    # non-causal pairs of the segments = same nonzero run across shard and chunk
    seg_vis = np.zeros((B * Lq, B * Lk), bool)
    for s in range(3 * B):
        seg_vis[cu_q[s]:cu_q[s + 1], cu_k[s]:cu_k[s + 1]] = True
    doc_vis = np.zeros_like(seg_vis)
    for b in range(B):
        for i in range(Lq):
            p = q0 + i
            for jj in range(Lk):
                j = k0 + jj
                run = ids[b, j:p + 1]
                if ids[b, p] != 0 and np.all(run == ids[b, p]):
                    doc_vis[b * Lq + i, b * Lk + jj] = True
    np.testing.assert_array_equal(seg_vis, doc_vis)


def _pad_fix(out, lse, qids):
    out = out.copy()
    lse = lse.copy()
    pad = np.asarray(qids).reshape(-1) == 0
    out[pad] = 0.0
    lse[:, pad] = -np.inf
    return out, lse


@pytest.mark.parametrize("seed", range(4))
def test_cross_chunk_decomposition_equals_document_mode(seed):
    # shard [q0, S) of one row: its own keys causally (segments from the
    # builder on the shard's sub-map) plus the earlier keys [0, q0) through the
    # cross segments (non-causal); the live-row merge, the pad fixup, each
    # chunk's backward fed the merged out/lse and the live-row gradient add
    # must give the document-mode result of the unsplit problem.
    r = np.random.default_rng(seed)
    S, Hq, Hkv, D = 40, 2, 1, 8
    ids = _random_doc_ids(1, S, 500 + seed, pad_prob=0.15)
    q0 = int(r.integers(8, 32))
    Lq = S - q0
    q, k, v, do = rnd(Lq, Hq, D), rnd(S, Hkv, D), rnd(S, Hkv, D), rnd(Lq, Hq, D)
    scale = 0.4
    cq1, ck1, _, _ = oracle.build_segments(ids[:, q0:], Lq, 0)
    cq2, ck2, _, _ = oracle.build_cross_segments(ids, q0, Lq, 0, q0)
    o1, l1 = oracle.attn_fwd_segments(q, k[q0:], v[q0:], cq1, ck1, scale, True)
    o2, l2 = oracle.attn_fwd_segments(q, k[:q0], v[:q0], cq2, ck2, scale, False)
    om, lm = oracle.lse_merge_live_rows(o1, l1, o2, l2, cq2, ck2)
    om, lm = _pad_fix(om, lm, ids[:, q0:])
    ref_o, ref_l = oracle.attn_fwd_document(q, k, v, ids, q0, scale, None)
    np.testing.assert_allclose(om, ref_o, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lm), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    np.testing.assert_allclose(lm[fin], ref_l[fin], atol=1e-12)
    dq1, dk1, dv1 = oracle.attn_bwd_segments(do, q, k[q0:], v[q0:], om, lm, cq1, ck1, scale, True)
    dq2, dk2, dv2 = oracle.attn_bwd_segments(do, q, k[:q0], v[:q0], om, lm, cq2, ck2, scale, False)
    dq = oracle.grad_add_live_rows(dq1, dq2, cq2, ck2)
    rq, rk, rv = oracle.attn_bwd_document(do, q, k, v, ref_o, ref_l, ids, q0, scale, None)
    np.testing.assert_allclose(dq, rq, atol=1e-10)
    np.testing.assert_allclose(np.concatenate([dk2, dk1]), rk, atol=1e-10)
    np.testing.assert_allclose(np.concatenate([dv2, dv1]), rv, atol=1e-10)
    # rows outside the cross chunk's live segments kept the local result
    live = oracle.live_rows(cq2, ck2)
    other = np.setdiff1d(np.arange(Lq), live)
    np.testing.assert_array_equal(dq[other], dq1[other])


# ---------------------------------------------------------------------------
# softcap pins

def _segments_case(seed, Tq_lens, Tk_lens, Hq=2, Hkv=1, D=6):
    r = np.random.default_rng(seed)
    cu_q = np.concatenate([[0], np.cumsum(Tq_lens)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(Tk_lens)]).astype(np.int32)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    return (cu_q, cu_k, r.standard_normal((Tq, Hq, D)), r.standard_normal((Tk, Hkv, D)),
            r.standard_normal((Tk, Hkv, D)), r.standard_normal((Tq, Hq, D)))


def test_softcap_huge_cap_is_the_plain_attention():
    cu_q, cu_k, q, k, v, do = _segments_case(1, [5, 9, 3], [7, 9, 6])
    o0, l0 = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.7, True)
    o1, l1 = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, 0.7, True, softcap=1e7)
    np.testing.assert_allclose(o1, o0, atol=1e-9)
    np.testing.assert_allclose(l1, l0, atol=1e-9)
    g0 = oracle.attn_bwd_segments(do, q, k, v, o0, l0, cu_q, cu_k, 0.7, True)
    g1 = oracle.attn_bwd_segments(do, q, k, v, o1, l1, cu_q, cu_k, 0.7, True, softcap=1e7)
    for a, b in zip(g1, g0):
        np.testing.assert_allclose(a, b, atol=1e-8)


def test_softcap_single_key_rows_closed_form():
    # one visible key: out = v exactly and lse = c * tanh(scale * q.k / c)
    cu_q, cu_k, q, k, v, _ = _segments_case(2, [1, 1], [1, 1], Hq=1)
    c, scale = 3.0, 2.5
    o, l = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, True, softcap=c)
    for row in range(2):
        np.testing.assert_allclose(o[row, 0], v[row, 0], atol=1e-14)
        z = scale * float(q[row, 0] @ k[row, 0])
        assert abs(l[0, row] - c * np.tanh(z / c)) < 1e-14


def test_softcap_bounds_every_logit():
    # all capped logits lie in (-c, c), so log n - c < lse < log n + c for a row
    # seeing n keys, however large the raw scores
    cu_q, cu_k, q, k, v, _ = _segments_case(3, [6, 4], [6, 11], Hq=2)
    c = 1.5
    _, l = oracle.attn_fwd_segments(q * 40, k * 40, v, cu_q, cu_k, 1.0, False, softcap=c)
    n = np.repeat(np.diff(cu_k), np.diff(cu_q))
    assert np.all(l < np.log(n)[None, :] + c) and np.all(l > np.log(n)[None, :] - c)


@pytest.mark.parametrize("causal,window", [(True, None), (False, 3)])
def test_softcap_gradients_match_finite_differences(causal, window):
    # d/dx of L = sum(dO * out) by central differences against the analytic
    # backward (which carries the 1 - tanh^2 factor of the cap)
    cu_q, cu_k, q, k, v, do = _segments_case(4, [4, 3], [5, 3], Hq=2, Hkv=1, D=3)
    c, scale = 1.2, 0.9

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd_segments(q_, k_, v_, cu_q, cu_k, scale, causal, window, softcap=c, nthreads=1)
        return float((o * do).sum())

    o, l = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, causal, window, softcap=c)
    dq, dk, dv = oracle.attn_bwd_segments(do, q, k, v, o, l, cu_q, cu_k, scale, causal, window, softcap=c)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=2e-7)
