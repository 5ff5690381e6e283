"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, at sizes that span several 128-row tiles and ragged tails.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import packed_sequence_flash_gb300 as psf
from packed_sequence_flash_gb300 import inputs
from gpu_helpers import assert_fwd, assert_grads, cuda, doc_case, np64

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _build_gpu(ids, Lq, q0, skip_pad=False):
    ids_t = torch.as_tensor(np.asarray(ids, np.int32)).to("cuda")
    cu_q, cu_k, meta, pad = psf.build_doc_segments(ids_t, Lq, q0, want_pad_flags=True, skip_pad=skip_pad)
    m = meta.cpu().tolist()
    n = m[0]
    return cu_q[: n + 1].cpu().numpy(), cu_k[: n + 1].cpu().numpy(), m[1], m[2], pad[:n].cpu().numpy()


# ---------------------------------------------------------------- builder (bit-exact)

def test_builder_golden_examples_bit_exact():
    with open(os.path.join(GOLDEN, "builder_examples.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        cu_q, cu_k, mq, mk, pad = _build_gpu(c["doc_ids"], c["q_length"], c["q_global_start"])
        assert cu_q.tolist() == c["cu_q"] and cu_k.tolist() == c["cu_k"], c
        assert (mq, mk) == (c["max_q"], c["max_k"])


@pytest.mark.parametrize("seed", range(12))
def test_builder_random_maps_bit_exact(seed):
    r = np.random.default_rng(seed)
    B = int(r.integers(1, 4))
    S = int(r.integers(1, 20000))
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        pos, d = 0, 1
        while pos < S:
            n = int(r.integers(1, 3000))
            ids[b, pos:pos + n] = 0 if r.random() < 0.2 else d
            d += 1
            pos += n
    q0 = int(r.integers(0, S))
    Lq = int(r.integers(0, S - q0 + 1))
    got = _build_gpu(ids, Lq, q0)
    ref = oracle.build_segments(ids, Lq, q0)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])
    assert (got[2], got[3]) == (ref[2], ref[3])
    starts = ref[1][:-1]
    np.testing.assert_array_equal(got[4], (ids.reshape(-1)[starts] == 0).astype(np.uint8))


def test_builder_skip_pad_golden_examples_bit_exact():
    with open(os.path.join(GOLDEN, "builder_skip_pad_examples.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        cu_q, cu_k, mq, mk, pad = _build_gpu(c["doc_ids"], c["q_length"], c["q_global_start"], skip_pad=True)
        assert cu_q.tolist() == c["cu_q"] and cu_k.tolist() == c["cu_k"], c
        assert (mq, mk) == (c["max_q"], c["max_k"])


@pytest.mark.parametrize("seed", range(8))
def test_builder_skip_pad_random_maps_bit_exact(seed):
    r = np.random.default_rng(50 + seed)
    B = int(r.integers(1, 4))
    S = int(r.integers(1, 20000))
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        pos, d = 0, 1
        while pos < S:
            n = int(r.integers(1, 3000 if seed % 2 else 40))
            ids[b, pos:pos + n] = 0 if r.random() < 0.3 else d
            d += 1
            pos += n
    q0 = int(r.integers(0, S))
    Lq = int(r.integers(0, S - q0 + 1))
    got = _build_gpu(ids, Lq, q0, skip_pad=True)
    ref = oracle.build_segments(ids, Lq, q0, skip_pad=True)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])
    assert (got[2], got[3]) == (ref[2], ref[3])
    # a padding flag on both segments of every padding piece
    kid = ids.reshape(-1)
    nk = np.diff(ref[1])
    first_key = np.where(nk > 0, ref[1][:-1], -1)
    for s_ in range(len(nk)):
        if first_key[s_] >= 0:
            assert got[4][s_] == (kid[first_key[s_]] == 0)


def test_document_path_skip_pad_equals_pad_fixup_path():
    # the two ways of zeroing padding queries give the same forward (bitwise:
    # every non-padding row runs the same tiles) and the same gradients
    w = inputs.config(2, seed=1)
    q, k, v, do = (cuda(t) for t in (w.q, w.k, w.v, w.dout))
    ids = torch.from_numpy(w.doc_ids).to("cuda")
    res = []
    for skip in (True, False):
        out, lse, seg = psf.document_causal_attention(q, k, v, ids, ids, 0, w.scale, None, skip_pad=skip)
        g = psf.document_causal_attention_backward(do, q, k, v, out, lse, seg, w.scale)
        res.append((out, lse, g))
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])
    for a, b in zip(res[0][2], res[1][2]):
        e = float(torch.linalg.norm(a.float() - b.float()) / torch.linalg.norm(b.float()))
        assert e <= 1e-3, e
    pad_rows = (ids[0] == 0).nonzero().flatten()
    assert pad_rows.numel() > 0
    assert float(res[0][0][pad_rows].abs().max()) == 0.0
    assert bool(torch.isneginf(res[0][1][:, pad_rows]).all())


def test_builder_rejects_unknown_flags():
    ids = torch.ones(1, 8, dtype=torch.int32, device="cuda")
    cu = torch.empty(20, dtype=torch.int32, device="cuda")
    meta = torch.empty(3, dtype=torch.int32, device="cuda")
    from packed_sequence_flash_gb300 import _lib
    rc = _lib.load().psf_build_doc_segments(ids.data_ptr(), 1, 8, 8, 0, cu.data_ptr(), cu.data_ptr(), 19,
                                            meta.data_ptr(), None, 2, None)
    assert rc == -1  # PSF_EINVAL


@pytest.mark.parametrize("cfg", [2, 4, 5])
def test_builder_full_size_configs_bit_exact(cfg):
    w = inputs.config(cfg, seed=0)
    Lq = w.q.shape[0]
    got = _build_gpu(w.doc_ids, Lq, w.q_global_start)
    ref = oracle.build_segments(w.doc_ids, Lq, w.q_global_start)
    for a, b in zip(got[:4], ref):
        np.testing.assert_array_equal(np.asarray(a), np.asarray(b))


def test_builder_capacity_too_small_reports_device_args():
    ids = torch.tensor([[1, 1, 2, 2, 3]], dtype=torch.int32, device="cuda")
    psf.build_doc_segments(ids, 5, 0, capacity=2)
    assert psf.device_status() == -4


def test_pipeline_wait_runs_out_and_reports_timeout():
    # The failure path of every bounded pipeline wait, without a fault: a wait
    # that nothing completes gives up after the limit, the status word reads
    # PSF_ETIMEOUT, and the context stays usable.
    assert psf.device_status() == 0
    psf.set_wait_limit_ns(2_000_000)
    try:
        psf.check_pipeline_wait(arrive=True)
        assert psf.device_status() == 0
        psf.check_pipeline_wait(arrive=False)
        assert psf.device_status() == -5
        assert psf.device_status() == 0
    finally:
        psf.set_wait_limit_ns(2_000_000_000)
    w = inputs.small_document_workload(500, 2, 1, 64, 64, 4, max_len=200)
    doc_case(w)


# ---------------------------------------------------------------- forward + backward, varlen

def _rand_segments(r, nseg, max_len, allow_empty=True):
    mq = r.integers(0 if allow_empty else 1, max_len, size=nseg)
    mk = r.integers(0 if allow_empty else 1, max_len, size=nseg)
    cu_q = np.concatenate([[0], np.cumsum(mq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(mk)]).astype(np.int32)
    return cu_q, cu_k


def _varlen_case(seed, Dqk, Dv, Hq, Hkv, causal, window, nseg=5, max_len=400, tail_q=0, tail_k=0,
                 dtype=torch.bfloat16, softcap=None, factor=1.0):
    r = np.random.default_rng(seed)
    cu_q, cu_k = _rand_segments(r, nseg, max_len)
    Tq, Tk = int(cu_q[-1]) + tail_q, int(cu_k[-1]) + tail_k
    q = inputs.randn16((Tq, Hq, Dqk), seed * 7 + 1, factor, dtype=dtype)
    k = inputs.randn16((Tk, Hkv, Dqk), seed * 7 + 2, factor, dtype=dtype)
    v = inputs.randn16((Tk, Hkv, Dv), seed * 7 + 3, dtype=dtype)
    do = inputs.randn16((Tq, Hq, Dv), seed * 7 + 4, dtype=dtype)
    scale = 1.0 / np.sqrt(Dqk)
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    mq, mk = int(np.diff(cu_q).max()), int(np.diff(cu_k).max())
    out, lse = psf.attn_varlen_fwd(cuda(q), cuda(k), cuda(v), cq, ck, mq, mk, scale, causal, window, softcap=softcap)
    assert out.dtype == dtype
    out_o, lse_o = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, causal, window, softcap=softcap)
    assert_fwd(out, lse, out_o, lse_o)
    grads = psf.attn_varlen_bwd(cuda(do), cuda(q), cuda(k), cuda(v), out, lse, cq, ck, mq, mk, scale, causal,
                                window, softcap=softcap)
    assert all(g.dtype == dtype for g in grads)
    ref = oracle.attn_bwd_segments(do, q, k, v, out_o, lse_o, cu_q, cu_k, scale, causal, window, softcap=softcap)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("causal,window", [(True, None), (False, None), (True, 97), (False, 150)])
def test_varlen_fwd_bwd_matches_oracle(dims, causal, window):
    _varlen_case(3, dims[0], dims[1], 4, 2, causal, window)


def test_varlen_gqa_ratio_4_with_uncovered_tail_rows():
    _varlen_case(5, 128, 128, 8, 2, True, None, nseg=4, max_len=300, tail_q=37, tail_k=21)


def test_varlen_many_small_and_empty_segments():
    _varlen_case(11, 128, 128, 2, 1, True, None, nseg=40, max_len=40)


@pytest.mark.parametrize("D,Hq,causal,pack,dtype", [(128, 1, True, False, torch.bfloat16),
                                                    (128, 1, False, False, torch.bfloat16),
                                                    (64, 2, True, False, torch.float16),
                                                    (128, 4, True, True, torch.bfloat16)])
def test_backward_cut_key_tiles_match_oracle(D, Hq, causal, pack, dtype):
    """One KV head and one long segment plus a short one: the schedule cuts
    almost every key tile of the long segment into sub-ranges (the per-range
    step cap is at its floor of 4), so most dK/dV rows come from the convert's
    sum of partial-sum slots, and the short segment's tiles and the ragged
    last tile from the attention kernel's direct writes."""
    Hkv = 1
    cu_q = np.array([0, 2048 - 37, 2048 - 37 + 150], dtype=np.int32)
    cu_k = np.array([0, 2048 - 37, 2048 - 37 + 150], dtype=np.int32)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    q = inputs.randn16((Tq, Hq, D), 901, dtype=dtype)
    k = inputs.randn16((Tk, Hkv, D), 902, dtype=dtype)
    v = inputs.randn16((Tk, Hkv, D), 903, dtype=dtype)
    do = inputs.randn16((Tq, Hq, D), 904, dtype=dtype)
    scale = 1.0 / np.sqrt(D)
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    mq, mk = int(np.diff(cu_q).max()), int(np.diff(cu_k).max())
    out, lse = psf.attn_varlen_fwd(cuda(q), cuda(k), cuda(v), cq, ck, mq, mk, scale, causal)
    out_o, lse_o = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, causal, None)
    assert_fwd(out, lse, out_o, lse_o)
    grads = psf.attn_varlen_bwd(cuda(do), cuda(q), cuda(k), cuda(v), out, lse, cq, ck, mq, mk, scale, causal,
                                pack_gqa=pack)
    ref = oracle.attn_bwd_segments(do, q, k, v, out_o, lse_o, cu_q, cu_k, scale, causal, None)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


@pytest.mark.parametrize("D", [64, 128, 512])
def test_degenerate_calls_no_rows_no_segments_no_keys(D):
    # Calls with nothing to attend: no query rows, no segments, no keys, and a
    # backward with no queries. Every query row comes out 0 with lse = -inf
    # and every gradient is 0 (rows that see no key carry no probability).
    dev, dt, H, Hkv = "cuda", torch.bfloat16, 4, 2
    g = torch.Generator().manual_seed(5)
    rnd = lambda *s: torch.randn(*s, generator=g).to(dt).to(dev)
    z = lambda *s: torch.tensor(s, dtype=torch.int32, device=dev)
    scale = D ** -0.5
    # no query rows (keys present)
    q0, k, v = rnd(0, H, D), rnd(10, Hkv, D), rnd(10, Hkv, D)
    out, lse = psf.attn_varlen_fwd(q0, k, v, z(0, 0), z(0, 10), 0, 10, scale, True)
    assert out.shape == (0, H, D) and lse.shape == (H, 0)
    dq, dk, dv = psf.attn_varlen_bwd(q0.clone(), q0, k, v, out, lse, z(0, 0), z(0, 10), 0, 10, scale, True)
    assert dq.shape == (0, H, D) and not dk.any() and not dv.any()
    # no segments at all: every row is uncovered
    q = rnd(50, H, D)
    out, lse = psf.attn_varlen_fwd(q, k, v, z(0), z(0), 0, 0, scale, True)
    assert not out.any() and bool(torch.isneginf(lse).all())
    dq, dk, dv = psf.attn_varlen_bwd(rnd(50, H, D), q, k, v, out, lse, z(0), z(0), 0, 0, scale, True)
    assert not dq.any() and not dk.any() and not dv.any()
    # no keys: segments with queries and zero keys
    k0, v0 = rnd(0, Hkv, D), rnd(0, Hkv, D)
    out, lse = psf.attn_varlen_fwd(q, k0, v0, z(0, 20, 50), z(0, 0, 0), 30, 0, scale, False)
    assert not out.any() and bool(torch.isneginf(lse).all())
    dq, dk, dv = psf.attn_varlen_bwd(rnd(50, H, D), q, k0, v0, out, lse, z(0, 20, 50), z(0, 0, 0), 30, 0, scale,
                                     False)
    assert not dq.any() and dk.shape == (0, Hkv, D) and dv.shape == (0, Hkv, D)
    assert psf.device_status() == 0


# ---------------------------------------------------------------- document-causal composition

@pytest.mark.parametrize("seed,skip_pad", [(0, True), (1, True), (1, False)])
def test_document_causal_small_rows(seed, skip_pad):
    w = inputs.small_document_workload(900, 4, 2, 128, 128, seed, max_len=350, pad_tail=61)
    doc_case(w, skip_pad=skip_pad)


def test_document_causal_d512_padding_skip():
    # the wide kernels' zero-key (padding query) and zero-query (padding key) units
    w = inputs.small_document_workload(600, 2, 1, 512, 512, 6, max_len=200, pad_tail=45)
    doc_case(w)


def test_document_causal_shard_and_window():
    w = inputs.small_document_workload(1000, 4, 4, 192, 128, 2, q_global_start=400, max_len=500, pad_tail=33)
    doc_case(w, window=150)


def test_document_causal_d64_window_one():
    w = inputs.small_document_workload(500, 2, 1, 64, 64, 3, max_len=200)
    doc_case(w, window=1)


# ---------------------------------------------------------------- dense

def _dense_case(B, Hq, Hkv, Nq, Nk, Dqk, Dv, causal, window=None, seed=0, factor=1.0, dtype=torch.bfloat16,
                softcap=None):
    w = inputs.dense_workload(B, Hq, Hkv, Nq, Nk, Dqk, Dv, seed, factor=factor, causal=causal)
    w.q, w.k, w.v, w.dout = (t.to(dtype) for t in (w.q, w.k, w.v, w.dout))
    q, k, v, do = (cuda(t) for t in (w.q, w.k, w.v, w.dout))
    out, lse = psf.attn_dense_fwd(q, k, v, w.scale, causal, window, softcap=softcap)
    out_o, lse_o = oracle.attn_fwd_dense(w.q, w.k, w.v, w.scale, causal, window, softcap=softcap)
    assert_fwd(out, lse, out_o, lse_o)
    grads = psf.attn_dense_bwd(do, q, k, v, out, lse, w.scale, causal, window, softcap=softcap)
    ref = oracle.attn_bwd_dense(w.dout, w.q, w.k, w.v, out_o, lse_o, w.scale, causal, window, softcap=softcap)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


def test_dense_config1_exact_shape():
    _dense_case(1, 2, 1, 128, 128, 64, 64, True)


@pytest.mark.parametrize("causal", [True, False])
def test_dense_rectangular_batched(causal):
    _dense_case(2, 4, 2, 200, 333, 128, 128, causal, seed=1)


def test_dense_more_queries_than_keys_bottom_right():
    _dense_case(1, 2, 2, 300, 130, 128, 128, True, seed=2)


def test_dense_d512_forward_backward():
    _dense_case(1, 4, 2, 300, 300, 512, 512, True, seed=3, factor=0.5)


def test_varlen_d512_window_noncausal():
    _varlen_case(4, 512, 512, 2, 1, False, 90, nseg=3, max_len=260)


def test_dense_d512_gqa8_window():
    # eight query heads per KV head (steps walk 8 heads x the query tiles of a
    # key tile) under a left window that leaves some key tiles few queries
    _dense_case(1, 8, 1, 520, 520, 512, 512, True, window=150, seed=6, factor=0.5)


@pytest.mark.parametrize("causal", [True, False])
def test_dense_d512_more_units_than_clusters(causal):
    # 2 batches x 4 KV heads x 6 key tiles = 48 (key tile, KV head) units for
    # the at most 38 four-CTA clusters of the head-dim-512 backward: some
    # clusters take a second unit (K_r reloaded, dV/dK read out and restarted,
    # no early S^T across the unit boundary), every row checked
    _dense_case(2, 8, 4, 768, 768, 512, 512, causal, seed=5, factor=0.5)


# ---------------------------------------------------------------- pad fixup and merge

def test_pad_fixup_zeroes_pad_rows():
    w = inputs.small_document_workload(400, 2, 2, 64, 64, 4, max_len=100, pad_tail=50)
    doc_case(w, check_bwd=False, skip_pad=False)


def test_lse_merge_matches_oracle_and_neg_inf_rows():
    r = np.random.default_rng(0)
    T, H, D = 300, 4, 128
    o1 = inputs.randn_bf16((T, H, D), 1)
    o2 = inputs.randn_bf16((T, H, D), 2)
    l1 = torch.from_numpy(r.standard_normal((H, T)).astype(np.float32))
    l2 = torch.from_numpy(r.standard_normal((H, T)).astype(np.float32))
    l1[:, :10] = -np.inf
    l2[:, 5:15] = -np.inf
    of, ob, l = psf.lse_merge(cuda(o1), cuda(l1), cuda(o2), cuda(l2), want_f32=True, want_bf16=True)
    o_ref, l_ref = oracle.lse_merge(o1, l1, o2, l2)
    assert np.max(np.abs(of.cpu().numpy() - o_ref)) < 1e-5
    assert np.max(np.abs(ob.float().cpu().numpy() - o_ref)) < 2e-2
    lg = l.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.max(np.abs(lg[fin] - l_ref[fin])) < 1e-5
    assert not np.isnan(of.cpu().numpy()).any()


# ---------------------------------------------------------------- cross-chunk pieces

def _build_cross_gpu(ids, q0, Lq, k0, Lk):
    ids_t = torch.as_tensor(np.asarray(ids, np.int32)).to("cuda")
    cu_q, cu_k, meta = psf.build_cross_segments(ids_t, q0, Lq, k0, Lk)
    m = meta.cpu().tolist()
    return cu_q.cpu().numpy(), cu_k.cpu().numpy(), m


def test_cross_builder_golden_examples_bit_exact():
    with open(os.path.join(GOLDEN, "cross_examples.json")) as fh:
        cases = json.load(fh)["cases"]
    for c in cases:
        cu_q, cu_k, m = _build_cross_gpu(c["doc_ids"], c["q_start"], c["q_length"], c["k_start"], c["k_length"])
        assert cu_q.tolist() == c["cu_q"] and cu_k.tolist() == c["cu_k"], c
        assert m == [len(c["cu_q"]) - 1, c["max_q"], c["max_k"]], c


@pytest.mark.parametrize("seed", range(12))
def test_cross_builder_random_maps_bit_exact(seed):
    r = np.random.default_rng(seed)
    B = int(r.integers(1, 4))
    S = int(r.integers(2, 40000))
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        pos, d = 0, 1
        while pos < S:
            n = int(r.integers(1, 6000))
            ids[b, pos:pos + n] = 0 if r.random() < 0.2 else d
            d += 1
            pos += n
    q0 = int(r.integers(1, S))
    Lq = int(r.integers(0, S - q0 + 1))
    k0 = int(r.integers(0, q0))
    Lk = int(r.integers(0, q0 - k0 + 1))
    cu_q, cu_k, m = _build_cross_gpu(ids, q0, Lq, k0, Lk)
    ref = oracle.build_cross_segments(ids, q0, Lq, k0, Lk)
    np.testing.assert_array_equal(cu_q, ref[0])
    np.testing.assert_array_equal(cu_k, ref[1])
    assert m == [3 * B, ref[2], ref[3]]


def test_cross_builder_rejects_chunk_after_shard():
    ids = torch.ones(1, 16, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        psf.build_cross_segments(ids, 4, 8, 2, 4)


def _live_case(seed, H=3, D=64):
    """30 segments with 0-59 query rows each; about a third have no keys."""
    r = np.random.default_rng(seed)
    nq = r.integers(0, 60, size=30)
    cu_q = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    nk = r.integers(0, 3, size=30) * r.integers(1, 50, size=30)
    cu_k = np.concatenate([[0], np.cumsum(nk)]).astype(np.int32)
    T = int(cu_q[-1])
    o_run = inputs.randn_bf16((T, H, D), seed * 3 + 1)
    o_new = inputs.randn_bf16((T, H, D), seed * 3 + 2)
    l_acc = torch.from_numpy(r.standard_normal((H, T)).astype(np.float32))
    l_new = torch.from_numpy(r.standard_normal((H, T)).astype(np.float32))
    l_acc[:, : T // 10] = -np.inf
    l_new[:, T // 20: T // 7] = -np.inf
    return cu_q, cu_k, o_run, l_acc, o_new, l_new


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lse_merge_live_rows_matches_oracle(seed):
    cu_q, cu_k, o_run, l_acc, o_new, l_new = _live_case(seed)
    o_ref, l_ref = oracle.lse_merge_live_rows(o_run, l_acc, o_new, l_new, cu_q, cu_k)
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    # running output held in bf16, merged in place
    ob, lb = cuda(o_run).clone(), cuda(l_acc).clone()
    psf.lse_merge_live_rows(ob, lb, cuda(o_new), cuda(l_new), cq, ck)
    # running output held in fp32 (and mirrored to bf16)
    of, lf, ob2 = cuda(o_run).float().clone(), cuda(l_acc).clone(), cuda(o_run).clone()
    psf.lse_merge_live_rows(ob2, lf, cuda(o_new), cuda(l_new), cq, ck, o_acc=of)
    assert psf.device_status() == 0
    live = oracle.live_rows(cu_q, cu_k)
    other = np.setdiff1d(np.arange(o_run.shape[0]), live)
    for o, l in ((ob, lb), (of, lf), (ob2, lf)):
        og, lg = np64(o), np64(l)
        assert not np.isnan(og).any() and not np.isnan(lg).any()
        assert np.max(np.abs(og - o_ref)) < 2e-2
        assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
        fin = np.isfinite(l_ref)
        assert np.max(np.abs(lg[fin] - l_ref[fin])) < 1e-5
    # rows outside the live segments are untouched, bit for bit
    np.testing.assert_array_equal(ob.cpu()[other].view(torch.int16).numpy(), o_run[other].view(torch.int16).numpy())
    np.testing.assert_array_equal(np64(lb)[:, other], np64(l_acc)[:, other])
    assert np.max(np.abs(np64(of) - o_ref)) < 1e-5


def test_grad_add_live_rows_matches_oracle():
    cu_q, cu_k, a, _, b, _ = _live_case(5, H=4, D=128)
    ref = oracle.grad_add_live_rows(a, b, cu_q, cu_k)
    dst = cuda(a).clone()
    psf.grad_add_live_rows(dst, cuda(b), torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda())
    assert psf.device_status() == 0
    got = np64(dst)
    # one bf16 rounding of the fp32 sum
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)) < 8e-3
    other = np.setdiff1d(np.arange(a.shape[0]), oracle.live_rows(cu_q, cu_k))
    np.testing.assert_array_equal(dst.cpu()[other].view(torch.int16).numpy(), a[other].view(torch.int16).numpy())


# ---------------------------------------------------------------- fp16 inputs

@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("causal,window", [(True, None), (False, 150)])
def test_varlen_fwd_bwd_fp16_matches_oracle(dims, causal, window):
    _varlen_case(13, dims[0], dims[1], 4, 2, causal, window, dtype=torch.float16)


def test_dense_d512_fp16_forward_backward():
    _dense_case(1, 4, 2, 260, 260, 512, 512, True, seed=4, factor=0.5, dtype=torch.float16)


def test_document_causal_fp16():
    w = inputs.small_document_workload(900, 4, 2, 128, 128, 5, max_len=350, pad_tail=61)
    w.q, w.k, w.v, w.dout = (t.to(torch.float16) for t in (w.q, w.k, w.v, w.dout))
    doc_case(w)


def test_lse_merge_and_live_rows_fp16():
    cu_q, cu_k, o_run, l_acc, o_new, l_new = _live_case(7)
    o_run, o_new = o_run.to(torch.float16), o_new.to(torch.float16)
    _, ob, l = psf.lse_merge(cuda(o_run), cuda(l_acc), cuda(o_new), cuda(l_new), want_f32=False, want_bf16=True)
    assert ob.dtype == torch.float16
    o_ref, l_ref = oracle.lse_merge(o_run, l_acc, o_new, l_new)
    assert np.max(np.abs(np64(ob) - o_ref)) < 5e-3
    run, lr = cuda(o_run).clone(), cuda(l_acc).clone()
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    psf.lse_merge_live_rows(run, lr, cuda(o_new), cuda(l_new), cq, ck)
    o_lv, _ = oracle.lse_merge_live_rows(o_run, l_acc, o_new, l_new, cu_q, cu_k)
    assert np.max(np.abs(np64(run) - o_lv)) < 5e-3
    dst = cuda(o_run).clone()
    psf.grad_add_live_rows(dst, cuda(o_new), cq, ck)
    ref = oracle.grad_add_live_rows(o_run, o_new, cu_q, cu_k)
    assert np.max(np.abs(np64(dst) - ref)) < 1e-2
    assert psf.device_status() == 0


def test_mixed_dtypes_are_rejected():
    q = torch.zeros(128, 2, 64, dtype=torch.float16, device="cuda")
    k = torch.zeros(128, 1, 64, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 128], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        psf.attn_varlen_fwd(q, k, k, cu, cu, 128, 128, 0.125, True)


# ---------------------------------------------------------------- dense routing of ring chunks

def test_chunk_dense_flags_golden_bit_exact():
    with open(os.path.join(GOLDEN, "dense_route_examples.json")) as fh:
        chunks = json.load(fh)["chunks"]
    for c in chunks:
        ids = torch.as_tensor(np.asarray(c["doc_ids"], np.int32)).to("cuda")
        got = psf.chunk_dense_eligible(ids, c["q_start"], c["q_length"], c["k_start"], c["k_length"])
        assert got == (c["local"], c["cross"]), c


@pytest.mark.parametrize("seed", range(10))
def test_chunk_dense_flags_random_bit_exact(seed):
    r = np.random.default_rng(70 + seed)
    B, S = int(r.integers(1, 4)), int(r.integers(2, 5000))
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        kind = int(r.integers(0, 3))
        if kind == 0:    # one document then padding
            ids[b, :int(r.integers(0, S + 1))] = 5
        elif kind == 1:  # one document
            ids[b] = 7
        else:            # several documents
            pos, d = 0, 1
            while pos < S:
                n = int(r.integers(1, S // 2 + 2))
                ids[b, pos:pos + n] = 0 if r.random() < 0.2 else d
                d += 1
                pos += n
    q0 = int(r.integers(1, S))
    Lq = S - q0 if seed % 2 else int(r.integers(1, S - q0 + 1))
    for k0, Lk in ((q0, Lq), (0, q0 + Lq), (0, q0), (int(r.integers(0, q0)), 1)):
        want = oracle.chunk_dense_flags(ids, q0, Lq, k0, Lk)
        got = psf.chunk_dense_eligible(torch.from_numpy(ids).cuda(), q0, Lq, k0, Lk)
        assert got == want, (k0, Lk)


def _chunk_case(role, seed, D=128, window=None):
    r = np.random.default_rng(seed)
    B, S, Hq, Hkv = 2, 700, 4, 2
    q0 = int(r.integers(200, 400))
    Lq = S - q0
    ids = np.zeros((B, S), np.int32)
    for b in range(B):
        ids[b, :q0 + int(r.integers(1, Lq + 1))] = b + 2
    if role == "local":  # the chunk ends where the shard ends
        k0 = int(r.integers(0, q0))
        Lk = S - k0
    else:  # the chunk lies before the shard, inside the shared document
        k0 = int(r.integers(0, q0 // 2))
        Lk = int(r.integers(1, q0 - k0 + 1))
    causal = role == "local"
    q = inputs.randn16((B, Hq, Lq, D), 10 * seed + 1)
    k = inputs.randn16((B, Hkv, Lk, D), 10 * seed + 2)
    v = inputs.randn16((B, Hkv, Lk, D), 10 * seed + 3)
    do = inputs.randn16((B, Hq, Lq, D), 10 * seed + 4)
    idt = torch.from_numpy(ids).cuda()
    res = {}
    for dense in (None, False):
        out, lse, plan = psf.chunk_attention(cuda(q), cuda(k), cuda(v), idt, q0, k0, 1.0 / np.sqrt(D), causal,
                                             window, dense=dense)
        grads = psf.chunk_attention_backward(cuda(do), cuda(q), cuda(k), cuda(v), out, lse, plan, 1.0 / np.sqrt(D))
        res[dense] = (out, lse, grads, plan[0])
    assert res[None][3] == "dense" and res[False][3] == "segments"
    # the oracle: document mode over the chunk (local) or the cross segments
    pk = lambda x: np64(x).transpose(0, 2, 1, 3).reshape(-1, x.shape[1], x.shape[3])
    if causal:
        ro, rl = oracle.attn_fwd_document(pk(q), pk(k), pk(v), ids[:, k0:], q0 - k0, 1.0 / np.sqrt(D), window)
        rg = oracle.attn_bwd_document(pk(do), pk(q), pk(k), pk(v), ro, rl, ids[:, k0:], q0 - k0, 1.0 / np.sqrt(D),
                                      window)
    else:
        cu_q, cu_k, _, _ = oracle.build_cross_segments(ids, q0, Lq, k0, Lk)
        ro, rl = oracle.attn_fwd_segments(pk(q), pk(k), pk(v), cu_q, cu_k, 1.0 / np.sqrt(D), False)
        rg = oracle.attn_bwd_segments(pk(do), pk(q), pk(k), pk(v), ro, rl, cu_q, cu_k, 1.0 / np.sqrt(D), False)
    for dense in (None, False):
        out, lse, grads, _ = res[dense]
        o_p = out.permute(0, 2, 1, 3).reshape(-1, Hq, D)
        l_p = lse.permute(1, 0, 2).reshape(Hq, -1)
        assert_fwd(o_p, l_p, ro, rl)
        assert_grads(tuple(g.permute(0, 2, 1, 3).reshape(-1, g.shape[1], g.shape[3]) for g in grads), rg)
    assert psf.device_status() == 0


@pytest.mark.parametrize("seed", [0, 1])
def test_chunk_attention_local_dense_route_matches_oracle(seed):
    _chunk_case("local", seed)


def test_chunk_attention_local_dense_route_window():
    _chunk_case("local", 5, D=64, window=90)


@pytest.mark.parametrize("seed", [2, 3])
def test_chunk_attention_cross_dense_route_matches_oracle(seed):
    _chunk_case("cross", seed)


# ---------------------------------------------------------------- packed query heads (pack-GQA forward)

@pytest.mark.parametrize("D,G,causal,window", [(128, 4, True, None), (128, 2, False, None), (64, 8, True, 37),
                                               (128, 16, True, None), (64, 4, False, 21)])
def test_varlen_fwd_pack_gqa_matches_unpacked_and_oracle(D, G, causal, window):
    # many short segments (and a few long ones, and empty ones) with the query
    # heads of a KV head packed into one tile
    r = np.random.default_rng(100 + G + D)
    lens_q = [int(x) for x in r.integers(0, 40, 60)] + [300, 129, 0, 1]
    lens_k = [lq + int(r.integers(0, 20)) if causal else int(r.integers(0, 60)) for lq in lens_q]
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    Hkv = 2
    Hq = G * Hkv
    Tq, Tk = int(cu_q[-1]) + 5, int(cu_k[-1])
    q = inputs.randn16((Tq, Hq, D), G * 31 + 1)
    k = inputs.randn16((Tk, Hkv, D), G * 31 + 2)
    v = inputs.randn16((Tk, Hkv, D), G * 31 + 3)
    scale = 1.0 / np.sqrt(D)
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    mq, mk = max(lens_q), max(lens_k)
    out_p, lse_p = psf.attn_varlen_fwd(cuda(q), cuda(k), cuda(v), cq, ck, mq, mk, scale, causal, window,
                                       pack_gqa=True)
    out_u, lse_u = psf.attn_varlen_fwd(cuda(q), cuda(k), cuda(v), cq, ck, mq, mk, scale, causal, window)
    out_o, lse_o = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, causal, window)
    assert_fwd(out_p, lse_p, out_o, lse_o)
    assert float((out_p.float() - out_u.float()).abs().max()) <= 1e-2
    fin = torch.isfinite(lse_u)
    assert torch.equal(fin, torch.isfinite(lse_p))
    assert float((lse_p[fin] - lse_u[fin]).abs().max()) <= 1e-4
    assert psf.device_status() == 0


def test_document_causal_pack_gqa_with_backward():
    w = inputs.small_document_workload(1500, 8, 2, 128, 128, 7, max_len=90, pad_tail=40)
    q, k, v, do = (cuda(t) for t in (w.q, w.k, w.v, w.dout))
    ids = torch.from_numpy(w.doc_ids).to("cuda")
    out, lse, seg = psf.document_causal_attention(q, k, v, ids, ids, 0, w.scale, None, pack_gqa=True)
    out_o, lse_o = oracle.attn_fwd_document(w.q, w.k, w.v, w.doc_ids, 0, w.scale, None)
    assert_fwd(out, lse, out_o, lse_o)
    grads = psf.document_causal_attention_backward(do, q, k, v, out, lse, seg, w.scale, pack_gqa=True)
    ref = oracle.attn_bwd_document(w.dout, w.q, w.k, w.v, out_o, lse_o, w.doc_ids, 0, w.scale, None)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


@pytest.mark.parametrize("D,G,causal,window,cap", [(128, 4, True, None, None), (64, 2, False, None, None),
                                                   (128, 2, True, 45, None), (64, 4, True, None, 2.0),
                                                   (128, 8, True, None, None)])
def test_varlen_bwd_pack_gqa_matches_oracle(D, G, causal, window, cap):
    # short and long segments, empty ones, uncovered tail rows; G = 8 asks for
    # packing that the backward does not do (same results either way)
    r = np.random.default_rng(300 + G + D)
    lens_q = [int(x) for x in r.integers(0, 50, 30)] + [260, 0, 3]
    lens_k = [lq + int(r.integers(0, 20)) if causal else int(r.integers(1, 70)) for lq in lens_q]
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    Hkv = 2
    Hq = G * Hkv
    Tq, Tk = int(cu_q[-1]) + 7, int(cu_k[-1])
    q = inputs.randn16((Tq, Hq, D), G * 41 + 1)
    k = inputs.randn16((Tk, Hkv, D), G * 41 + 2)
    v = inputs.randn16((Tk, Hkv, D), G * 41 + 3)
    do = inputs.randn16((Tq, Hq, D), G * 41 + 4)
    scale = 1.0 / np.sqrt(D)
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    mq, mk = max(lens_q), max(lens_k)
    out, lse = psf.attn_varlen_fwd(cuda(q), cuda(k), cuda(v), cq, ck, mq, mk, scale, causal, window, softcap=cap,
                                   pack_gqa=True)
    out_o, lse_o = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, causal, window, softcap=cap)
    assert_fwd(out, lse, out_o, lse_o)
    grads = psf.attn_varlen_bwd(cuda(do), cuda(q), cuda(k), cuda(v), out, lse, cq, ck, mq, mk, scale, causal,
                                window, softcap=cap, pack_gqa=True)
    ref = oracle.attn_bwd_segments(do, q, k, v, out_o, lse_o, cu_q, cu_k, scale, causal, window, softcap=cap)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


def test_dense_fwd_pack_gqa_matches_oracle():
    q = inputs.randn16((2, 8, 100, 64), 501)
    k = inputs.randn16((2, 2, 160, 64), 502)
    v = inputs.randn16((2, 2, 160, 64), 503)
    out, lse = psf.attn_dense_fwd(cuda(q), cuda(k), cuda(v), 0.125, True, pack_gqa=True)
    out_o, lse_o = oracle.attn_fwd_dense(q, k, v, 0.125, True)
    assert_fwd(out.reshape(-1, 64), lse.reshape(-1), out_o.reshape(-1, 64), lse_o.reshape(-1))
    assert psf.device_status() == 0


# ---------------------------------------------------------------- logit softcap

@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("causal,window,cap", [(True, None, 1.5), (False, None, 4.0), (True, 97, 30.0)])
def test_varlen_softcap_matches_oracle(dims, causal, window, cap):
    # inputs scaled up so that the cap bends the logits
    _varlen_case(21, dims[0], dims[1], 4, 2, causal, window, factor=2.0, softcap=cap)


def test_dense_d512_softcap_forward_backward():
    _dense_case(1, 4, 2, 300, 300, 512, 512, True, seed=9, factor=1.0, softcap=2.0)


def test_varlen_softcap_fp16_and_gqa():
    _varlen_case(23, 128, 128, 8, 2, True, None, nseg=6, max_len=300, dtype=torch.float16, factor=2.0,
                 softcap=3.0)


def test_document_causal_softcap():
    w = inputs.small_document_workload(900, 4, 2, 128, 128, 8, max_len=350, pad_tail=61)
    q, k, v, do = (cuda(t) for t in (w.q, w.k, w.v, w.dout))
    ids = torch.from_numpy(w.doc_ids).to("cuda")
    out, lse, seg = psf.document_causal_attention(q, k, v, ids, ids, 0, w.scale, None, softcap=2.5)
    out_o, lse_o = oracle.attn_fwd_document(w.q, w.k, w.v, w.doc_ids, 0, w.scale, None, softcap=2.5)
    assert_fwd(out, lse, out_o, lse_o)
    grads = psf.document_causal_attention_backward(do, q, k, v, out, lse, seg, w.scale, softcap=2.5)
    ref = oracle.attn_bwd_document(w.dout, w.q, w.k, w.v, out_o, lse_o, w.doc_ids, 0, w.scale, None, softcap=2.5)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


def test_softcap_rejects_negative():
    q = torch.zeros(8, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(8, 1, 64, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 8], dtype=torch.int32, device="cuda")
    with pytest.raises(psf.PSFError):
        psf.attn_varlen_fwd(q, k, k, cu, cu, 8, 8, 0.125, True, softcap=-1.0)
