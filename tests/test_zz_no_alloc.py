"""The forward entry point that allocates nothing (psf_attn_varlen_fwd_noalloc).

It exists for callers that cannot call cudaMalloc while they run, for example
runtimes that reserve all device memory up front or plugin hosts that own
every allocation. It keeps its tile schedule in a fixed array inside the
library instead of a caller workspace. These checks call it through the C ABI
twice in a row, a large call and then a small one, and once at its segment
limit, and compare each result with the ordinary workspace-taking entry point
on the same inputs, within the parity tolerances of the other GPU tests. This
file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


def _case(seed, nseg, max_len):
    from packed_sequence_flash_gb300 import inputs

    r = np.random.default_rng(seed)
    mq = r.integers(0, max_len, size=nseg)
    mk = r.integers(1, max_len, size=nseg)
    cu_q = np.concatenate([[0], np.cumsum(mq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(mk)]).astype(np.int32)
    Tq, Tk = int(cu_q[-1]) + 5, int(cu_k[-1])
    q = inputs.randn_bf16((Tq, 4, 128), 100 + seed).cuda()
    k = inputs.randn_bf16((Tk, 2, 128), 200 + seed).cuda()
    v = inputs.randn_bf16((Tk, 2, 128), 300 + seed).cuda()
    return q, k, v, torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda(), int(mq.max()), int(mk.max())


def _call(lib, noalloc, q, k, v, cu_q, cu_k, mq, mk, window):
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    nseg = cu_q.numel() - 1
    out = torch.full((Tq, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((Hq, Tq), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    head = [q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), cu_q.data_ptr(),
            cu_k.data_ptr(), None, nseg, mq, mk, 0, 0, 1, Tq, Tk, Hq, Hkv, D, D]
    tail = [1.0 / np.sqrt(D), 1, window]
    if noalloc:
        rc = lib.psf_attn_varlen_fwd_noalloc(*head, *tail, stream)
        ws = None
    else:
        ws = torch.empty(lib.psf_attn_fwd_workspace_size(Tq, nseg), dtype=torch.uint8, device="cuda")
        rc = lib.psf_attn_varlen_fwd(*head, None, *tail, 0.0, 0, ws.data_ptr(), ws.numel(), stream)
    assert rc == 0, lib.psf_last_error()
    torch.cuda.synchronize()
    return out, lse


def _same(out_n, lse_n, out_w, lse_w, call):
    o_n, o_w = out_n.double().cpu().numpy(), out_w.double().cpu().numpy()
    l_n, l_w = lse_n.double().cpu().numpy(), lse_w.double().cpu().numpy()
    assert not np.isnan(o_n).any() and not np.isnan(l_n).any(), f"call {call}: unwritten output"
    assert np.max(np.abs(o_n - o_w)) <= OUT_TOL, f"call {call}"
    assert np.array_equal(np.isneginf(l_n), np.isneginf(l_w)), f"call {call}"
    fin = np.isfinite(l_w)
    if fin.any():
        assert np.max(np.abs(l_n[fin] - l_w[fin])) <= LSE_TOL, f"call {call}"


def test_noalloc_forward_matches_workspace_forward_twice():
    # A large call (many segments and tiles) and then a much smaller one: the
    # second must not see anything the first left in the shared array.
    from packed_sequence_flash_gb300 import _lib

    lib = _lib.load()
    for call, (seed, nseg, max_len, window) in enumerate([(1, 40, 700, -(2 ** 31)), (2, 1, 40, 120)]):
        args = _case(seed, nseg, max_len)
        out_n, lse_n = _call(lib, True, *args, window)
        out_w, lse_w = _call(lib, False, *args, window)
        assert lib.psf_device_status(1) == 0
        _same(out_n, lse_n, out_w, lse_w, call)


def test_noalloc_forward_at_its_segment_limit():
    # PSF_NOALLOC_MAX_SEGMENTS segments: all but the last have one key and no
    # query; the last holds 200 queries against 300 keys.
    from packed_sequence_flash_gb300 import _lib, inputs

    lib = _lib.load()
    nseg = 65536
    mq = np.zeros(nseg, np.int64)
    mk = np.ones(nseg, np.int64)
    mq[-1], mk[-1] = 200, 300
    cu_q = torch.from_numpy(np.concatenate([[0], np.cumsum(mq)]).astype(np.int32)).cuda()
    cu_k = torch.from_numpy(np.concatenate([[0], np.cumsum(mk)]).astype(np.int32)).cuda()
    Tq, Tk = 200, int(mk.sum())
    q = inputs.randn_bf16((Tq, 4, 128), 7).cuda()
    k = inputs.randn_bf16((Tk, 2, 128), 8).cuda()
    v = inputs.randn_bf16((Tk, 2, 128), 9).cuda()
    out_n, lse_n = _call(lib, True, q, k, v, cu_q, cu_k, 200, 300, -(2 ** 31))
    assert lib.psf_device_status(1) == 0
    out_w, lse_w = _call(lib, False, q, k, v, cu_q, cu_k, 200, 300, -(2 ** 31))
    assert lib.psf_device_status(1) == 0
    _same(out_n, lse_n, out_w, lse_w, "at the segment limit")


def test_noalloc_forward_rejects_sizes_beyond_its_limit():
    from packed_sequence_flash_gb300 import _lib

    lib = _lib.load()
    q, k, v, cu_q, cu_k, mq, mk = _case(3, 6, 300)
    rc = lib.psf_attn_varlen_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), q.data_ptr(),
                                         cu_q.data_ptr(), cu_k.data_ptr(), None, 65537, mq, mk, 0, 0, 1, q.shape[0],
                                         k.shape[0], 4, 2, 128, 128, 0.1, 1, -1, None)
    assert rc == -1 and b"segments" in lib.psf_last_error()
    rc = lib.psf_attn_varlen_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), q.data_ptr(),
                                         cu_q.data_ptr(), cu_k.data_ptr(), None, 6, mq, mk, 1, 0, 2, 1 << 20, 16, 4, 2,
                                         128, 128, 0.1, 1, -1, None)
    assert rc == -1 and b"query rows" in lib.psf_last_error()
