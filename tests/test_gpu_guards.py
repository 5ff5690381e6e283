"""GPU checks of the failure paths and of write bounds, through the C ABI.

* Segment arrays the schedule kernels reject on the device (a decreasing
  cu_q, a segment that runs past the last query row, a segment longer than
  max_q): the call launches, the device status reads PSF_EDEVICE_ARGS and no
  attention work runs (the outputs keep their sentinel values; the backward's
  gradients come out zero). Every array here keeps cu_q[nseg] within the rows,
  so even the preparation kernels' fill of rows past the last segment writes
  inside the tensors.
* Guard bands: out, lse, dq, dk and dv are views into larger buffers filled
  with a sentinel; after a ragged varlen forward and backward at each head-dim
  pair the bands must be untouched and the views must match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from packed_sequence_flash_gb300 import _lib, inputs
from gpu_helpers import assert_fwd, assert_grads

pytestmark = pytest.mark.gpu

EDEVICE_ARGS = -4
NO_WINDOW = -(2 ** 31)
SENTINEL = 7.0
BAND = 4096  # elements on each side of every output view (a multiple of 8: views stay 16-byte aligned)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _fwd(lib, q, k, v, out, lse, cu_q, cu_k, max_q, max_k, scale, causal, window=NO_WINDOW):
    Tq, Hq, Dqk = q.shape
    Tk, Hkv, Dv = v.shape
    nseg = cu_q.numel() - 1
    ws = torch.empty(lib.psf_attn_fwd_workspace_size(Tq, nseg), dtype=torch.uint8, device="cuda")
    return lib.psf_attn_varlen_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   cu_q.data_ptr(), cu_k.data_ptr(), None, nseg, max_q, max_k, 0, 0, 1, Tq, Tk, Hq,
                                   Hkv, Dqk, Dv, None, scale, int(causal), window, 0.0, 0, ws.data_ptr(), ws.numel(),
                                   _stream())


def _bwd(lib, do, q, k, v, out, lse, dq, dk, dv, cu_q, cu_k, max_q, max_k, scale, causal, window=NO_WINDOW):
    Tq, Hq, Dqk = q.shape
    Tk, Hkv, Dv = v.shape
    nseg = cu_q.numel() - 1
    ws = torch.empty(lib.psf_attn_bwd_workspace_size(Tq, Tk, nseg, Hq, Hkv, Dqk, Dv), dtype=torch.uint8,
                     device="cuda")
    return lib.psf_attn_varlen_bwd(do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_q.data_ptr(),
                                   cu_k.data_ptr(), None, nseg, max_q, max_k, 0, 0, 1, Tq, Tk, Hq, Hkv, Dqk, Dv, None,
                                   scale, int(causal), window, 0.0, 0, ws.data_ptr(), ws.numel(), _stream())


@pytest.mark.parametrize("case", ["decreasing_cu_q", "segment_past_the_rows", "longer_than_max_q"])
@pytest.mark.parametrize("D", [64, 192])
def test_device_rejects_bad_segment_arrays(case, D):
    lib = _lib.load()
    assert lib.psf_device_status(1) == 0
    Dqk, Dv = (D, D) if D != 192 else (192, 128)
    T, Hq, Hkv = 512, 2, 1
    max_q = max_k = 512
    cu_k = [0, 256, 512]
    if case == "decreasing_cu_q":
        cu_q, cu_k = [0, 300, 200, 512], [0, 200, 400, 512]
    elif case == "segment_past_the_rows":
        cu_q = [0, 256, 600]  # cu_q[nseg] > T: no row lies past it
    else:
        cu_q, max_q = [0, 256, 512], 128
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    q = inputs.randn_bf16((T, Hq, Dqk), 1).cuda()
    k = inputs.randn_bf16((T, Hkv, Dqk), 2).cuda()
    v = inputs.randn_bf16((T, Hkv, Dv), 3).cuda()
    out = torch.full((T, Hq, Dv), SENTINEL, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((Hq, T), SENTINEL, dtype=torch.float32, device="cuda")
    scale = Dqk ** -0.5
    assert _fwd(lib, q, k, v, out, lse, cq, ck, max_q, max_k, scale, True) == 0
    assert lib.psf_device_status(1) == EDEVICE_ARGS
    assert bool((out == SENTINEL).all()) and bool((lse == SENTINEL).all()), "attention work ran"
    do = inputs.randn_bf16((T, Hq, Dv), 4).cuda()
    out_ok = inputs.randn_bf16((T, Hq, Dv), 5).cuda()
    lse_ok = torch.zeros(Hq, T, dtype=torch.float32, device="cuda")
    dq = torch.full((T, Hq, Dqk), SENTINEL, dtype=torch.bfloat16, device="cuda")
    dk = torch.full((T, Hkv, Dqk), SENTINEL, dtype=torch.bfloat16, device="cuda")
    dv = torch.full((T, Hkv, Dv), SENTINEL, dtype=torch.bfloat16, device="cuda")
    assert _bwd(lib, do, q, k, v, out_ok, lse_ok, dq, dk, dv, cq, ck, max_q, max_k, scale, True) == 0
    assert lib.psf_device_status(1) == EDEVICE_ARGS
    # no step ran: dQ is the zeroed accumulator; the dK/dV rows of the
    # rejected segments are never written (the attention kernel writes them
    # per key tile, the convert only for the cut tiles of a valid schedule)
    assert not dq.any()
    assert bool((dk == SENTINEL).all()) and bool((dv == SENTINEL).all())
    # the context is still usable: a valid call afterwards succeeds
    good_q = torch.tensor([0, 256, 512], dtype=torch.int32, device="cuda")
    assert _fwd(lib, q, k, v, out, lse, good_q, good_q, 256, 256, scale, True) == 0
    assert lib.psf_device_status(1) == 0


def _banded(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * BAND,), SENTINEL, dtype=dtype, device="cuda")
    return buf, buf[BAND:BAND + n].view(shape)


def _bands_intact(buf, n):
    return bool((buf[:BAND] == SENTINEL).all()) and bool((buf[BAND + n:] == SENTINEL).all())


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128), (512, 512)])
def test_guard_bands_around_ragged_varlen_outputs(dqk, dv):
    lib = _lib.load()
    r = np.random.default_rng(dqk + dv)
    nseg = 4
    mq = r.integers(1, 260, size=nseg)
    mk = r.integers(1, 260, size=nseg)
    mq[0] = 129  # one tile and one row
    cu_q = np.concatenate([[0], np.cumsum(mq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(mk)]).astype(np.int32)
    Tq, Tk = int(cu_q[-1]) + 3, int(cu_k[-1])  # 3 rows outside every segment
    Hq, Hkv = 4, 2
    factor = 0.5 if dqk == 512 else 1.0
    q = inputs.randn_bf16((Tq, Hq, dqk), 11, factor)
    k = inputs.randn_bf16((Tk, Hkv, dqk), 12, factor)
    v = inputs.randn_bf16((Tk, Hkv, dv), 13)
    do = inputs.randn_bf16((Tq, Hq, dv), 14)
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    scale = dqk ** -0.5
    mxq, mxk = int(mq.max()), int(mk.max())
    out_buf, out = _banded((Tq, Hq, dv), torch.bfloat16)
    lse_buf, lse = _banded((Hq, Tq), torch.float32)
    assert _fwd(lib, q.cuda(), k.cuda(), v.cuda(), out, lse, cq, ck, mxq, mxk, scale, True) == 0
    assert lib.psf_device_status(1) == 0
    assert _bands_intact(out_buf, out.numel()) and _bands_intact(lse_buf, lse.numel())
    out_o, lse_o = oracle.attn_fwd_segments(q, k, v, cu_q, cu_k, scale, True)
    assert_fwd(out, lse, out_o, lse_o)
    dq_buf, dq = _banded((Tq, Hq, dqk), torch.bfloat16)
    dk_buf, dk = _banded((Tk, Hkv, dqk), torch.bfloat16)
    dv_buf, dv = _banded((Tk, Hkv, dv), torch.bfloat16)
    assert _bwd(lib, do.cuda(), q.cuda(), k.cuda(), v.cuda(), out, lse, dq, dk, dv, cq, ck, mxq, mxk, scale,
                True) == 0
    assert lib.psf_device_status(1) == 0
    for buf, t in ((dq_buf, dq), (dk_buf, dk), (dv_buf, dv), (out_buf, out), (lse_buf, lse)):
        assert _bands_intact(buf, t.numel())
    ref = oracle.attn_bwd_segments(do, q, k, v, out_o, lse_o, cu_q, cu_k, scale, True)
    assert_grads((dq, dk, dv), ref)
