"""GPU parity of strided tensor views: the attention calls read q, k, v, dout
and write out, dq, dk, dv in place through their element strides.

* Dense calls on SDPA-layout [B, H, N, D] views of [B, N, H, D] tensors
  (``x.transpose(1, 2)``), the layout callers usually hold
  [ffpa_attention page, ``_ffpa_dense_fwd`` / ``_ffpa_dense_bwd``].
* Varlen calls on packed THD views cut from one fused [T, Hq + 2 Hkv, D] QKV
  buffer, and a dout view with a padded row.

Every result is compared with the fp64 oracle on contiguous copies of the same
values; the strided forward must also equal the contiguous forward bit for bit
(the kernels load the same tiles).
"""
import numpy as np
import pytest
import torch

import oracle
import packed_sequence_flash_gb300 as psf
from packed_sequence_flash_gb300 import inputs
from gpu_helpers import assert_fwd, assert_grads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128), (512, 512)])
@pytest.mark.parametrize("causal", [True, False])
def test_dense_bnhd_views(dqk, dv, causal):
    B, Hq, Hkv, N = 2, 4, 2, 200
    factor = 0.5 if dqk == 512 else 1.0
    seed = dqk + int(causal)
    q_b = inputs.randn_bf16((B, N, Hq, dqk), seed * 4 + 0, factor)
    k_b = inputs.randn_bf16((B, N, Hkv, dqk), seed * 4 + 1, factor)
    v_b = inputs.randn_bf16((B, N, Hkv, dv), seed * 4 + 2)
    do_b = inputs.randn_bf16((B, N, Hq, dv), seed * 4 + 3)
    q, k, v, do = (t.cuda().transpose(1, 2) for t in (q_b, k_b, v_b, do_b))
    assert not q.is_contiguous()
    scale = dqk ** -0.5
    out, lse = psf.attn_dense_fwd(q, k, v, scale, causal)
    qc, kc, vc = (t.transpose(1, 2).contiguous() for t in (q_b, k_b, v_b))
    doc = do_b.transpose(1, 2).contiguous()
    out_o, lse_o = oracle.attn_fwd_dense(qc, kc, vc, scale, causal)
    assert_fwd(out, lse, out_o, lse_o)
    out_c, lse_c = psf.attn_dense_fwd(qc.cuda(), kc.cuda(), vc.cuda(), scale, causal)
    assert torch.equal(out, out_c) and torch.equal(lse, lse_c)
    grads = psf.attn_dense_bwd(do, q, k, v, out, lse, scale, causal)
    for g, x in zip(grads, (q, k, v)):
        assert g.stride() == x.stride()  # gradients keep their inputs' [B, N, H, D] storage
    ref = oracle.attn_bwd_dense(doc, qc, kc, vc, out_o, lse_o, scale, causal)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


@pytest.mark.parametrize("dqk,dv", [(64, 64), (128, 128), (192, 128)])
def test_varlen_views_of_a_fused_qkv_buffer(dqk, dv):
    r = np.random.default_rng(dqk)
    nseg, Hq, Hkv = 5, 4, 2
    mq = r.integers(1, 300, size=nseg)
    cu_q = np.concatenate([[0], np.cumsum(mq)]).astype(np.int32)
    cu_k = cu_q.copy()  # self-attention: one packed row of queries and keys
    T = int(cu_q[-1])
    if dqk == dv:
        qkv = inputs.randn_bf16((T, Hq + 2 * Hkv, dqk), 31).cuda()
        q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    else:
        # unequal head dims: q and k from one [T, Hq + Hkv, Dqk] buffer, v from another
        qk = inputs.randn_bf16((T, Hq + Hkv, dqk), 31).cuda()
        q, k = qk[:, :Hq], qk[:, Hq:]
        v = inputs.randn_bf16((T, Hkv, dv + 64), 32).cuda()[:, :, :dv]
    do = inputs.randn_bf16((T + 1, Hq, dv), 33).cuda()[1:]  # offset by one row: still 16-byte aligned
    assert not q.is_contiguous() and not k.is_contiguous()
    scale = dqk ** -0.5
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    m = int(mq.max())
    out, lse = psf.attn_varlen_fwd(q, k, v, cq, ck, m, m, scale, True, 100)
    qc, kc, vc, doc = (t.contiguous().cpu() for t in (q, k, v, do))
    out_o, lse_o = oracle.attn_fwd_segments(qc, kc, vc, cu_q, cu_k, scale, True, 100)
    assert_fwd(out, lse, out_o, lse_o)
    out_c, lse_c = psf.attn_varlen_fwd(qc.cuda(), kc.cuda(), vc.cuda(), cq, ck, m, m, scale, True, 100)
    assert torch.equal(out, out_c) and torch.equal(lse, lse_c)
    grads = psf.attn_varlen_bwd(do, q, k, v, out, lse, cq, ck, m, m, scale, True, 100)
    ref = oracle.attn_bwd_segments(doc, qc, kc, vc, out_o, lse_o, cu_q, cu_k, scale, True, 100)
    assert_grads(grads, ref)
    assert psf.device_status() == 0


def test_binding_rejects_views_the_kernels_cannot_read():
    x = torch.zeros(2, 64, 4, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="head\\) dim must be contiguous"):
        psf.attn_dense_fwd(x.transpose(1, 3), x.transpose(1, 3), x.transpose(1, 3), 0.1, True)
    y = torch.zeros(2, 4, 64, 136, dtype=torch.bfloat16, device="cuda")[..., 4:132]  # starts 8 bytes in
    with pytest.raises(ValueError, match="16-byte"):
        psf.attn_dense_fwd(y, y, y, 0.1, True)
    z = torch.zeros(2, 4, 64, 132, dtype=torch.bfloat16, device="cuda")[..., :128]  # row stride 132: not 16-byte
    with pytest.raises(ValueError, match="multiple of 8"):
        psf.attn_dense_fwd(z, z, z, 0.1, True)
