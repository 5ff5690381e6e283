"""Host-side argument validation of the C ABI, on the CPU.

Every call here is rejected by the library's host checks before it touches a
device, so no GPU is needed. The pointers are stand-in addresses that are never
dereferenced; each call also passes a NULL workspace, so that even a call whose
argument check failed to fire would stop at the workspace check (PSF_EWORKSPACE)
and never reach a launch. The pages' error contract is a ValueError on an
unusable layout [attention utils page, ``preprocess_args_and_kwargs_for_attn``,
Raises]; the binding raises ``PSFError`` (a ValueError) on any nonzero code.
"""
import ctypes

import pytest
import torch

from packed_sequence_flash_gb300 import _lib

EINVAL, EUNSUPPORTED, EWORKSPACE = -1, -2, -6
A = 0x10000  # a 16-byte-aligned stand-in address (never dereferenced)
NO_WINDOW = -(2 ** 31)


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def varlen_fwd(lib, **kw):
    a = dict(q=A, k=A, v=A, out=A, lse=A, cu_q=A, cu_k=A, meta=None, nseg=4, max_q=64, max_k=64, layout=0, dtype=0,
             B=1, Sq=256, Sk=256, Hq=4, Hkv=2, Dqk=128, Dv=128, strides=None, scale=0.125, causal=1,
             window=NO_WINDOW, softcap=0.0, flags=0, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.psf_attn_varlen_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["cu_q"], a["cu_k"], a["meta"],
                                   a["nseg"], a["max_q"], a["max_k"], a["layout"], a["dtype"], a["B"], a["Sq"],
                                   a["Sk"], a["Hq"], a["Hkv"], a["Dqk"], a["Dv"], a["strides"], a["scale"],
                                   a["causal"], a["window"], a["softcap"], a["flags"], a["ws"], a["ws_bytes"], None)


def varlen_bwd(lib, **kw):
    a = dict(dout=A, q=A, k=A, v=A, out=A, lse=A, dq=A, dk=A, dv=A, cu_q=A, cu_k=A, meta=None, nseg=4, max_q=64,
             max_k=64, layout=0, dtype=0, B=1, Sq=256, Sk=256, Hq=4, Hkv=2, Dqk=128, Dv=128, strides=None,
             scale=0.125, causal=1, window=NO_WINDOW, softcap=0.0, flags=0, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.psf_attn_varlen_bwd(a["dout"], a["q"], a["k"], a["v"], a["out"], a["lse"], a["dq"], a["dk"], a["dv"],
                                   a["cu_q"], a["cu_k"], a["meta"], a["nseg"], a["max_q"], a["max_k"], a["layout"],
                                   a["dtype"], a["B"], a["Sq"], a["Sk"], a["Hq"], a["Hkv"], a["Dqk"], a["Dv"],
                                   a["strides"], a["scale"], a["causal"], a["window"], a["softcap"], a["flags"],
                                   a["ws"], a["ws_bytes"], None)


def dense_fwd(lib, **kw):
    a = dict(q=A, k=A, v=A, out=A, lse=A, B=2, Hq=4, Hkv=2, Nq=128, Nk=128, Dqk=64, Dv=64, strides=None, dtype=0,
             scale=0.125, causal=1, window=NO_WINDOW, softcap=0.0, flags=0, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.psf_attn_dense_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Nq"],
                                  a["Nk"], a["Dqk"], a["Dv"], a["strides"], a["dtype"], a["scale"], a["causal"],
                                  a["window"], a["softcap"], a["flags"], a["ws"], a["ws_bytes"], None)


def test_the_baseline_call_stops_at_the_workspace_check(lib):
    # the reference call below is valid but for its missing workspace
    assert varlen_fwd(lib) == EWORKSPACE
    assert varlen_bwd(lib) == EWORKSPACE
    assert dense_fwd(lib) == EWORKSPACE
    assert b"workspace" in lib.psf_last_error()


@pytest.mark.parametrize("call", [varlen_fwd, varlen_bwd])
@pytest.mark.parametrize("kw,code,word", [
    (dict(Hq=6, Hkv=4), EINVAL, b"Hq"),               # Hq % Hkv != 0
    (dict(Hq=0), EINVAL, b"Hq"),
    (dict(Dqk=96, Dv=96), EUNSUPPORTED, b"head dims"),
    (dict(Dqk=128, Dv=64), EUNSUPPORTED, b"head dims"),
    (dict(window=0), EINVAL, b"window"),               # window_left == 0 is undefined
    (dict(scale=0.0), EINVAL, b"scale"),
    (dict(scale=float("nan")), EINVAL, b"scale"),
    (dict(scale=-1.0), EINVAL, b"scale"),
    (dict(softcap=-1.0), EINVAL, b"softcap"),
    (dict(softcap=float("inf")), EINVAL, b"softcap"),
    (dict(dtype=2), EINVAL, b"dtype"),
    (dict(layout=2), EINVAL, b"layout"),
    (dict(B=2), EINVAL, b"B = 1"),                     # packed THD takes one row
    (dict(Sq=-1), EINVAL, b"sizes"),
    (dict(nseg=-1), EINVAL, b"nseg"),
    (dict(flags=2), EINVAL, b"flags"),
    (dict(q=A + 8), EINVAL, b"align"),                 # base pointers must be 16-byte aligned
    (dict(v=A + 2), EINVAL, b"align"),
    (dict(q=None), EINVAL, None),
    (dict(cu_q=None), EINVAL, b"cu_q"),
])
def test_host_validation_codes(lib, call, kw, code, word):
    rc = call(lib, **kw)
    assert rc == code, (rc, lib.psf_last_error())
    if word is not None:
        assert word in lib.psf_last_error()


def test_backward_checks_its_gradient_pointers(lib):
    assert varlen_bwd(lib, dk=A + 4) == EINVAL
    assert varlen_bwd(lib, dq=None) == EINVAL
    assert varlen_bwd(lib, lse=None) == EINVAL


def test_dense_validation_codes(lib):
    assert dense_fwd(lib, Hq=3) == EINVAL
    assert dense_fwd(lib, Dqk=512, Dv=128) == EUNSUPPORTED
    assert dense_fwd(lib, window=0) == EINVAL
    assert dense_fwd(lib, out=A + 8) == EINVAL


def i64(vals):
    return (ctypes.c_int64 * len(vals))(*vals)


def test_strides_validation(lib):
    # [B, N, H, D] tensors seen as [B, H, N, D]: (batch, head, row) = (N*H*D, D, H*D)
    B, H, Hkv, N, D = 2, 4, 2, 128, 64
    bnhd = [N * H * D, D, H * D, N * Hkv * D, D, Hkv * D, N * Hkv * D, D, Hkv * D, N * H * D, D, H * D]
    assert dense_fwd(lib, strides=i64(bnhd)) == EWORKSPACE  # legal: stops at the workspace
    bad = list(bnhd)
    bad[1] = 4  # q's head stride: not a multiple of 8 elements (16 bytes)
    assert dense_fwd(lib, strides=i64(bad)) == EINVAL and b"q: head stride" in lib.psf_last_error()
    bad = list(bnhd)
    bad[8] = -Hkv * D  # v's row stride negative
    assert dense_fwd(lib, strides=i64(bad)) == EINVAL and b"v: row stride" in lib.psf_last_error()
    bad = list(bnhd)
    bad[10] = 0  # out's head stride 0: heads overlap
    assert dense_fwd(lib, strides=i64(bad)) == EINVAL and b"out" in lib.psf_last_error()
    bad = list(bnhd)
    bad[11] = 32  # out rows 32 elements apart with D = 64: rows overlap
    assert dense_fwd(lib, strides=i64(bad)) == EINVAL and b"overlaps" in lib.psf_last_error()
    # an input may overlap itself (it is only read): k's heads aliased
    ok = list(bnhd)
    ok[4] = 8
    assert dense_fwd(lib, strides=i64(ok)) == EWORKSPACE
    # THD: the batch stride is ignored, head/row strides checked
    thd = [0, 128, 4 * 128] * 4
    assert varlen_fwd(lib, Hq=4, Hkv=4, strides=i64(thd)) == EWORKSPACE
    thd_bad = list(thd)
    thd_bad[2] = 4 * 128 + 4
    assert varlen_fwd(lib, Hq=4, Hkv=4, strides=i64(thd_bad)) == EINVAL
    # the backward checks its eight tensors; dk overlapping itself is rejected
    g = [0, 128, 4 * 128] * 8
    assert varlen_bwd(lib, Hq=4, Hkv=4, strides=i64(g)) == EWORKSPACE
    g[6 * 3 + 2] = 64
    assert varlen_bwd(lib, Hq=4, Hkv=4, strides=i64(g)) == EINVAL and b"dk" in lib.psf_last_error()


def test_workspace_smaller_than_its_header_is_rejected(lib):
    # 255 bytes is below any layout's 256-byte header, so this call cannot pass
    assert lib.psf_attn_fwd_workspace_size(256, 4) > 255
    assert varlen_fwd(lib, ws=A, ws_bytes=255) == EWORKSPACE
    assert varlen_bwd(lib, ws=A, ws_bytes=255) == EWORKSPACE


def test_builder_and_memory_kernels_validation(lib):
    # builder: the shard must lie in the row; unknown flags
    assert lib.psf_build_doc_segments(A, 1, 100, 60, 50, A, A, 200, A, None, 0, None) == EINVAL
    assert lib.psf_build_doc_segments(A, 0, 100, 10, 0, A, A, 200, A, None, 0, None) == EINVAL
    assert lib.psf_build_doc_segments(A, 1, 100, 10, 0, A, A, 200, A, None, 4, None) == EINVAL
    assert lib.psf_build_doc_segments(A, 1, 100, 10, 0, None, A, 200, A, None, 0, None) == EINVAL
    # cross builder: the chunk must lie before the shard
    assert lib.psf_build_cross_segments(A, 1, 100, 50, 50, 40, 20, A, A, A, None) == EINVAL
    # dense flags: shard and chunk inside the row
    assert lib.psf_chunk_dense_flags(A, 1, 100, 90, 20, 0, 10, A, None) == EINVAL
    # merges and fixup: head dim a multiple of 8, aligned operands
    assert lib.psf_lse_merge(A, A, A, A, A, None, A, 16, 2, 12, 0, None) == EINVAL
    assert lib.psf_lse_merge(A + 8, A, A, A, A, None, A, 16, 2, 64, 0, None) == EINVAL
    assert lib.psf_lse_merge(A, A, A, A, None, None, A, 16, 2, 64, 0, None) == EINVAL
    assert lib.psf_lse_merge_live_rows(None, None, A, A, A, A, A, None, 3, 16, 2, 64, 0, None) == EINVAL
    assert lib.psf_grad_add_live_rows(A, A + 8, A, A, None, 3, 16, 2, 64, 0, None) == EINVAL
    assert lib.psf_pad_fixup(A, A, A, 0, 2, 16, 2, 64, None) == EINVAL
    assert lib.psf_pad_fixup(A, A, A, 0, 1, 16, 2, 60, None) == EINVAL


def test_noalloc_forward_limits_are_host_checks(lib):
    big = _lib.load().psf_attn_varlen_fwd_noalloc
    # more query rows or segments than the fixed schedule array holds
    rc = big(A, A, A, A, A, A, A, None, 4, 64, 64, 0, 0, 1, (1 << 20) + 1, 256, 4, 2, 128, 128, 0.125, 1, NO_WINDOW,
             None)
    assert rc == EINVAL and b"query rows" in lib.psf_last_error()
    rc = big(A, A, A, A, A, A, A, None, 65537, 64, 64, 0, 0, 1, 256, 256, 4, 2, 128, 128, 0.125, 1, NO_WINDOW, None)
    assert rc == EINVAL and b"segments" in lib.psf_last_error()


def test_binding_raises_value_error():
    import packed_sequence_flash_gb300 as psf

    q = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
    cu = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        psf.attn_varlen_fwd(q, q, q, cu, cu, 8, 8, 0.125, True)
    with pytest.raises(ValueError, match="bfloat16 or float16"):
        psf.attn_varlen_fwd(q.float(), q, q, cu, cu, 8, 8, 0.125, True)
    assert issubclass(_lib.PSFError, ValueError)
    e = _lib.PSFError(EINVAL, "window_left == 0 is undefined")
    assert "PSF_EINVAL" in str(e) and e.code == EINVAL
