"""CPU-side checks of the C ABI: the library builds, loads and exports every
symbol include/psf.h declares, and the binding's signature table matches it.
No compute call is made (there may be no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "psf.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(psf_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ["psf_attn_varlen_fwd", "psf_attn_varlen_bwd", "psf_attn_dense_fwd", "psf_attn_dense_bwd",
                 "psf_build_doc_segments", "psf_pad_fixup", "psf_lse_merge", "psf_device_supported",
                 "psf_last_error", "psf_device_status", "psf_attn_fwd_workspace_size",
                 "psf_attn_bwd_workspace_size"]:
        assert must in names


def test_library_exports_every_declared_symbol():
    from packed_sequence_flash_gb300 import build

    path = build.build()
    lib = ctypes.CDLL(path)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from packed_sequence_flash_gb300 import _lib

    assert sorted(_lib.SIGNATURES) == declared_symbols()


def test_workspace_size_queries_need_no_gpu():
    from packed_sequence_flash_gb300 import _lib

    lib = _lib.load()
    a = lib.psf_attn_fwd_workspace_size(8192, 11)
    b = lib.psf_attn_bwd_workspace_size(8192, 8192, 11, 16, 4, 128, 128)
    assert a >= 256 + 8 * (8192 // 128)
    assert b >= 4 * 8192 * 16 * 128 + 4 * 16 * 8192 + 4 * 8192 * 4 * 256
    assert lib.psf_attn_fwd_workspace_size(-1, 0) == 0


def test_last_error_is_a_string():
    from packed_sequence_flash_gb300 import _lib

    assert isinstance(_lib.load().psf_last_error(), bytes)
