"""ctypes loader for libpsf.so and the argument types of its C ABI.

There is no fallback: if the library cannot be found or built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lib = None
_lock = threading.Lock()

P = ctypes.c_void_p
I = ctypes.c_int
I32 = ctypes.c_int32
I64 = ctypes.c_int64
F = ctypes.c_float
SZ = ctypes.c_size_t
U64 = ctypes.c_uint64

# name -> (restype, argtypes); mirrors include/psf.h
SIGNATURES = {
    "psf_last_error": (ctypes.c_char_p, []),
    "psf_device_supported": (I, []),
    "psf_device_status": (I, [I]),
    "psf_set_wait_limit_ns": (None, [U64]),
    "psf_check_pipeline_wait": (I, [I, P]),
    "psf_kernel_timing": (I, [I]),
    "psf_kernel_times_ms": (I, [I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
    "psf_attn_fwd_workspace_size": (SZ, [I64, I]),
    "psf_attn_bwd_workspace_size": (SZ, [I64, I64, I, I, I, I, I]),
    "psf_attn_varlen_fwd": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, I, I, P, F, I, I32, F, I, P, SZ,
                                P]),
    "psf_attn_varlen_fwd_noalloc": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, I, I, F, I, I32, P]),
    "psf_attn_varlen_bwd": (I, [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, I, I, P, F, I,
                                I32, F, I, P, SZ, P]),
    "psf_attn_dense_fwd": (I, [P, P, P, P, P, I, I, I, I, I, I, I, P, I, F, I, I32, F, I, P, SZ, P]),
    "psf_attn_dense_bwd": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, I, F, I, I32, F, I, P, SZ, P]),
    "psf_build_doc_segments": (I, [P, I, I, I, I, P, P, I, P, P, I, P]),
    "psf_chunk_dense_flags": (I, [P, I, I, I, I, I, I, P, P]),
    "psf_pad_fixup": (I, [P, P, P, I, I, I, I, I, P]),
    "psf_lse_merge": (I, [P, P, P, P, P, P, P, I, I, I, I, P]),
    "psf_build_cross_segments": (I, [P, I, I, I, I, I, I, P, P, P, P]),
    "psf_lse_merge_live_rows": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, P]),
    "psf_grad_add_live_rows": (I, [P, P, P, P, P, I, I, I, I, I, P]),
}

PSF_LAYOUT_THD = 0
PSF_LAYOUT_BHSD = 1
PSF_DTYPE_BF16 = 0
PSF_DTYPE_F16 = 1
PSF_SEGMENTS_SKIP_PAD = 1
PSF_FWD_PACK_GQA = 1
PSF_BWD_PACK_GQA = 1
ERRORS = {-1: "PSF_EINVAL", -2: "PSF_EUNSUPPORTED", -3: "PSF_ECUDA", -4: "PSF_EDEVICE_ARGS",
          -5: "PSF_ETIMEOUT", -6: "PSF_EWORKSPACE"}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libpsf.so (building it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libpsf.so not found at {path}; run packed_sequence_flash_gb300.build")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class PSFError(ValueError):
    """A nonzero return code from the C ABI (raised as ValueError, like the pages' layout errors)."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code


def check(rc: int) -> None:
    if rc != 0:
        msg = load().psf_last_error().decode(errors="replace")
        raise PSFError(rc, msg)
