"""ctypes loader of ``libnvfp4attn.so``: the C ABI of include/nvfp4attn.h, same names.

Loading fails loudly (``NvqLibraryError``) when the library is missing: there is
no fallback implementation of any entry point.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libnvfp4attn.so")

c_void_p = ctypes.c_void_p
c_int = ctypes.c_int
c_int64 = ctypes.c_int64
c_size_t = ctypes.c_size_t
c_float = ctypes.c_float

# name -> (restype, argtypes); mirrors include/nvfp4attn.h
SIGNATURES = {
    "nvq_status_string": (ctypes.c_char_p, [c_int]),
    "nvq_version": (c_int, []),
    "nvq_last_error_detail": (ctypes.c_char_p, []),
    "nvq_device_status": (c_int, [c_void_p]),
    "nvfp4_global_sf": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p]),
    "nvfp4_fake_quant": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p, c_int64,
                                 c_void_p, c_int64, c_void_p]),
    "nvfp4_quantize_codes": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p,
                                     c_int64, c_void_p, c_int64, c_void_p]),
    "attn_qat_fwd_workspace": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_qat_fwd_layout": (c_int, [c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "attn_qat_bwd_layout": (c_int, [c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "attn_qat_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                             c_float, c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "attn_qat_fwd_hp": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                c_void_p]),
    "attn_qat_bwd_workspace": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_qat_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                             c_void_p, c_size_t, c_void_p]),
    "attn_qat_bwd_saved_workspace": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_qat_bwd_saved": (c_int, [c_void_p, c_size_t, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float,
                                   c_int, c_void_p, c_size_t, c_void_p]),
    "attn_qat_bwd_builtin_scratch": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                             c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "nvfp4_tiled_scale_bytes": (c_size_t, [c_int64, c_int64]),
    "nvfp4_quantize_tiled": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p,
                                     c_void_p, c_void_p]),
    "nvfp4_linear_workspace": (c_size_t, [c_int64, c_int64, c_int64]),
    "nvfp4_linear_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "nvfp4_linear_bwd_workspace": (c_size_t, [c_int64, c_int64, c_int64]),
    "nvfp4_linear_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "vsa_reorder": (c_int, [c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                            c_int, c_void_p, c_void_p]),
    "vsa_select_workspace": (c_size_t, [c_int, c_int, c_int, c_int]),
    "vsa_select_tiles": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p,
                                 c_void_p, c_size_t, c_void_p]),
    "attn_qat_fwd_sparse": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                    c_float, c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                                    c_size_t, c_void_p]),
    "attn_qat_bwd_sparse_workspace": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_qat_bwd_sparse": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                    c_int, c_int, c_float, c_void_p, c_size_t, c_void_p]),
    "attn_qat_bwd_sparse_saved_workspace": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_qat_bwd_sparse_saved": (c_int, [c_void_p, c_size_t, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int,
                                          c_int, c_int, c_int, c_float, c_void_p, c_size_t,
                                          c_void_p]),
    "nvq_timing_enable": (c_int, [c_int]),
    "nvq_timing_read": (c_int, [c_int, c_void_p, c_void_p]),
    "nvq_selftest_umma": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                  c_void_p]),
    "nvq_selftest_timeout": (c_int, [c_int64, c_void_p]),
    "nvq_selftest_ex2_monotone": (c_int, [c_void_p, c_void_p]),
    "nvq_selftest_fp4": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_int, c_int, c_int, c_int, c_void_p]),
}


class AttnLayout(ctypes.Structure):
    """nvq_attn_layout: byte offsets of the regions of an attention workspace."""
    _fields_ = [(name, c_size_t) for name in (
        "q_codes", "k_codes", "q_scales", "k_scales", "v_f16", "q_bf16", "k_bf16", "v_bf16",
        "delta", "total")]


STATUS = {0: "NVQ_OK", 1: "NVQ_ERR_INVALID", 2: "NVQ_ERR_UNSUPPORTED", 3: "NVQ_ERR_WORKSPACE",
          4: "NVQ_ERR_CUDA", 5: "NVQ_ERR_TIMEOUT"}


class NvqLibraryError(RuntimeError):
    """libnvfp4attn.so is missing or does not export the C ABI."""


class NvqError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        msg = f"{fn} returned {STATUS.get(status, status)}"
        super().__init__(f"{msg}: {detail}" if detail else msg)
        self.status = status
        self.detail = detail


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """The loaded library (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise NvqLibraryError(
                    f"{path} not found: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                try:
                    fn = getattr(lib, name)
                except AttributeError as e:
                    raise NvqLibraryError(f"{path} does not export {name}") from e
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def call(name: str, *args) -> int:
    """Call an entry point returning nvq_status; raise NvqError unless NVQ_OK."""
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        detail = lib.nvq_last_error_detail().decode() if st == 4 else ""
        raise NvqError(name, st, detail)
    return st
