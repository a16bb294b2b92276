"""ctypes loader for libattnmask.so (the C ABI in include/attn_block_mask.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  There is no fallback: if the library is missing this module raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattnmask.so")

c_int32 = ctypes.c_int32
c_void_p = ctypes.c_void_p


class AttnMaskParams(ctypes.Structure):
    """Mirror of ``attn_mask_params``."""
    _fields_ = [("role_think", c_int32), ("dense_bits", c_void_p), ("dense_offsets", c_void_p)]


class AttnBlockMask(ctypes.Structure):
    """Mirror of ``attn_block_mask`` in include/attn_block_mask.h."""
    _fields_ = [
        ("magic", ctypes.c_uint32),
        ("kind", c_int32),
        ("role_think", c_int32),
        ("batch", c_int32),
        ("total_tokens", c_int32),
        ("max_seqlen", c_int32),
        ("block_m", c_int32),
        ("block_n", c_int32),
        ("max_qtiles", c_int32),
        ("max_ktiles", c_int32),
        ("cu_seqlens", c_void_p),
        ("dense_bits", c_void_p),
        ("dense_offsets", c_void_p),
        ("workspace", c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("off_header", ctypes.c_uint64),
        ("off_qt_seq", ctypes.c_uint64),
        ("off_qt_idx", ctypes.c_uint64),
        ("off_labels", ctypes.c_uint64),
        ("off_kcount", ctypes.c_uint64),
        ("off_koff", ctypes.c_uint64),
        ("off_kidx", ctypes.c_uint64),
        ("off_klabel", ctypes.c_uint64),
        ("off_order", ctypes.c_uint64),
        ("off_qt_off", ctypes.c_uint64),
        ("off_summary", ctypes.c_uint64),
        ("off_pair_off", ctypes.c_uint64),
        ("off_pair_q0", ctypes.c_uint64),
        ("off_pair_order", ctypes.c_uint64),
        ("off_qcount", ctypes.c_uint64),
        ("off_qoff", ctypes.c_uint64),
        ("off_qidx", ctypes.c_uint64),
        ("off_qlabel", ctypes.c_uint64),
        ("off_korder", ctypes.c_uint64),
    ]


_lib = None


def _configure(L: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.POINTER
    L.attn_block_mask_workspace_size.argtypes = [c_int32, c_int32, c_int32, c_int32, c_int32,
                                                 P(ctypes.c_size_t)]
    L.attn_block_mask_workspace_size.restype = ctypes.c_int
    L.attn_block_mask_build.argtypes = [
        ctypes.c_int, P(AttnMaskParams), c_void_p, c_int32, c_int32, c_int32,
        c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p, ctypes.c_size_t,
        P(AttnBlockMask), c_void_p]
    L.attn_block_mask_build.restype = ctypes.c_int
    L.attn_block_mask_build_noalloc.argtypes = L.attn_block_mask_build.argtypes
    L.attn_block_mask_build_noalloc.restype = ctypes.c_int
    L.attn_fwd.argtypes = [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, ctypes.c_int, c_int32, c_int32,
        c_int32, ctypes.c_float, c_void_p, c_int32, c_int32, ctypes.c_int, P(AttnMaskParams),
        c_void_p, c_void_p, c_void_p, P(AttnBlockMask), c_void_p]
    L.attn_fwd.restype = ctypes.c_int
    L.attn_bwd_workspace_size.argtypes = [P(AttnBlockMask), c_int32, c_int32, P(ctypes.c_size_t)]
    L.attn_bwd_workspace_size.restype = ctypes.c_int
    L.attn_bwd.argtypes = [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
        ctypes.c_int, c_int32, c_int32, c_int32, ctypes.c_float, c_void_p, c_int32, c_int32,
        ctypes.c_int, P(AttnMaskParams), c_void_p, c_void_p, c_void_p, P(AttnBlockMask), c_void_p,
        ctypes.c_size_t, c_void_p]
    L.attn_bwd.restype = ctypes.c_int
    L.attn_get_status.argtypes = [P(AttnBlockMask), c_void_p]
    L.attn_get_status.restype = ctypes.c_int
    L.attn_status_string.argtypes = [ctypes.c_int]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_last_error_message.argtypes = []
    L.attn_last_error_message.restype = ctypes.c_char_p
    L.attn_version.argtypes = []
    L.attn_version.restype = c_int32
    return L


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(or block_sparse_masked_mask_gb300.build.build()).")
    _lib = _configure(ctypes.CDLL(LIB_PATH))
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Run the binding's calls through another build of the library (a copy
    compiled with other settings) inside the ``with`` block."""
    global _lib
    saved = lib()
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield _lib
    finally:
        _lib = saved
