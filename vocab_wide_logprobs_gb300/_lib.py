"""Loader of the in-tree libvp.so (the CUDA library) with every C signature declared.

There is no fallback: if the library is missing it is built from csrc/ with
nvcc (the same CUDA path), and if that fails the error propagates.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_handle = None

P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int

# name -> argument types (all return int status unless noted)
SIGNATURES = {
    "vp_logprobs_fwd": [P, I32, I64, I64, I64, I64, I64, I64, P, P, P, P, P],
    "vp_logprobs_bwd": [P, I32, I64, I64, I64, I64, I64, I64, P, P, P, P, P, P],
    "vp_logprobs_topk_fwd": [P, I32, I64, I64, I64, I64, I64, I64, P, I64, P, P, P, P],
    "vp_logprobs_topk_bwd": [P, I32, I64, I64, I64, I64, I64, I64, P, I64, P, P, P, P, P],
    "vp_entropy_fwd": [P, I32, I64, I64, I64, I64, I64, P, P, P],
    "vp_entropy_bwd": [P, I32, I64, I64, I64, I64, I64, P, P, P, P],
    "vp_kl_fwd": [P, P, I32, I64, I64, I64, I64, I64, I32, P, P, P, P],
    "vp_kl_bwd": [P, P, I32, I64, I64, I64, I64, I64, I32, P, P, P, P, P, P],
    "vp_linear_logp_fwd": [P, P, I64, I64, I64, I64, P, P, P, P, ctypes.c_size_t, P, P],
    "vp_linear_logp_fwd_noalloc": [P, P, I64, I64, I64, I64, P, P, P, P, P],
    "vp_linear_logp_bwd": [P, P, I64, I64, I64, I64, P, P, P, P, P, I32, P, ctypes.c_size_t, P, P],
    "vp_linear_entropy_fwd": [P, P, I64, I64, I64, P, P, P, ctypes.c_size_t, P],
    "vp_linear_entropy_bwd": [P, P, I64, I64, I64, P, P, P, P, I32, P, ctypes.c_size_t, P],
    "vp_linear_kl_fwd": [P, P, P, P, I64, I64, I64, I64, I32, P, P, P, P, ctypes.c_size_t, P],
    "vp_linear_kl_bwd": [P, P, P, P, I64, I64, I64, I64, I32, P, P, P, P, P, P, P, I32, P, ctypes.c_size_t, P],
    "vp_linear_jsd_fwd": [P, P, P, P, I64, I64, I64, I64, ctypes.c_double, P, P, P, P, ctypes.c_size_t, P],
    "vp_linear_logp_partial": [P, P, I64, I64, I64, I64, P, P, P, ctypes.c_size_t, P],
    "vp_linear_entropy_partial": [P, P, I64, I64, I64, P, P, ctypes.c_size_t, P],
    "vp_linear_kl_partial": [P, P, P, P, I64, I64, I64, I64, I32, P, P, ctypes.c_size_t, P],
    "vp_linear_jsd_bwd": [P, P, P, P, I64, I64, I64, I64, ctypes.c_double, P, P, P, P, P, P, P, I32, P,
                          ctypes.c_size_t, P],
    "vp_upload": [P, P, ctypes.c_size_t, P],
    "vp_download": [P, P, ctypes.c_size_t, P],
    "vp_jsd_fwd": [P, P, I32, I64, I64, I64, I64, I64, ctypes.c_double, P, P, P, P],
    "vp_jsd_bwd": [P, P, I32, I64, I64, I64, I64, I64, ctypes.c_double, P, P, P, P, P, P],
    "vp_logprobs_partial": [P, I32, I64, I64, I64, I64, I64, I64, P, P, P],
    "vp_entropy_partial": [P, I32, I64, I64, I64, I64, I64, P, P],
    "vp_kl_partial": [P, P, I32, I64, I64, I64, I64, I64, I32, P, P],
    "vp_logprobs_merge": [P, I64, I64, P, P, P, P],
    "vp_entropy_merge": [P, I64, I64, P, P, P],
    "vp_kl_merge": [P, I64, I64, I32, P, P, P, P],
}


def path() -> str:
    return _build.LIB


def lib():
    """The loaded libvp (building it first if it is absent or stale)."""
    global _handle
    with _lock:
        if _handle is None:
            so = _build.build()
            h = ctypes.CDLL(so, mode=os.RTLD_NOW | getattr(os, "RTLD_LOCAL", 0))
            for name, args in SIGNATURES.items():
                fn = getattr(h, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            h.vp_status_string.argtypes = [ctypes.c_int]
            h.vp_status_string.restype = ctypes.c_char_p
            h.vp_linear_logp_workspace_size.argtypes = [I64, I64, I64]
            h.vp_linear_logp_workspace_size.restype = ctypes.c_size_t
            h.vp_linear_logp_bwd_workspace_size.argtypes = [I64, I64, I64]
            h.vp_linear_logp_bwd_workspace_size.restype = ctypes.c_size_t
            for name, args in (("vp_linear_entropy_workspace_size", [I64, I64, I64]),
                               ("vp_linear_entropy_bwd_workspace_size", [I64, I64, I64]),
                               ("vp_linear_kl_workspace_size", [I64, I64]),
                               ("vp_linear_kl_bwd_workspace_size", [I64, I64, I64, I64]),
                               ("vp_linear_jsd_workspace_size", [I64, I64]),
                               ("vp_linear_jsd_bwd_workspace_size", [I64, I64, I64, I64])):
                fn = getattr(h, name)
                fn.argtypes = args
                fn.restype = ctypes.c_size_t
            h.vp_fault_status.argtypes = [P, I32]
            h.vp_fault_status.restype = ctypes.c_int
            h.vp_version.argtypes = []
            h.vp_version.restype = ctypes.c_int
            h.vp_set_row_split.argtypes = [I32]
            h.vp_set_row_split.restype = ctypes.c_int
            h.vp_get_row_split.argtypes = []
            h.vp_get_row_split.restype = ctypes.c_int
            _handle = h
    return _handle


def status_string(status: int) -> str:
    return lib().vp_status_string(int(status)).decode()
