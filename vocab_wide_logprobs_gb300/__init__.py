"""Vocab-wide logprobs, entropy and KL (and fused linear logp) on GB300.

The compute runs in ``libvp.so`` (hand-written CUDA for sm_103a behind a C-ABI,
declared in ``include/vp.h``). ``api`` is a thin ctypes binding with the same
function names: it turns torch tensors into pointers, sizes and strides and
calls the C functions. There is no CPU fallback: every call raises if the
library cannot be built or loaded, or if no sm_103 device is present.
"""
from .api import (KL_FORWARD, KL_REVERSE, ROW_EMPTY, ROW_MISMATCH, ROW_NANINF, VPError, decode_rowstats, rows_of,
                  rowstats, vp_entropy_bwd, vp_entropy_fwd, vp_fault_status, vp_kl_bwd, vp_kl_fwd, vp_linear_logp_bwd, vp_linear_logp_bwd_workspace_size, vp_linear_logp_fwd,
                  vp_linear_logp_workspace_size, vp_logprobs_bwd, vp_logprobs_fwd)

__all__ = ["KL_FORWARD", "KL_REVERSE", "ROW_EMPTY", "ROW_MISMATCH", "ROW_NANINF", "VPError", "decode_rowstats",
           "rows_of", "rowstats", "vp_entropy_bwd", "vp_entropy_fwd", "vp_kl_bwd", "vp_kl_fwd", "vp_logprobs_bwd",
           "vp_logprobs_fwd", "vp_fault_status",
           "vp_linear_logp_fwd", "vp_linear_logp_workspace_size", "vp_linear_logp_bwd",
           "vp_linear_logp_bwd_workspace_size"]
