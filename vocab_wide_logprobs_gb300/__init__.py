"""Vocab-wide logprobs, entropy, KL and JSD (and their fused linear forms) on GB300.

The compute runs in ``libvp.so`` (hand-written CUDA for sm_103a behind a C-ABI,
declared in ``include/vp.h``). ``api`` is a thin ctypes binding with the same
function names: it turns torch tensors into pointers, sizes and strides and
calls the C functions. There is no CPU fallback: every call raises if the
library cannot be built or loaded, or if no sm_103 device is present.
"""
from .api import (GRAD_EXACT, GRAD_FAST, KL_FORWARD, KL_REVERSE, PART_HAS_TARGET, PART_IGNORED, PART_MISMATCH,
                 PART_NANINF, PART_NANINF_B, ROW_BADTARGET, ROW_EMPTY, ROW_MISMATCH, ROW_NANINF, ROW_SHARDED, VPError,
                 decode_partials, decode_rowstats, partials, rows_of, rowstats, vp_download, vp_entropy_bwd,
                 vp_entropy_fwd, vp_entropy_merge, vp_entropy_partial, vp_fault_status, vp_get_row_split, vp_jsd_bwd,
                 vp_jsd_fwd, vp_kl_bwd, vp_kl_fwd, vp_kl_merge, vp_kl_partial, vp_linear_entropy_bwd,
                 vp_linear_entropy_bwd_workspace_size, vp_linear_entropy_fwd, vp_linear_entropy_partial,
                 vp_linear_entropy_workspace_size, vp_linear_jsd_bwd, vp_linear_jsd_bwd_workspace_size,
                 vp_linear_jsd_fwd, vp_linear_jsd_workspace_size, vp_linear_kl_bwd, vp_linear_kl_bwd_workspace_size,
                 vp_linear_kl_fwd, vp_linear_kl_partial, vp_linear_kl_workspace_size, vp_linear_logp_bwd,
                 vp_linear_logp_bwd_workspace_size, vp_linear_logp_fwd, vp_linear_logp_fwd_noalloc,
                 vp_linear_logp_partial, vp_linear_logp_workspace_size, vp_logprobs_bwd, vp_logprobs_fwd,
                 vp_logprobs_merge, vp_logprobs_partial, vp_logprobs_topk_bwd, vp_logprobs_topk_fwd, vp_set_row_split,
                 vp_status_string, vp_upload, vp_version)

__all__ = ["GRAD_EXACT", "GRAD_FAST", "KL_FORWARD", "KL_REVERSE", "PART_HAS_TARGET", "PART_IGNORED", "PART_MISMATCH",
           "PART_NANINF", "PART_NANINF_B", "ROW_BADTARGET", "ROW_EMPTY", "ROW_MISMATCH", "ROW_NANINF", "ROW_SHARDED",
           "VPError", "decode_partials", "decode_rowstats", "partials", "rows_of", "rowstats", "vp_download",
           "vp_entropy_bwd", "vp_entropy_fwd", "vp_entropy_merge", "vp_entropy_partial", "vp_fault_status",
           "vp_get_row_split", "vp_jsd_bwd", "vp_jsd_fwd", "vp_kl_bwd", "vp_kl_fwd", "vp_kl_merge", "vp_kl_partial",
           "vp_linear_entropy_bwd", "vp_linear_entropy_bwd_workspace_size", "vp_linear_entropy_fwd",
           "vp_linear_entropy_partial", "vp_linear_entropy_workspace_size", "vp_linear_jsd_bwd",
           "vp_linear_jsd_bwd_workspace_size", "vp_linear_jsd_fwd", "vp_linear_jsd_workspace_size",
           "vp_linear_kl_bwd", "vp_linear_kl_bwd_workspace_size", "vp_linear_kl_fwd", "vp_linear_kl_partial",
           "vp_linear_kl_workspace_size", "vp_linear_logp_bwd", "vp_linear_logp_bwd_workspace_size",
           "vp_linear_logp_fwd", "vp_linear_logp_fwd_noalloc", "vp_linear_logp_partial",
           "vp_linear_logp_workspace_size", "vp_logprobs_bwd", "vp_logprobs_fwd", "vp_logprobs_merge",
           "vp_logprobs_partial", "vp_logprobs_topk_bwd", "vp_logprobs_topk_fwd", "vp_set_row_split",
           "vp_status_string", "vp_upload", "vp_version"]
