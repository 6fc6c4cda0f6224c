"""Host plumbing of the vocabulary-sharded forms across ranks (torch.distributed).

Each rank holds one shard of the vocabulary and computes one vp_partial record
per row with ``vp_*_partial``. ``gather_partials`` collects every rank's
records into one ``[world, N, 5]`` tensor in rank order, which is the
shard-major layout ``vp_*_merge`` takes (the records of rank k become shard k;
the merge does not depend on which columns a shard holds). This is the
one exchange step of the sharded forms: a single all-gather of 40 bytes per row
and rank, in place of the pages' MAX then SUM all-reduces ([P1] page "Add
Triton kernels for vocab-parallel logprobs, entropy and KL", second commit
message). The library itself calls no collective.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


def gather_partials(parts: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather one rank's ``[N, 5]`` float64 records into ``[world, N, 5]`` (rank order)."""
    if parts.dim() != 2 or parts.shape[1] != api.PARTIAL_DOUBLES or parts.dtype != torch.float64:
        raise api.VPError(2, "records must be a float64 [N, 5] tensor")
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(parts.shape), dtype=parts.dtype, device=parts.device)
    dist.all_gather(list(out.unbind(0)), parts.contiguous(), group=group)
    return out


def tp_entropy_fwd(x_shard, group=None):
    """Entropy of rows whose vocabulary is split across the ranks of `group`: (H, stats) on every rank."""
    return api.vp_entropy_merge(gather_partials(api.vp_entropy_partial(x_shard), group))


def tp_logprobs_fwd(x_shard, targets, vocab_start: int, group=None, err_word=None):
    """logp of global target ids over rows split across ranks: (logp, stats) on every rank."""
    parts = api.vp_logprobs_partial(x_shard, targets, vocab_start)
    return api.vp_logprobs_merge(gather_partials(parts, group), err_word=err_word)


def tp_kl_fwd(a_shard, b_shard, direction: int = api.KL_REVERSE, group=None):
    """KL over rows split across ranks: (kl, stats_a, stats_b) on every rank."""
    return api.vp_kl_merge(gather_partials(api.vp_kl_partial(a_shard, b_shard, direction), group), direction)


# ---------------------------------------------------------------------------
# The fused linear ops with the head's rows split across ranks ([P2] page "[Feat]
# [Kernel] Add TP Fused linear logp Triton", "Implementation"): each rank holds
# hidden in full and its shard of W's rows; the forward is one record gather,
# and the backward's dhidden is the sum of every rank's term (reduce_dhidden).
# ---------------------------------------------------------------------------
def tp_linear_logp_fwd(hidden, w_shard, targets, vocab_start: int, group=None, err_word=None):
    """logp of global target ids with the head's rows split across ranks: (logp, stats) on every rank."""
    parts = api.vp_linear_logp_partial(hidden, w_shard, targets, vocab_start)
    return api.vp_logprobs_merge(gather_partials(parts, group), err_word=err_word)


def tp_linear_entropy_fwd(hidden, w_shard, group=None):
    """Entropy of softmax(hidden @ W^T) with W's rows split across ranks: (H, stats) on every rank."""
    return api.vp_entropy_merge(gather_partials(api.vp_linear_entropy_partial(hidden, w_shard), group))


def tp_linear_kl_fwd(ha, wa_shard, hb, wb_shard, direction: int = api.KL_REVERSE, group=None):
    """KL of two models whose heads' rows are split the same way across ranks: (kl, stats_a, stats_b)."""
    parts = api.vp_linear_kl_partial(ha, wa_shard, hb, wb_shard, direction)
    return api.vp_kl_merge(gather_partials(parts, group), direction)


def reduce_dhidden(dh_term: torch.Tensor, group=None) -> torch.Tensor:
    """dhidden from every rank's bf16 term dz_k . W_k: summed in fp32 across the ranks, rounded to bf16."""
    total = dh_term.float()
    dist.all_reduce(total, op=dist.ReduceOp.SUM, group=group)
    return total.to(torch.bfloat16)
