"""Vocabulary-sharded forms across two CPU ranks (gloo): the host exchange step.

Each rank holds one shard of the same rows and builds that shard's vp_partial
records (the layout the partial kernels write) from the oracle's per-shard
sums. ``gather_partials`` must hand every rank the records of all ranks in rank
order, and merging the gathered records must give the unsharded result.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

N, V, CUT = 24, 301, 117   # shard 0 = columns [0, 117), shard 1 = [117, 301)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows():
    rng = np.random.default_rng(7)
    a = rng.normal(0, 3, (N, V))
    a[6] += 1e4                   # a large common offset
    a = a.astype(np.float32).astype(np.float64)   # fp32 values, so the records' fp32 maxima are exact
    a[3, :CUT] = -np.inf          # an all -inf shard 0
    a[5, 200] = np.nan            # a NaN in shard 1
    return a


def _pack(recs):
    """[N, 4] oracle shard records (m, S, W, bad) -> vp_partial layout, float64 [N, 5]."""
    out = np.zeros((recs.shape[0], 5))
    f32 = out.view(np.float32).reshape(-1, 10)
    u32 = out.view(np.uint32).reshape(-1, 10)
    m = recs[:, 0].copy()
    m[m == -np.inf] = -np.finfo(np.float32).max      # the library's marker of "no finite logit"
    f32[:, 0] = m
    out[:, 1] = recs[:, 1]
    out[:, 3] = recs[:, 2]
    u32[:, 9] = np.where(recs[:, 3] != 0, 1, 0)         # VP_PART_NANINF
    return out


def _unpack(parts):
    """vp_partial float64 [K, N, 5] -> oracle records [K, N, 4] through the binding's decoder."""
    from vocab_wide_logprobs_gb300.api import PART_NANINF, decode_partials
    d = decode_partials(parts)
    m = d["m"].double().numpy()
    m[m == -np.finfo(np.float32).max] = -np.inf
    bad = (d["flags"].numpy() & PART_NANINF) != 0
    return np.stack([m, d["S"].numpy(), d["W"].numpy(), bad.astype(np.float64)], axis=-1)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from vocab_wide_logprobs_gb300.tp import gather_partials
        a = _rows()
        lo, hi = (0, CUT) if rank == 0 else (CUT, V)
        mine = torch.from_numpy(_pack(oracle.shard_stats(a, lo, hi)))
        gathered = gather_partials(mine)
        H = oracle.merge_entropy_records(_unpack(gathered))
        q.put((rank, gathered.numpy(), mine.numpy(), H))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_gather_partials_two_ranks_merge_to_the_unsharded_entropy():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r, gathered, mine, H = q.get(timeout=150)
        res[r] = (gathered, mine, H)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    # every rank sees both ranks' records, in rank order, bit for bit
    for r in range(2):
        gathered = res[r][0]
        assert gathered.shape == (2, N, 5)
        for k in range(2):
            assert gathered[k].tobytes() == res[k][1].tobytes()
    # the merge of the gathered records is the unsharded entropy
    ref = oracle.entropy_fwd(_rows())[0]
    for r in range(2):
        H = res[r][2]
        assert np.array_equal(np.isnan(H), np.isnan(ref))
        fin = ~np.isnan(ref)
        assert np.allclose(H[fin], ref[fin], rtol=1e-13, atol=1e-13)


def _reduce_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from vocab_wide_logprobs_gb300.tp import reduce_dhidden
        g = torch.Generator().manual_seed(100 + rank)
        term = torch.randn(16, 64, generator=g).to(torch.bfloat16)   # this rank's dz_k . W_k
        q.put((rank, term.float().numpy(), reduce_dhidden(term).float().numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_reduce_dhidden_two_ranks_sums_the_terms_in_fp32():
    """The backward's exchange step of the sharded fused linear ops: every rank gets
    bf16(fp32 term_0 + fp32 term_1)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reduce_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r, term, total = q.get(timeout=150)
        res[r] = (term, total)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    ref = torch.from_numpy(res[0][0] + res[1][0]).to(torch.bfloat16).float().numpy()
    for r in range(2):
        assert np.array_equal(res[r][1], ref)


def test_gather_partials_rejects_records_of_the_wrong_layout():
    """The record layout is checked before any collective (no process group needed)."""
    from vocab_wide_logprobs_gb300.api import VPError
    from vocab_wide_logprobs_gb300.tp import gather_partials
    for bad in (torch.zeros(4, 4, dtype=torch.float64), torch.zeros(4, 5, dtype=torch.float32),
                torch.zeros(2, 4, 5, dtype=torch.float64)):
        with pytest.raises(VPError):
            gather_partials(bad)
