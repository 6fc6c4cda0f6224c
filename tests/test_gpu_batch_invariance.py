"""Bitwise batch invariance and the two row-split settings of the forward scans.

A row's results (outputs, saved statistics, gradient rows) must not depend on
how many rows share the call, nor on which rows they are: each case runs a
batch, then sub-batches of it, and compares the sub-batch rows bit for bit.
Every forward-scan case runs under both settings of vp_set_row_split (one CTA
per row, or the two CTAs of a cluster per row, which engages for rows of 64 KB
or more); under the split the results are also held to the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import vocab_wide_logprobs_gb300 as vp
from vocab_wide_logprobs_gb300 import workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(v):
    if v.dtype == torch.bfloat16:
        return v.view(torch.int16)
    if v.dtype in (torch.float32, torch.int32):
        return v.view(torch.int32)
    return v.contiguous().view(torch.uint8)   # row records


def _same_rows(full: dict, part: dict, lo: int, hi: int, tag: str):
    for k, v in part.items():
        if k == "err" or v is None:
            continue
        ref = full[k][lo:hi]
        assert torch.equal(_bits(v.contiguous()), _bits(ref.contiguous())), f"{tag}{k}: rows {lo}:{hi} differ bitwise"


@pytest.fixture(params=[1, 2], ids=["one CTA per row", "two CTAs per row"])
def row_split(request):
    old = vp.vp_get_row_split()
    vp.vp_set_row_split(request.param)
    yield request.param
    vp.vp_set_row_split(old)


def test_row_split_setting_round_trips():
    old = vp.vp_get_row_split()
    try:
        vp.vp_set_row_split(2)
        assert vp.vp_get_row_split() == 2
        with pytest.raises(vp.VPError):
            vp.vp_set_row_split(3)
        assert vp.vp_get_row_split() == 2
    finally:
        vp.vp_set_row_split(old)


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 75968), (torch.float32, 20011)], ids=["bf16", "fp32"])
def test_all_ops_sub_batches(row_split, dtype, V):
    N = 400
    w = workloads.pages_shape(seed=41, N=N, V=V, dtype=dtype)
    a, b, t, g = (w[k].to(DEV) for k in ("a", "b", "targets", "grad"))
    full = parity.gpu_all(a, b, t, g)
    for lo, hi in ((0, 1), (0, 7), (5, 12), (100, 333), (N - 1, N)):
        _same_rows(full, parity.gpu_all(a[lo:hi], b[lo:hi], t[lo:hi], g[lo:hi]), lo, hi, f"{dtype} ")


def test_strided_unaligned_sub_batches(row_split):
    # rows read in place from [B, T, V + 2] tensors, starting one element in (not 16-byte aligned)
    gen = torch.Generator().manual_seed(12)
    B, T, V = 4, 40, 40001
    A = (torch.randn(B, T, V + 2, generator=gen) * 3).to(torch.bfloat16).to(DEV)
    Bt = (torch.randn(B, T, V + 2, generator=gen) * 3).to(torch.bfloat16).to(DEV)
    tg = torch.randint(0, V, (B, T - 1), generator=gen).to(DEV)
    g = torch.randn(B, T - 1, generator=gen).to(DEV)
    a, b = A[:, 1:, 1:V + 1], Bt[:, 1:, 1:V + 1]
    full = parity.gpu_all(a, b, tg, g)
    for b0, b1 in ((0, 1), (1, 3), (3, 4)):
        part = parity.gpu_all(a[b0:b1], b[b0:b1], tg[b0:b1], g[b0:b1])
        _same_rows(full, part, b0 * (T - 1), b1 * (T - 1), "strided ")


def test_jsd_sub_batches(row_split):
    w = workloads.pages_shape(seed=43, N=96, V=75968)
    a, b, g = (w[k].to(DEV) for k in ("a", "b", "grad"))

    def run(lo, hi):
        j, sa, sb = vp.vp_jsd_fwd(a[lo:hi], b[lo:hi], 0.3)
        da, db = vp.vp_jsd_bwd(a[lo:hi], b[lo:hi], 0.3, sa, sb, g[lo:hi])
        torch.cuda.synchronize()
        return {"jsd": j, "sa": sa, "sb": sb, "da": da, "db": db}

    full = run(0, 96)
    for lo, hi in ((0, 1), (17, 40), (95, 96)):
        _same_rows(full, run(lo, hi), lo, hi, "jsd ")


def test_topk_sub_batches(row_split):
    w = workloads.pages_shape(seed=44, N=128, V=75968)
    x = w["a"].to(DEV)
    gen = torch.Generator().manual_seed(44)
    t = torch.randint(0, 75968, (128, 5), generator=gen).to(DEV)
    g = torch.randn(128, 5, generator=gen).to(DEV)

    def run(lo, hi):
        lp, st = vp.vp_logprobs_topk_fwd(x[lo:hi], t[lo:hi])
        dx = vp.vp_logprobs_topk_bwd(x[lo:hi], t[lo:hi], st, g[lo:hi])
        torch.cuda.synchronize()
        return {"logp": lp, "stats": st, "dx": dx}

    full = run(0, 128)
    for lo, hi in ((0, 3), (64, 65), (100, 128)):
        _same_rows(full, run(lo, hi), lo, hi, "top-k ")


def test_shard_partials_sub_batches(row_split):
    w = workloads.pages_shape(seed=45, N=64, V=75968)
    a, b, t = (w[k].to(DEV) for k in ("a", "b", "targets"))

    def run(lo, hi):
        out = {"lp": vp.vp_logprobs_partial(a[lo:hi], t[lo:hi] + 1000, vocab_start=1000),
               "H": vp.vp_entropy_partial(a[lo:hi]), "kl": vp.vp_kl_partial(a[lo:hi], b[lo:hi])}
        torch.cuda.synchronize()
        return out

    full = run(0, 64)
    for lo, hi in ((0, 1), (9, 30)):
        _same_rows(full, run(lo, hi), lo, hi, "partials ")


def test_linear_dhidden_sub_batches():
    # the backward's vocabulary chunk is fixed for N <= 8192, so each dhidden row's sums are too
    w = workloads.linear(seed=46, N=384, V=2000, D=256)
    h, W, t, g = (w[k].to(DEV) for k in ("hidden", "weight", "targets", "grad"))

    def run(lo, hi):
        lp, st = vp.vp_linear_logp_fwd(h[lo:hi].contiguous(), W, t[lo:hi].contiguous())
        dh, _ = vp.vp_linear_logp_bwd(h[lo:hi].contiguous(), W, t[lo:hi].contiguous(), st, g[lo:hi].contiguous(),
                                      want_dW=False)
        torch.cuda.synchronize()
        return {"logp": lp, "stats": st, "dhidden": dh}

    full = run(0, 384)
    for lo, hi in ((0, 1), (128, 256), (383, 384)):
        _same_rows(full, run(lo, hi), lo, hi, "linear ")


# ---------------------------------------------------------------------------
# Under the split: parity with the oracle (the merge of the two segments is
# the re-centred sum the one-CTA path uses for its warp partials)
# ---------------------------------------------------------------------------
SPLIT_SHAPES = [(24, 75968, torch.bfloat16), (9, 32768, torch.bfloat16), (7, 16384, torch.float32),
                (5, 40001, torch.float32), (6, 131072, torch.bfloat16)]


@pytest.mark.parametrize("N,V,dtype", SPLIT_SHAPES, ids=[f"{n}x{v}-{str(d)[6:]}" for n, v, d in SPLIT_SHAPES])
def test_split_rows_against_oracle(N, V, dtype):
    old = vp.vp_get_row_split()
    vp.vp_set_row_split(2)
    try:
        w = workloads.pages_shape(seed=N + V, N=N, V=V, dtype=dtype)
        a, b, t, g = (w[k].to(DEV) for k in ("a", "b", "targets", "grad"))
        got = parity.gpu_all(a, b, t, g)
        ref = parity.oracle_all(parity.rows2d(a), parity.rows2d(b), t.cpu().numpy(), g.cpu().numpy())
        parity.compare_all(got, ref, tag=f"split {N}x{V} ")
        assert int(got["err"].item()) == ref["err"]
    finally:
        vp.vp_set_row_split(old)


def test_split_unaligned_rows_against_oracle():
    # head and tail elements read directly by the first and the last CTA of the pair
    old = vp.vp_get_row_split()
    vp.vp_set_row_split(2)
    try:
        gen = torch.Generator().manual_seed(47)
        V = 40003
        A = (torch.randn(6, V + 3, generator=gen) * 3).to(torch.bfloat16).to(DEV)
        Bt = (torch.randn(6, V + 3, generator=gen) * 3).to(torch.bfloat16).to(DEV)
        a, b = A[:, 3:], Bt[:, 3:]
        t = torch.randint(0, V, (6,), generator=gen)
        t[0], t[1], t[2] = 0, 1, V - 1           # targets in the head and in the tail
        g = torch.randn(6, generator=gen)
        got = parity.gpu_all(a, b, t.to(DEV), g.to(DEV))
        ref = parity.oracle_all(parity.rows2d(a), parity.rows2d(b), t.numpy(), g.numpy())
        parity.compare_all(got, ref, tag="split unaligned ")
    finally:
        vp.vp_set_row_split(old)


def test_split_against_one_cta_per_row_within_tolerance():
    w = workloads.pages_shape(seed=48, N=32, V=75968)
    a, b, t, g = (w[k].to(DEV) for k in ("a", "b", "targets", "grad"))
    old = vp.vp_get_row_split()
    try:
        vp.vp_set_row_split(1)
        one = parity.gpu_all(a, b, t, g)
        vp.vp_set_row_split(2)
        two = parity.gpu_all(a, b, t, g)
    finally:
        vp.vp_set_row_split(old)
    for k in ("logp", "H", "kl_rev", "kl_fwd"):
        x, y = parity.to64(one[k]), parity.to64(two[k])
        assert np.allclose(x, y, rtol=2e-6, atol=2e-6), k
    ref = oracle.entropy_fwd(parity.to64(w["a"]))[0]
    assert np.allclose(parity.to64(two["H"]), ref, rtol=2e-5, atol=2e-5)


def test_split_many_rows_per_cluster_against_oracle():
    # two CTAs per row and more than 32 rows per cluster (4999 rows over at most 152 clusters): the
    # finisher's batches roll over under the split too; sampled rows include every cluster's later rows
    old = vp.vp_get_row_split()
    vp.vp_set_row_split(2)
    try:
        N, V = 4999, 32768
        w = workloads.pages_shape(seed=72, N=N, V=V)
        t = w["targets"].clone()
        t[4900] = -1
        a, b, g = w["a"].to(DEV), w["b"].to(DEV), w["grad"].to(DEV)
        got = parity.gpu_all(a, b, t.to(DEV), g)
        rows = np.unique(np.concatenate([np.arange(0, 40), np.arange(4860, N), [1000, 2500, 4000]]))
        ref = parity.oracle_all(parity.to64(w["a"][rows]), parity.to64(w["b"][rows]), t[rows].numpy(),
                                w["grad"][rows].numpy())
        parity.compare_all(got, ref, rows=torch.as_tensor(rows, device=DEV), tag="split 4999 rows ")
    finally:
        vp.vp_set_row_split(old)
