"""GPU parity of the logprobs of several target ids per row (top-k) against the fp64 oracle.

Element by element: logp [N, K] (2e-5 + 2e-5 relative), the saved records'
exact maxima and log-sums, and the gradient dx [N, V] (one bf16 ulp plus the
fp32 evaluation term of the formula's operands, 1e-6 for fp32), on the pages'
recipe with ragged tails, K from 1 to past a warp, duplicate and ignored ids,
fully ignored rows, ids outside the shard, NaN / empty / -inf-target rows,
strided views and vocab_start; K = 1 against the single-target calls; batch
invariance.
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


def _mag(x64, t, g):
    """M_j: |g| summed over the row's used ids times p_j, plus |g| summed over the ids equal to j
    (the operands of the element's formula, for parity.KAPPA_BF16 and parity.ORACLE_EPS)."""
    N, V = x64.shape
    _, m, ls = oracle.entropy_fwd(x64)
    with np.errstate(all="ignore"):
        p = np.exp((x64 - m[:, None]) - ls[:, None])
    used = t >= 0
    gabs = np.where(used, np.abs(g), 0.0)
    M = p * gabs.sum(1)[:, None]
    for r in range(N):
        for k in np.nonzero(used[r])[0]:
            j = t[r, k]
            if 0 <= j < V:
                M[r, j] += gabs[r, k]
    return np.nan_to_num(M, nan=0.0, posinf=0.0)


def _check(x, t, g, tag, vocab_start=0):
    err = torch.zeros(1, dtype=torch.int32, device=x.device)
    lp, st = vp.vp_logprobs_topk_fwd(x, t, vocab_start, err_word=err)
    dx = vp.vp_logprobs_topk_bwd(x, t, st, g, vocab_start, err_word=err)
    torch.cuda.synchronize()
    x64 = parity.rows2d(x)
    t64 = t.cpu().numpy()
    g64 = g.cpu().double().numpy()
    rlp, rerr = oracle.logprobs_topk_fwd(x64, t64, vocab_start)
    rdx = oracle.logprobs_topk_bwd(x64, t64, g64, vocab_start)
    worst = {"logp": parity.check_out(lp, rlp, f"{tag} logp")}
    assert int(err.item()) == rerr, f"{tag} error word {int(err.item())} vs {rerr}"
    _, m, ls = oracle.entropy_fwd(x64)
    d = vp.decode_rowstats(st)
    ok = np.isfinite(m) & np.isfinite(ls) & ~(np.isnan(x64) | np.isposinf(x64)).any(1)   # rows with a record
    assert (parity.to64(d["m"])[ok] == m[ok]).all(), f"{tag} row max"
    parity.check_out(parity.to64(d["logS"])[ok], ls[ok], f"{tag} logS")
    M = _mag(x64, t64 - vocab_start * (t64 >= 0), g64)
    worst["dx"] = parity.check_grad(dx, rdx, f"{tag} dx", M, oracle_mag=M)
    return worst, (lp, st, dx)


SHAPES = [(37, 20011, torch.bfloat16), (33, 20011, torch.float32), (16, 75968, torch.bfloat16),
          (8, 1, torch.bfloat16), (9, 7, torch.float32), (5, 4101, torch.bfloat16), (3, 16392, torch.float32)]


@pytest.mark.parametrize("K", [1, 5, 33, 100])
@pytest.mark.parametrize("N,V,dtype", SHAPES, ids=[f"{n}x{v}-{str(d)[6:]}" for n, v, d in SHAPES])
def test_topk_pages_recipe(N, V, dtype, K):
    w = workloads.pages_shape(seed=N * 100 + V, N=N, V=V, dtype=dtype)
    ids = workloads.topk_ids(seed=N + V + K, N=N, V=V, K=K)
    worst, _ = _check(w["a"].to(DEV), ids["targets"].to(DEV), ids["grad"].to(DEV), f"{N}x{V} {dtype} K={K}")
    print("topk worst/tol:", {k: round(v, 3) for k, v in worst.items()})


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_topk_special_rows(dtype):
    V, K = 4103, 6
    gen = torch.Generator().manual_seed(13)
    x = torch.randn(10, V, generator=gen) * 2
    inf = float("inf")
    x[1, 100] = float("nan")              # NaN row
    x[2, :] = -inf                        # all -inf row
    x[3, ::3] = -inf                      # masked entries; an id on a -inf logit
    x[4, :] = -3e38                       # one-hot spanning +-3e38
    x[4, 17] = 3e38
    x[5] += 1e4 if dtype == torch.float32 else 100.0
    x[6, :] = 0.0                         # uniform row
    t = torch.randint(0, V, (10, K), generator=gen)
    t[0, :] = -1                          # fully ignored row
    t[3, 0] = 0                           # id on a -inf logit (logp = -inf, finite gradient)
    t[4, :] = 17                          # every id the same (duplicates add up)
    t[7, 2] = V + 5                       # id outside the shard: NaN, error bit
    t[8, 1:] = t[8, 0]                    # duplicates of one id
    t[9, ::2] = -1                        # some ignored
    t[1, 0] = -1                          # NaN row with an ignored id: that id gives 0
    g = torch.randn(10, K, generator=gen)
    worst, (lp, st, dx) = _check(x.to(dtype).to(DEV), t.to(DEV), g.to(DEV), f"special {dtype}")
    lp64, dx64 = parity.to64(lp), parity.to64(dx)
    assert (lp64[0] == 0).all() and (dx64[0] == 0).all()
    assert lp64[1, 0] == 0.0 and np.isnan(lp64[1, 1:]).all()
    assert np.isnan(dx64[7]).all() and np.isnan(lp64[7, 2])
    assert np.isneginf(lp64[3, 0])
    assert (dx64[4] == 0).all()           # one-hot row: p = onehot, G = Gsum at the single id


def test_topk_vocab_start_and_err_word():
    N, V, K, vs = 16, 3000, 7, 50000
    w = workloads.pages_shape(seed=9, N=N, V=V, dtype=torch.bfloat16)
    ids = workloads.topk_ids(seed=19, N=N, V=V, K=K, vocab_start=vs)
    t = ids["targets"]
    t[3, 1] = vs - 1          # below the shard
    t[4, 6] = vs + V          # past the shard
    _check(w["a"].to(DEV), t.to(DEV), ids["grad"].to(DEV), "vocab_start", vocab_start=vs)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_topk_strided_views(dtype):
    gen = torch.Generator().manual_seed(11)
    B, T, V, K = 3, 9, 4099, 9
    A = (torch.randn(B, T, V + 2, generator=gen) * 3).to(dtype).to(DEV)
    n = B * (T - 1)
    ids = workloads.topk_ids(seed=5, N=n, V=V, K=K)
    t, g = ids["targets"].to(DEV), ids["grad"].to(DEV)
    for name, a in (("causal slice", A[:, :-1, :V]), ("unaligned rows", A[:, 1:, 1:V + 1])):
        _check(a, t, g, f"{name} {dtype}")


def test_topk_k1_matches_single_target_calls():
    w = workloads.pages_shape(seed=41, N=64, V=20011, dtype=torch.bfloat16)
    x, t, g = w["a"].to(DEV), w["targets"].to(DEV), w["grad"].to(DEV)
    t[5] = -1
    lp1, st1 = vp.vp_logprobs_fwd(x, t)
    dx1 = vp.vp_logprobs_bwd(x, t, st1, g)
    lpk, stk = vp.vp_logprobs_topk_fwd(x, t[:, None].contiguous())
    dxk = vp.vp_logprobs_topk_bwd(x, t[:, None].contiguous(), stk, g[:, None].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(lp1, lpk[:, 0])
    d1, dk = vp.decode_rowstats(st1), vp.decode_rowstats(stk)
    assert torch.equal(d1["m"], dk["m"]) and torch.equal(d1["logS"], dk["logS"])
    assert torch.equal(dx1, dxk)


def test_topk_empty_batch_is_a_noop():
    x = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    t = torch.empty(0, 4, dtype=torch.int64, device=DEV)
    g = torch.empty(0, 4, dtype=torch.float32, device=DEV)
    lp, st = vp.vp_logprobs_topk_fwd(x, t)
    assert lp.shape == (0, 4)
    assert vp.vp_logprobs_topk_bwd(x, t, st, g).shape == (0, 128)
    torch.cuda.synchronize()


def _bits(v):
    return v.view(torch.int16 if v.dtype == torch.bfloat16 else torch.int32)


def test_topk_batch_invariance_bitwise():
    N, V, K = 512, 75968, 16
    w = workloads.pages_shape(seed=34, N=N, V=V, dtype=torch.bfloat16)
    ids = workloads.topk_ids(seed=35, N=N, V=V, K=K)
    x, t, g = w["a"].to(DEV), ids["targets"].to(DEV), ids["grad"].to(DEV)
    lp, st = vp.vp_logprobs_topk_fwd(x, t)
    dx = vp.vp_logprobs_topk_bwd(x, t, st, g)
    for lo, hi in ((0, 1), (5, 12), (300, 512), (511, 512)):
        lpp, stp = vp.vp_logprobs_topk_fwd(x[lo:hi], t[lo:hi])
        dxp = vp.vp_logprobs_topk_bwd(x[lo:hi], t[lo:hi], stp, g[lo:hi])
        assert torch.equal(_bits(lpp), _bits(lp[lo:hi])), f"logp rows {lo}:{hi}"
        assert torch.equal(_bits(dxp), _bits(dx[lo:hi])), f"dx rows {lo}:{hi}"


@pytest.mark.slow
def test_topk_full_pages_shape_sampled():
    """8192 x 75968 bf16, K = 20: sampled rows against the oracle, sum of dx per row on every row."""
    N, V, K = 8192, 75968, 20
    w = workloads.pages_shape(seed=1, N=N, V=V, dtype=torch.bfloat16)
    ids = workloads.topk_ids(seed=101, N=N, V=V, K=K)
    x, t, g = w["a"].to(DEV), ids["targets"].to(DEV), ids["grad"].to(DEV)
    lp, st = vp.vp_logprobs_topk_fwd(x, t)
    dx = vp.vp_logprobs_topk_bwd(x, t, st, g)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(7).choice(N, 48, replace=False))
    rows[-1] = N - 1
    x64 = parity.to64(w["a"][rows])
    t64, g64 = ids["targets"][rows].numpy(), ids["grad"][rows].double().numpy()
    rlp, _ = oracle.logprobs_topk_fwd(x64, t64)
    parity.check_out(lp[rows], rlp, "full topk logp")
    rdx = oracle.logprobs_topk_bwd(x64, t64, g64)
    M = _mag(x64, t64, g64)
    parity.check_grad(dx[rows], rdx, "full topk dx", M, oracle_mag=M)
    # every row: the gradient sums to ~0 (shift invariance), logp <= 0
    s = dx.float().sum(1).abs()
    assert float(s.max()) < 1e-2 * float(g.abs().sum(1).max())
    lpv = lp[t >= 0]
    assert bool((lpv <= 0).all())
