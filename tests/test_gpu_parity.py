"""GPU parity: libvp (through the C ABI) against the fp64 oracle, element by element.

Covers the five workloads' recipes at oracle-sized shapes (several vector
iterations per thread and ragged tails), unaligned and strided rows read in
place, every special row of the readings, the device error word, N = 0, batch
invariance (bitwise), and the full-size workloads on sampled rows plus
properties that hold on every row.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import vocab_wide_logprobs_gb300 as vp
from vocab_wide_logprobs_gb300 import workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"
ALL = ("logprobs", "entropy", "kl_rev", "kl_fwd")


def _run_and_compare(a, b, targets, grad, ops=ALL, vocab_start=0, tag=""):
    got = parity.gpu_all(a, b, targets, grad, ops, vocab_start)
    ref = parity.oracle_all(parity.rows2d(a), parity.rows2d(b), targets.cpu().numpy(), grad.cpu().numpy(),
                            ops, vocab_start)
    worst = parity.compare_all(got, ref, tag=tag)
    if "logprobs" in ops:
        assert int(got["err"].item()) == ref["err"], f"{tag}err word"
    return got, ref, worst


def test_tiny_config_all_ops():
    w = workloads.tiny()
    a, b = w["a"].to(DEV), w["b"].to(DEV)
    _, ref, worst = _run_and_compare(a, b, w["targets"].to(DEV), w["grad"].to(DEV), tag="tiny ")
    # 4 rows of B are masked: forward KL(B||A) stays finite; reverse KL(A||B) is flagged there
    rows = w["masked_rows"].numpy()
    assert np.isinf(ref["kl_rev"][rows]).all() and np.isfinite(ref["kl_fwd"]).all()
    print("tiny worst/tol:", {k: round(v, 3) for k, v in worst.items()})


SHAPES = [
    (48, 75968, torch.bfloat16), (37, 20011, torch.bfloat16), (33, 20011, torch.float32),
    (16, 75968, torch.float32), (8, 1, torch.bfloat16), (8, 1, torch.float32), (8, 2, torch.bfloat16),
    (8, 3, torch.float32), (9, 7, torch.bfloat16), (9, 9, torch.bfloat16), (5, 31, torch.float32),
    (5, 4101, torch.bfloat16), (3, 16385, torch.float32), (3, 16392, torch.bfloat16),
]


@pytest.mark.parametrize("N,V,dtype", SHAPES, ids=[f"{n}x{v}-{str(d)[6:]}" for n, v, d in SHAPES])
def test_pages_recipe_shapes(N, V, dtype):
    w = workloads.pages_shape(seed=N * 1000 + V, N=N, V=V, dtype=dtype)
    _run_and_compare(w["a"].to(DEV), w["b"].to(DEV), w["targets"].to(DEV), w["grad"].to(DEV),
                     tag=f"{N}x{V} {dtype} ")


def test_large_offset_fp32_with_masks():
    w = workloads.numerics_stress(seed=5, N=24, V=20011)
    _, ref, _ = _run_and_compare(w["a"].to(DEV), w["b"].to(DEV), w["targets"].to(DEV), w["grad"].to(DEV),
                                 tag="offset 1e4 ")
    assert np.isinf(ref["kl_rev"]).all() and np.isfinite(ref["kl_fwd"]).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_strided_and_unaligned_views(dtype):
    gen = torch.Generator().manual_seed(11)
    B, T, V = 3, 9, 4099
    A = (torch.randn(B, T, V + 2, generator=gen) * 3).to(dtype).to(DEV)
    Bt = (torch.randn(B, T, V + 2, generator=gen) * 3).to(dtype).to(DEV)
    tg = torch.randint(0, V, (B * (T - 1),), generator=gen).to(DEV)
    g = torch.randn(B * (T - 1), generator=gen).to(DEV)
    views = {
        "causal slice [:, :-1]": (A[:, :-1, :V], Bt[:, :-1, :V]),
        "shifted rows [:, 1:]": (A[:, 1:, 1:V + 1], Bt[:, 1:, 1:V + 1]),       # unaligned row starts
        "different phases": (A[:, :-1, 1:V + 1], Bt[:, :-1, 2:V + 2]),        # A and B differ mod 16
        "2-D row stride": (A[0, :-1, :V], Bt[0, :-1, :V]),
    }
    for name, (a, b) in views.items():
        n = a.shape[0] * a.shape[1] if a.dim() == 3 else a.shape[0]
        _run_and_compare(a, b, tg[:n], g[:n], tag=f"{name} ")


def _special_rows(dtype):
    V = 4103
    gen = torch.Generator().manual_seed(3)
    base = torch.randn(14, V, generator=gen) * 2
    a, b = base.clone(), (torch.randn(14, V, generator=gen) * 2)
    inf = float("inf")
    a[1, 100] = float("nan")             # NaN in A
    a[2, 4000] = inf                     # +inf in A
    a[3, :] = -inf                       # all -inf A row
    a[4, ::3] = -inf                     # masked entries in A (finite results)
    a[5, :] = -3e38                      # one-hot spanning +-3e38
    a[5, 17] = 3e38
    b[5] = a[5]
    b[6, 9] = -inf                       # mismatch for KL(A||B)
    a[7, 0] = -1000.0                    # A's probability underflows where B masks it
    b[7, 0] = -inf
    a[8, 5:] = -inf                      # both masked at the same places
    b[8, 5:] = -inf
    b[9, :] = -inf                       # all -inf B row
    a[10] += 1e4 if dtype == torch.float32 else 100.0   # large common offset
    b[10] -= 1e4 if dtype == torch.float32 else 100.0
    a[11, :] = 0.0                       # uniform row
    b[11, :] = 7.0
    a[12, 2] = float("nan")              # NaN together with a mismatch: NaN wins
    b[12, 3] = -inf
    b[13, 20] = float("nan")             # NaN in B only
    tg = torch.randint(0, V, (14,), generator=gen)
    tg[0] = -1                           # ignored
    tg[4] = 0                            # a target on a -inf logit
    tg[6] = V + 5                        # out of range (data error)
    return a.to(dtype), b.to(dtype), tg, torch.randn(14, generator=gen)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_special_rows(dtype):
    a, b, tg, g = _special_rows(dtype)
    got, ref, _ = _run_and_compare(a.to(DEV), b.to(DEV), tg.to(DEV), g.to(DEV), tag=f"special {dtype} ")
    assert ref["err"] == 1 and int(got["err"].item()) == 1
    H = parity.to64(got["H"])
    assert H[5] == 0.0 and abs(H[11] - math.log(a.shape[1])) < 1e-5
    assert parity.to64(got["kl_rev"])[5] == 0.0
    assert (parity.to64(got["dH"][5]) == 0).all() and (parity.to64(got["dkl_rev_a"][5]) == 0).all()
    assert parity.to64(got["logp"])[0] == 0.0 and (parity.to64(got["dlogp"][0]) == 0).all()


def test_vocab_start_and_err_word():
    w = workloads.pages_shape(seed=9, N=16, V=3000, dtype=torch.bfloat16)
    t = w["targets"] + 50000
    t[3] = 50000 - 1          # below the shard
    t[4] = 50000 + 3000       # past the shard
    t[5] = -7                 # ignored
    _run_and_compare(w["a"].to(DEV), w["b"].to(DEV), t.to(DEV), w["grad"].to(DEV), ops=("logprobs",),
                     vocab_start=50000, tag="vocab_start ")


def test_empty_batch_is_a_noop():
    x = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    t = torch.empty(0, dtype=torch.int64, device=DEV)
    g = torch.empty(0, dtype=torch.float32, device=DEV)
    lp, st = vp.vp_logprobs_fwd(x, t)
    assert lp.numel() == 0
    assert vp.vp_logprobs_bwd(x, t, st, g).shape == (0, 128)
    H, st = vp.vp_entropy_fwd(x)
    vp.vp_entropy_bwd(x, st, g)
    kl, sa, sb = vp.vp_kl_fwd(x, x)
    vp.vp_kl_bwd(x, x, vp.KL_REVERSE, sa, sb, g)
    torch.cuda.synchronize()


def test_kl_single_gradient_outputs():
    w = workloads.pages_shape(seed=21, N=12, V=9000, dtype=torch.bfloat16)
    a, b, g = w["a"].to(DEV), w["b"].to(DEV), w["grad"].to(DEV)
    for d in (vp.KL_REVERSE, vp.KL_FORWARD):
        kl, sa, sb = vp.vp_kl_fwd(a, b, d)
        da_both, db_both = vp.vp_kl_bwd(a, b, d, sa, sb, g)
        da, none_b = vp.vp_kl_bwd(a, b, d, sa, sb, g, want_db=False)
        none_a, db = vp.vp_kl_bwd(a, b, d, sa, sb, g, want_da=False)
        torch.cuda.synchronize()
        assert none_a is None and none_b is None
        assert torch.equal(da, da_both) and torch.equal(db, db_both)


def _bits(v):
    return v.view(torch.int16 if v.dtype == torch.bfloat16 else torch.int32)


def test_batch_invariance_bitwise():
    w = workloads.pages_shape(seed=33, N=1024, V=75968, dtype=torch.bfloat16)
    a, b, t, g = (w[k].to(DEV) for k in ("a", "b", "targets", "grad"))
    full = parity.gpu_all(a, b, t, g)
    for lo, hi in ((0, 1), (0, 7), (5, 12), (300, 1024), (1023, 1024)):
        part = parity.gpu_all(a[lo:hi], b[lo:hi], t[lo:hi], g[lo:hi])
        for k, v in part.items():
            if k == "err":
                continue
            assert torch.equal(_bits(v), _bits(full[k][lo:hi])), f"{k} rows {lo}:{hi} differ bitwise"


# ---------------------------------------------------------------------------
# Full-size workloads: sampled rows against the oracle, properties on every row
# ---------------------------------------------------------------------------
def _properties(got, V, grads=True):
    logV = math.log(V)
    if "H" in got:
        H = got["H"]
        fin = torch.isfinite(H)
        assert (H[fin] >= -1e-5).all() and (H[fin] <= logV + 1e-4).all(), "0 <= H <= log V"
    for k in ("kl_rev", "kl_fwd"):
        if k in got:
            kl = got[k]
            assert (kl[torch.isfinite(kl)] >= -1e-4).all(), "KL >= 0"
    if "logp" in got:
        lp = got["logp"]
        assert (lp[torch.isfinite(lp)] <= 1e-6).all(), "logp <= 0"
    if grads:
        for k, d in got.items():
            if not k.startswith("d"):
                continue
            d32 = d.float()
            ok = torch.isfinite(d32).all(dim=1)
            s = d32[ok].double().sum(1).abs()
            scale = d32[ok].double().abs().sum(1)
            tol = (2.0 ** -8 if d.dtype == torch.bfloat16 else 1e-5) * scale + 1e-6
            assert (s <= tol).all(), f"{k}: rows do not sum to 0"


def _sampled(n, N, seed):
    rng = np.random.default_rng(seed)
    return np.sort(np.concatenate([[0, N - 1], rng.choice(np.arange(1, N - 1), n - 2, replace=False)]))


@pytest.mark.slow
def test_full_pages_shape_sampled():
    w = workloads.pages_shape()
    a, b, t, g = (w[k].to(DEV) for k in ("a", "b", "targets", "grad"))
    got = parity.gpu_all(a, b, t, g)
    _properties(got, a.shape[1])
    rows = _sampled(24, a.shape[0], 1)
    ref = parity.oracle_all(parity.to64(w["a"][rows]), parity.to64(w["b"][rows]), w["targets"][rows].numpy(),
                            w["grad"][rows].numpy())
    parity.compare_all(got, ref, rows=torch.as_tensor(rows, device=DEV), tag="config 2 ")


@pytest.mark.slow
def test_full_numerics_stress_sampled():
    w = workloads.numerics_stress()
    a, b, t, g = (w[k].to(DEV) for k in ("a", "b", "targets", "grad"))
    ops = ("entropy", "kl_rev", "kl_fwd")
    got = parity.gpu_all(a, b, t, g, ops)
    _properties(got, a.shape[1])
    assert torch.isinf(got["kl_rev"]).all() and torch.isfinite(got["kl_fwd"]).all()
    rows = _sampled(16, a.shape[0], 2)
    ref = parity.oracle_all(parity.to64(w["a"][rows]), parity.to64(w["b"][rows]), w["targets"][rows].numpy(),
                            w["grad"][rows].numpy(), ops)
    parity.compare_all(got, ref, rows=torch.as_tensor(rows, device=DEV), tag="config 3 ")


@pytest.mark.slow
def test_full_strided_sampled():
    w = workloads.strided()
    A, B = w["a_full"].to(DEV), w["b_full"].to(DEV)
    a, b = A[:, :-1], B[:, :-1]
    t, g = w["targets"].reshape(-1).to(DEV), w["grad"].reshape(-1).to(DEV)
    got = parity.gpu_all(a, b, t, g)
    _properties(got, a.shape[-1])
    rows = _sampled(16, a.shape[0] * a.shape[1], 3)
    a2d = w["a_full"][:, :-1].reshape(-1, a.shape[-1])
    b2d = w["b_full"][:, :-1].reshape(-1, a.shape[-1])
    ref = parity.oracle_all(parity.to64(a2d[rows]), parity.to64(b2d[rows]), w["targets"].reshape(-1)[rows].numpy(),
                            w["grad"].reshape(-1)[rows].numpy())
    parity.compare_all(got, ref, rows=torch.as_tensor(rows, device=DEV), tag="config 4 ")
    # reading in place equals reading a contiguous copy, bitwise
    got_c = parity.gpu_all(a.contiguous(), b.contiguous(), t, g)
    for k, v in got.items():
        if k != "err":
            assert torch.equal(_bits(v), _bits(got_c[k])), k


@pytest.mark.slow
def test_short_rows_sampled():
    w = workloads.short_rows()
    a, b, t, g = (w[k].to(DEV) for k in ("a", "b", "targets", "grad"))
    got = parity.gpu_all(a, b, t, g)
    _properties(got, a.shape[1])
    rows = _sampled(96, a.shape[0], 4)
    ref = parity.oracle_all(parity.to64(w["a"][rows]), parity.to64(w["b"][rows]), w["targets"][rows].numpy(),
                            w["grad"][rows].numpy())
    parity.compare_all(got, ref, rows=torch.as_tensor(rows, device=DEV), tag="N=1024 ")


def test_zz_report_error_stats():
    """Prints the worst error / tolerance seen by the parity tests above (informational)."""
    for k, v in sorted(parity.STATS.items()):
        print(k, v)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_many_rows_per_cta(dtype):
    # more rows than 32 per persistent CTA (20011 rows, at most 304 CTAs): the forward finisher's batches
    # of 32 rows roll over, with the next batch's target ids and target logits read a batch ahead
    N, V = 20011, 1537
    w = workloads.pages_shape(seed=71, N=N, V=V, dtype=dtype)
    t = w["targets"].clone()
    t[::97] = -1                     # ignored
    t[5::1301] = V + 3               # outside the shard: NaN rows and the error bit
    a, b = w["a"].to(DEV), w["b"].to(DEV)
    _run_and_compare(a, b, t.to(DEV), w["grad"].to(DEV), tag=f"{N} rows {dtype} ")
    if dtype != torch.bfloat16:
        return
    a64, b64 = parity.rows2d(a), parity.rows2d(b)
    # the JSD's statistics-only first pass and the shard records take the same batched finisher
    j, _, _ = vp.vp_jsd_fwd(a, b, 0.3)
    parity.check_out(j, oracle.jsd_fwd(a64, b64, 0.3), f"{N} rows jsd")
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp, _ = vp.vp_logprobs_merge(vp.vp_logprobs_partial(a, t.to(DEV))[None], err_word=err)
    ref_lp, _, _, ref_err = oracle.logprobs_fwd(a64, t.numpy())
    parity.check_out(lp, ref_lp, f"{N} rows logprobs via shard records")
    torch.cuda.synchronize()
    assert int(err.item()) == ref_err


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_peaked_rows(dtype):
    # one logit 12 above the rest in every row (p near 1), at different columns in A and B, so that P's
    # mode lies far down in Q (a large KL and a large centred mean c); targets at the peak or elsewhere,
    # upstream gradients of a few units: the fp32 sums of such rows are dominated by one term
    N, V = 512, 3001
    gen = torch.Generator().manual_seed(73)
    a = torch.randn(N, V, generator=gen) * 3
    b = torch.randn(N, V, generator=gen) * 3
    pa = torch.randint(0, V, (N,), generator=gen)
    pb = torch.randint(0, V, (N,), generator=gen)
    a[torch.arange(N), pa] += 12.0 + 4.0 * torch.rand(N, generator=gen)
    b[torch.arange(N), pb] += 12.0 + 4.0 * torch.rand(N, generator=gen)
    t = torch.where(torch.rand(N, generator=gen) < 0.5, pa, torch.randint(0, V, (N,), generator=gen))
    g = torch.randn(N, generator=gen) * 2.0
    _run_and_compare(a.to(dtype).to(DEV), b.to(dtype).to(DEV), t.to(DEV), g.to(DEV), tag=f"peaked {dtype} ")


def _late_peaks(seed, N, V):
    # N(0, 1) rows with one logit 18 to 24 higher past the first 8192 columns, at different columns in A
    # and B; half the targets at A's peak; upstream gradients of a few units
    gen = torch.Generator().manual_seed(seed)
    a = torch.randn(N, V, generator=gen)
    b = torch.randn(N, V, generator=gen)
    pa = torch.randint(8192, V, (N,), generator=gen)
    pb = torch.randint(8192, V, (N,), generator=gen)
    a[torch.arange(N), pa] += 18.0 + 6.0 * torch.rand(N, generator=gen)
    b[torch.arange(N), pb] += 18.0 + 6.0 * torch.rand(N, generator=gen)
    t = torch.where(torch.rand(N, generator=gen) < 0.5, pa, torch.randint(0, V, (N,), generator=gen))
    return a, b, t, torch.randn(N, generator=gen) * 2.0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_peaked_rows_late_chunks(dtype):
    # rows of many ring stages: each warp centres its sums on its own largest value of the first stage, so
    # a peak that arrives in a later stage sits ~20 above the centre, and the sums' terms near it (e and
    # e t) are 20 units' worth of exponent and distance large: a plain fp32 running sum of them would
    # leave W/S about 2^-24 times that distance off, which the gradients at the peak (p near 1) resolve
    a, b, t, g = _late_peaks(74, 96, 75968)
    _run_and_compare(a.to(dtype).to(DEV), b.to(dtype).to(DEV), t.to(DEV), g.to(DEV), tag=f"late peaks {dtype} ")
