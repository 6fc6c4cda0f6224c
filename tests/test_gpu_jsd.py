"""GPU parity of the generalized JSD (interior beta, two passes) against the fp64 oracle.

Element by element: the per-row divergence (2e-5 + 2e-5 relative), the saved
records' exact maxima and log-sums, and both gradients (one bf16 ulp plus the
fp32 evaluation term of the formula's operands, 1e-6 for fp32), on the pages'
recipe with ragged tails, unaligned and strided rows, A and B that differ
modulo 16 bytes, NaN / empty / disjoint / +-3e38 rows and large offsets; the
beta = 0 / 1 endpoints as the KL calls; frozen inputs; batch invariance.
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


def _mags(a64, b64, beta, g):
    """M_j of the bf16 tolerance: |g| w p (|log p| + |log mix| + |KL(p||mix)| + 1), likewise for q."""
    _, ma, la = oracle.entropy_fwd(a64)
    _, mb, lb = oracle.entropy_fwd(b64)
    with np.errstate(all="ignore"):
        lp = (a64 - ma[:, None]) - la[:, None]
        lq = (b64 - mb[:, None]) - lb[:, None]
        p, q = np.exp(lp), np.exp(lq)
        lmix = np.log(beta * q + (1 - beta) * p)
        ka = np.sum(np.where(p > 0, p * (lp - lmix), 0.0), 1)
        kb = np.sum(np.where(q > 0, q * (lq - lmix), 0.0), 1)
        ag = np.abs(np.asarray(g, np.float64))[:, None]
        Ma = ag * (1 - beta) * p * (np.abs(lp) + np.abs(lmix) + np.abs(ka)[:, None] + 1.0)
        Mb = ag * beta * q * (np.abs(lq) + np.abs(lmix) + np.abs(kb)[:, None] + 1.0)
    return np.nan_to_num(Ma, nan=0.0, posinf=0.0), np.nan_to_num(Mb, nan=0.0, posinf=0.0), (ma, la), (mb, lb)


def _check(a, b, g, beta, tag, want=(True, True)):
    jsd, sa, sb = vp.vp_jsd_fwd(a, b, beta)
    da, db = vp.vp_jsd_bwd(a, b, beta, sa, sb, g, want_da=want[0], want_db=want[1])
    torch.cuda.synchronize()
    a64, b64 = parity.rows2d(a), parity.rows2d(b)
    g64 = g.cpu().double().numpy()
    ref = oracle.jsd_fwd(a64, b64, beta)
    rda, rdb = oracle.jsd_bwd(a64, b64, beta, g64)
    Ma, Mb, (ma, la), (mb, lb) = _mags(a64, b64, beta, g64)
    worst = {"jsd": parity.check_out(jsd, ref, f"{tag} jsd")}
    ok = ~np.isnan(ref)
    for name, st, m, ls in (("a", sa, ma, la), ("b", sb, mb, lb)):
        d = vp.decode_rowstats(st)
        m64 = parity.to64(d["m"])
        fin = ok & np.isfinite(m)
        assert (m64[fin] == m[fin]).all(), f"{tag} row max of {name}"
        parity.check_out(parity.to64(d["logS"])[ok], ls[ok], f"{tag} logS of {name}")
    if want[0]:
        worst["da"] = parity.check_grad(da, rda, f"{tag} dA", Ma, kappa=parity.KAPPA_JSD)
    else:
        assert da is None
    if want[1]:
        worst["db"] = parity.check_grad(db, rdb, f"{tag} dB", Mb, kappa=parity.KAPPA_JSD)
    else:
        assert db is None
    return worst, (jsd, sa, sb, da, db)


SHAPES = [(37, 20011, torch.bfloat16), (33, 20011, torch.float32), (16, 75968, torch.bfloat16),
          (8, 1, torch.bfloat16), (9, 7, torch.float32), (5, 4101, torch.bfloat16), (3, 16392, torch.bfloat16)]


@pytest.mark.parametrize("beta", [0.3, 0.5, 0.9])
@pytest.mark.parametrize("N,V,dtype", SHAPES, ids=[f"{n}x{v}-{str(d)[6:]}" for n, v, d in SHAPES])
def test_jsd_pages_recipe(N, V, dtype, beta):
    w = workloads.pages_shape(seed=N * 100 + V, N=N, V=V, dtype=dtype)
    worst, _ = _check(w["a"].to(DEV), w["b"].to(DEV), w["grad"].to(DEV), beta, f"{N}x{V} {dtype} beta={beta}")
    print("jsd worst/tol:", {k: round(v, 3) for k, v in worst.items()})


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_jsd_peaked_rows_late_chunks(dtype):
    # one logit 18 to 24 above N(0, 1) rows past the first 8192 columns, at different columns in A and B
    # (each distribution's mode lies in the other's far tail, the mixture's log there near log(1 - beta))
    gen = torch.Generator().manual_seed(75)
    N, V = 48, 75968
    a = torch.randn(N, V, generator=gen)
    b = torch.randn(N, V, generator=gen)
    a[torch.arange(N), torch.randint(8192, V, (N,), generator=gen)] += 18.0 + 6.0 * torch.rand(N, generator=gen)
    b[torch.arange(N), torch.randint(8192, V, (N,), generator=gen)] += 18.0 + 6.0 * torch.rand(N, generator=gen)
    g = torch.randn(N, generator=gen) * 2.0
    for beta in (0.3, 0.9):
        _check(a.to(dtype).to(DEV), b.to(dtype).to(DEV), g.to(DEV), beta, f"late peaks {dtype} beta={beta}")


def test_jsd_special_rows():
    N, V = 10, 3001
    for dtype in (torch.bfloat16, torch.float32):
        w = workloads.pages_shape(seed=77, N=N, V=V, dtype=torch.float32)
        a, b, g = w["a"], w["b"], w["grad"]
        a[0, 17] = float("nan")                  # NaN in A
        b[1, 3] = float("inf")                   # +inf in B
        a[2] = float("-inf")                     # no finite logit in A
        a[3, V // 2:] = float("-inf")            # disjoint supports
        b[3, :V // 2] = float("-inf")
        a[4] = -3e38                              # one-hot rows spanning +-3e38
        a[4, 9] = 3e38
        b[4] = a[4]
        a[5] += 1e4 if dtype == torch.float32 else 250.0   # large offsets
        b[5] -= 1e4 if dtype == torch.float32 else 250.0
        b[6, ::3] = float("-inf")                # B masked on a third of the row
        a, b = a.to(dtype).to(DEV), b.to(dtype).to(DEV)
        _, (jsd, *_rest) = _check(a, b, g.to(DEV), 0.4, f"special {dtype}")
        j = jsd.cpu().double().numpy()
        assert np.isnan(j[:3]).all() and np.isfinite(j[3:]).all()
        hb = -0.4 * np.log(0.4) - 0.6 * np.log(0.6)
        assert abs(j[3] - hb) <= 2e-5 * (1 + hb)            # disjoint supports: H(beta)
        assert abs(j[4]) <= 2e-5                             # identical one-hot rows: 0


def test_jsd_strided_unaligned_and_misaligned_pair():
    B_, T, V = 3, 9, 5003
    g = torch.Generator().manual_seed(5)
    base_a = (torch.randn(B_, T + 1, V + 1, generator=g) * 3).to(torch.bfloat16).to(DEV)
    base_b = (torch.randn(B_, T + 1, V + 2, generator=g) * 3).to(torch.bfloat16).to(DEV)
    grad = torch.randn(B_ * T, generator=g).to(DEV)
    a = base_a[:, :-1, 1:]                       # strided rows, 2-byte offset
    b = base_b[:, :-1, 2:V + 2]
    # same layout is required of A and B: copy B into A's layout at another 16-byte phase
    b_same = torch.empty_like(base_a)[:, :-1, 1:]
    b_same.copy_(b)
    _check(a, b_same, grad, 0.25, "strided")
    # A and B differing modulo 16 bytes: the element-wise second pass
    holder = torch.empty(B_ * T * V + 8, dtype=torch.bfloat16, device=DEV)
    a2 = a.reshape(-1, V).contiguous()
    b2 = holder[3:3 + B_ * T * V].view(B_ * T, V)
    b2.copy_(b.reshape(-1, V))
    assert (a2.data_ptr() ^ b2.data_ptr()) & 15
    with pytest.raises(vp.VPError):
        vp.vp_jsd_fwd(a2, b2[:, :V - 1], 0.25)   # shapes must match
    # same shape and strides, different phase
    _check(a2, b2, grad, 0.25, "pair misaligned")


def test_jsd_endpoints_are_the_kl_calls_and_frozen_inputs():
    w = workloads.pages_shape(seed=8, N=12, V=9000)
    a, b, g = w["a"].to(DEV), w["b"].to(DEV), w["grad"].to(DEV)
    for beta, d in ((0.0, vp.KL_FORWARD), (1.0, vp.KL_REVERSE)):
        j, sa, sb = vp.vp_jsd_fwd(a, b, beta)
        k, ka, kb = vp.vp_kl_fwd(a, b, d)
        assert torch.equal(j, k) and torch.equal(sa, ka) and torch.equal(sb, kb)
        assert all(torch.equal(x, y) for x, y in zip(vp.vp_jsd_bwd(a, b, beta, sa, sb, g), vp.vp_kl_bwd(a, b, d, ka, kb, g)))
    # frozen teacher / student: the other gradient is bitwise the same as with both
    _, (j, sa, sb, da, db) = _check(a, b, g, 0.6, "both")
    da1, none = vp.vp_jsd_bwd(a, b, 0.6, sa, sb, g, want_db=False)
    none2, db1 = vp.vp_jsd_bwd(a, b, 0.6, sa, sb, g, want_da=False)
    assert none is None and none2 is None and torch.equal(da1, da) and torch.equal(db1, db)
    with pytest.raises(vp.VPError):
        vp.vp_jsd_fwd(a, b, 1.5)
    with pytest.raises(vp.VPError):
        vp.vp_jsd_fwd(a, b, float("nan"))


def test_jsd_batch_invariance():
    w = workloads.pages_shape(seed=9, N=64, V=20011)
    a, b, g = w["a"].to(DEV), w["b"].to(DEV), w["grad"].to(DEV)
    j, sa, sb = vp.vp_jsd_fwd(a, b, 0.3)
    da, db = vp.vp_jsd_bwd(a, b, 0.3, sa, sb, g)
    j2, sa2, sb2 = vp.vp_jsd_fwd(a[20:23], b[20:23], 0.3)
    da2, db2 = vp.vp_jsd_bwd(a[20:23], b[20:23], 0.3, sa2, sb2, g[20:23])
    torch.cuda.synchronize()
    assert torch.equal(j[20:23].view(torch.int32), j2.view(torch.int32))
    assert torch.equal(sa[20:23], sa2) and torch.equal(da[20:23], da2) and torch.equal(db[20:23], db2)
