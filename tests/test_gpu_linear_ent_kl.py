"""GPU parity of the fused linear entropy and the fused linear KL of two models (tcgen05 path)
against the fp64 oracle.

Forward outputs (H, KL) at 2e-5 + 2e-5 relative, the records' maxima and log-sums
likewise (fp32 accumulations against fp64 logits); gradients (dhidden, dW of each
model) at one bf16 ulp plus the forward error bound of a GEMM with bf16-rounded
dz (parity.check_gemm_grad). Shapes span several 128-row and 256-column tiles
with ragged edges, several backward vocabulary chunks, models of different
hidden sizes, both KL directions, a frozen model, a model compared with itself
(exactly 0) and batch invariance.
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


def _model(seed, N, V, D, scale=25.0):
    """hidden ~ N(0, 1), head ~ N(0, (0.02 scale)^2): logits with a spread of several units."""
    w = workloads.linear(seed=seed, N=N, V=V, D=D)
    return w["hidden"], (w["weight"].float() * scale).to(torch.bfloat16), w["grad"]


# ---------------------------------------------------------------------------
# Entropy
# ---------------------------------------------------------------------------
ENT_SHAPES = [(256, 1024, 256), (200, 777, 128), (130, 300, 64), (64, 4096, 1024), (72, 70000, 64)]


@pytest.mark.parametrize("N,V,D", ENT_SHAPES)
def test_linear_entropy_fwd_bwd(N, V, D):
    h, W, g = _model(N + 3 * V + D, N, V, D)
    hd, Wd, gd = h.to(DEV), W.to(DEV), g.to(DEV)
    H, st = vp.vp_linear_entropy_fwd(hd, Wd)
    dh, dW = vp.vp_linear_entropy_bwd(hd, Wd, st, gd)
    torch.cuda.synchronize()
    h64, W64, g64 = parity.to64(h), parity.to64(W), g.double().numpy()
    rH, rm, rls = oracle.linear_entropy_fwd(h64, W64)
    parity.check_out(H, rH, f"{N}x{V}x{D} H")
    d = vp.decode_rowstats(st)
    parity.check_out(d["m"], rm, f"{N}x{V}x{D} max logit")
    parity.check_out(d["logS"], rls, f"{N}x{V}x{D} logS")
    rdh, rdW = oracle.linear_entropy_bwd(h64, W64, g64)
    z = oracle.linear_logits(h64, W64)
    dz = np.abs(oracle.entropy_bwd(z, g64))
    M = parity.oracle_all(z, z, np.zeros(N, np.int64), g64, ops=("entropy",))["_mag"]["dH"]
    M = M * (1.0 + parity.logit_scale((h64, W64)))[:, None]
    parity.check_gemm_grad(dh, rdh, parity.gemm_norms(dz, W64), f"{N}x{V}x{D} entropy dhidden", M @ np.abs(W64))
    parity.check_gemm_grad(dW, rdW, parity.gemm_norms(dz.T, h64), f"{N}x{V}x{D} entropy dW", M.T @ np.abs(h64))


def test_linear_entropy_single_outputs_and_batch_invariance():
    N, V, D = 384, 2000, 256
    h, W, g = (t.to(DEV) for t in _model(7, N, V, D))
    H, st = vp.vp_linear_entropy_fwd(h, W)
    dh, dW = vp.vp_linear_entropy_bwd(h, W, st, g)
    dh_only, none_w = vp.vp_linear_entropy_bwd(h, W, st, g, want_dW=False)
    none_h, dW_only = vp.vp_linear_entropy_bwd(h, W, st, g, want_dhidden=False)
    part, _ = vp.vp_linear_entropy_fwd(h[128:256].contiguous(), W)
    torch.cuda.synchronize()
    assert none_w is None and none_h is None
    assert torch.equal(dh_only, dh) and torch.equal(dW_only, dW)
    assert torch.equal(H[128:256].view(torch.int32), part.view(torch.int32))


def test_linear_entropy_zero_head_is_uniform():
    N, V, D = 130, 1000, 128
    h = _model(8, N, V, D)[0].to(DEV)
    W = torch.zeros(V, D, dtype=torch.bfloat16, device=DEV)
    g = torch.randn(N, generator=torch.Generator().manual_seed(8)).to(DEV)
    H, st = vp.vp_linear_entropy_fwd(h, W)
    dh, dW = vp.vp_linear_entropy_bwd(h, W, st, g)
    torch.cuda.synchronize()
    parity.check_out(H, np.full(N, np.log(V)), "zero head H")
    assert (dh == 0).all() and (dW == 0).all()


# ---------------------------------------------------------------------------
# KL of two models
# ---------------------------------------------------------------------------
KL_SHAPES = [(256, 1024, 256, 128), (200, 777, 128, 192), (130, 300, 64, 64), (72, 70000, 64, 128)]


def _kl_case(N, V, Da, Db, seed):
    ha, Wa, g = _model(seed, N, V, Da)
    hb, Wb, _ = _model(seed + 1, N, V, Db, scale=20.0)
    return ha, Wa, hb, Wb, g


def _check_kl(ha, Wa, hb, Wb, g, direction, tag):
    dev = [t.to(DEV) for t in (ha, Wa, hb, Wb, g)]
    kl, sa, sb = vp.vp_linear_kl_fwd(*dev[:4], direction)
    grads = vp.vp_linear_kl_bwd(*dev[:4], direction, sa, sb, dev[4])
    torch.cuda.synchronize()
    ha64, Wa64, hb64, Wb64 = (parity.to64(t) for t in (ha, Wa, hb, Wb))
    g64 = g.double().numpy()
    rkl, rma, rla, rmb, rlb = oracle.linear_kl_fwd(ha64, Wa64, hb64, Wb64, direction)
    parity.check_out(kl, rkl, f"{tag} KL")
    for st, rm, rl, name in ((sa, rma, rla, "A"), (sb, rmb, rlb, "B")):
        d = vp.decode_rowstats(st)
        parity.check_out(d["m"], rm, f"{tag} max logit of {name}")
        parity.check_out(d["logS"], rl, f"{tag} logS of {name}")
    ref = oracle.linear_kl_bwd(ha64, Wa64, hb64, Wb64, g64, direction)
    za, zb = oracle.linear_logits(ha64, Wa64), oracle.linear_logits(hb64, Wb64)
    dza, dzb = (np.abs(x) for x in oracle.kl_bwd(za, zb, g64, direction))
    op = "kl_rev" if direction == vp.KL_REVERSE else "kl_fwd"
    M = parity.oracle_all(za, zb, np.zeros(za.shape[0], np.int64), g64, ops=(op,))["_mag"]
    Ma, Mb = M["d" + op + "_a"], M["d" + op + "_b"]
    pa, pb = _probs(za), _probs(zb)
    pP = pa if direction == vp.KL_REVERSE else pb
    Fa, Fb = parity.flushed(Ma, pP, pa, pb), parity.flushed(Mb, pP, pa, pb)
    lam = (1.0 + parity.logit_scale((ha64, Wa64), (hb64, Wb64)))[:, None]
    Ma, Mb = Ma * lam, Mb * lam
    norms = (parity.gemm_norms(dza, Wa64), parity.gemm_norms(dza.T, ha64), parity.gemm_norms(dzb, Wb64),
             parity.gemm_norms(dzb.T, hb64))
    evals = (Ma @ np.abs(Wa64), Ma.T @ np.abs(ha64), Mb @ np.abs(Wb64), Mb.T @ np.abs(hb64))
    flush = (Fa @ np.abs(Wa64), Fa.T @ np.abs(ha64), Fb @ np.abs(Wb64), Fb.T @ np.abs(hb64))
    for got, r, nm, ev, fl, name in zip(grads, ref, norms, evals, flush, ("dhidden A", "dW A", "dhidden B", "dW B")):
        parity.check_gemm_grad(got, r, nm, f"{tag} {name}", ev, fl)
    return kl, grads


def _probs(z):
    """softmax of fp64 logits, row by row."""
    e = np.exp(z - z.max(1, keepdims=True))
    return e / e.sum(1, keepdims=True)


@pytest.mark.parametrize("direction", [vp.KL_REVERSE, vp.KL_FORWARD], ids=["reverse", "forward"])
@pytest.mark.parametrize("N,V,Da,Db", KL_SHAPES)
def test_linear_kl_fwd_bwd(N, V, Da, Db, direction):
    _check_kl(*_kl_case(N, V, Da, Db, seed=N + V + Da + Db), direction, f"{N}x{V} Da={Da} Db={Db} dir={direction}")


def test_linear_kl_close_models():
    """A student close to its teacher: small KL, cancellation in the W sums."""
    N, V, D = 192, 3000, 128
    ha, Wa, g = _model(31, N, V, D)
    gen = torch.Generator().manual_seed(32)
    Wb = (Wa.float() + 0.01 * torch.randn(V, D, generator=gen)).to(torch.bfloat16)
    hb = (ha.float() + 0.01 * torch.randn(N, D, generator=gen)).to(torch.bfloat16)
    for d in (vp.KL_REVERSE, vp.KL_FORWARD):
        kl, _ = _check_kl(ha, Wa, hb, Wb, g, d, f"close models dir={d}")
        assert float(kl.max()) < 0.05


def test_linear_kl_model_with_itself_and_frozen_teacher():
    N, V, Da, Db = 136, 1500, 128, 64
    ha, Wa, hb, Wb, g = (t.to(DEV) for t in _kl_case(N, V, Da, Db, seed=41))
    for d in (vp.KL_REVERSE, vp.KL_FORWARD):
        kl, sa, sb = vp.vp_linear_kl_fwd(ha, Wa, ha, Wa, d)
        zero = vp.vp_linear_kl_bwd(ha, Wa, ha, Wa, d, sa, sb, g)
        torch.cuda.synchronize()
        assert (kl == 0).all(), "KL of a model with itself"
        assert all((z == 0).all() for z in zero)
        kl, sa, sb = vp.vp_linear_kl_fwd(ha, Wa, hb, Wb, d)
        full = vp.vp_linear_kl_bwd(ha, Wa, hb, Wb, d, sa, sb, g)
        student = vp.vp_linear_kl_bwd(ha, Wa, hb, Wb, d, sa, sb, g, want=(True, True, False, False))
        head_b = vp.vp_linear_kl_bwd(ha, Wa, hb, Wb, d, sa, sb, g, want=(False, False, False, True))
        torch.cuda.synchronize()
        assert student[2] is None and student[3] is None and head_b[0] is None
        assert torch.equal(student[0], full[0]) and torch.equal(student[1], full[1])
        assert torch.equal(head_b[3], full[3])


def test_linear_kl_batch_invariance():
    N, V, Da, Db = 384, 2000, 128, 256
    ha, Wa, hb, Wb, _ = (t.to(DEV) for t in _kl_case(N, V, Da, Db, seed=51))
    kl, _, _ = vp.vp_linear_kl_fwd(ha, Wa, hb, Wb)
    part, _, _ = vp.vp_linear_kl_fwd(ha[128:256].contiguous(), Wa, hb[128:256].contiguous(), Wb)
    torch.cuda.synchronize()
    assert torch.equal(kl[128:256].view(torch.int32), part.view(torch.int32))


def test_linear_ent_kl_argument_errors():
    h = torch.zeros(4, 96, dtype=torch.bfloat16, device=DEV)     # D not a multiple of 64
    W = torch.zeros(8, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(vp.VPError):
        vp.vp_linear_entropy_fwd(h, W)
    h = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(8, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(vp.VPError):
        vp.vp_linear_kl_fwd(h, W, h, W, direction=2)
    H, st = vp.vp_linear_entropy_fwd(h[:0], W)
    assert H.numel() == 0


# ---------------------------------------------------------------------------
# Full size: hidden [8192, 4096] x W [75968, 4096], sampled rows
# ---------------------------------------------------------------------------
@pytest.mark.slow
def test_linear_entropy_kl_full_size_sampled():
    w = workloads.linear()
    t = workloads.linear(seed=14)
    ha, Wa, hb, Wb, g = (x.to(DEV) for x in (w["hidden"], w["weight"], t["hidden"], t["weight"], w["grad"]))
    H, st = vp.vp_linear_entropy_fwd(ha, Wa)
    kl, sa, sb = vp.vp_linear_kl_fwd(ha, Wa, hb, Wb)
    dha, dWa = vp.vp_linear_entropy_bwd(ha, Wa, st, g)
    torch.cuda.synchronize()
    rows = [0, 777, 8191]
    h64, W64, hb64, Wb64 = (parity.to64(x) for x in (w["hidden"][rows], w["weight"], t["hidden"][rows], t["weight"]))
    parity.check_out(H[rows], oracle.linear_entropy_fwd(h64, W64)[0], "full-size H")
    parity.check_out(kl[rows], oracle.linear_kl_fwd(h64, W64, hb64, Wb64)[0], "full-size KL")
    g64 = w["grad"][rows].double().numpy()
    rdh, _ = oracle.linear_entropy_bwd(h64, W64, g64, want_dW=False)
    z = oracle.linear_logits(h64, W64)
    dz = np.abs(oracle.entropy_bwd(z, g64))
    M = parity.oracle_all(z, z, np.zeros(len(rows), np.int64), g64, ops=("entropy",))["_mag"]["dH"]
    M = M * (1.0 + parity.logit_scale((h64, W64)))[:, None]
    parity.check_gemm_grad(dha[rows], rdh, parity.gemm_norms(dz, W64), "full-size entropy dhidden", M @ np.abs(W64))
    assert torch.isfinite(dWa).all()


# ---------------------------------------------------------------------------
# Generalized JSD of two models (interior beta; the endpoints are the KL calls)
# ---------------------------------------------------------------------------
def _jsd_mags(za, zb, beta, g):
    """M_j of the fp32 evaluation of dA and dB (as for the logits-level JSD)."""
    _, ma, la = oracle.entropy_fwd(za)
    _, mb, lb = oracle.entropy_fwd(zb)
    lp, lq = (za - ma[:, None]) - la[:, None], (zb - mb[:, None]) - lb[:, None]
    p, q = np.exp(lp), np.exp(lq)
    lmix = np.log(beta * q + (1 - beta) * p)
    ka, kb = np.sum(p * (lp - lmix), 1), np.sum(q * (lq - lmix), 1)
    ag = np.abs(g)[:, None]
    Ma = ag * (1 - beta) * p * (np.abs(lp) + np.abs(lmix) + np.abs(ka)[:, None] + 1.0)
    Mb = ag * beta * q * (np.abs(lq) + np.abs(lmix) + np.abs(kb)[:, None] + 1.0)
    return Ma, Mb


@pytest.mark.parametrize("beta", [0.3, 0.5, 0.9])
@pytest.mark.parametrize("N,V,Da,Db", [(256, 1024, 256, 128), (130, 300, 64, 64), (72, 70000, 64, 128)])
def test_linear_jsd_fwd_bwd(N, V, Da, Db, beta):
    ha, Wa, hb, Wb, g = _kl_case(N, V, Da, Db, seed=N + V + Da + Db + 7)
    dev = [t.to(DEV) for t in (ha, Wa, hb, Wb, g)]
    jsd, sa, sb = vp.vp_linear_jsd_fwd(*dev[:4], beta)
    grads = vp.vp_linear_jsd_bwd(*dev[:4], beta, sa, sb, dev[4])
    torch.cuda.synchronize()
    ha64, Wa64, hb64, Wb64 = (parity.to64(t) for t in (ha, Wa, hb, Wb))
    g64 = g.double().numpy()
    tag = f"{N}x{V} Da={Da} Db={Db} beta={beta}"
    parity.check_out(jsd, oracle.linear_jsd_fwd(ha64, Wa64, hb64, Wb64, beta), f"{tag} JSD")
    ref = oracle.linear_jsd_bwd(ha64, Wa64, hb64, Wb64, beta, g64)
    za, zb = oracle.linear_logits(ha64, Wa64), oracle.linear_logits(hb64, Wb64)
    dza, dzb = (np.abs(x) for x in oracle.jsd_bwd(za, zb, beta, g64))
    Ma, Mb = _jsd_mags(za, zb, beta, g64)
    lam = (1.0 + parity.logit_scale((ha64, Wa64), (hb64, Wb64)))[:, None]
    Ma, Mb = Ma * lam, Mb * lam
    norms = (parity.gemm_norms(dza, Wa64), parity.gemm_norms(dza.T, ha64), parity.gemm_norms(dzb, Wb64),
             parity.gemm_norms(dzb.T, hb64))
    evals = (Ma @ np.abs(Wa64), Ma.T @ np.abs(ha64), Mb @ np.abs(Wb64), Mb.T @ np.abs(hb64))
    for got, r, nm, ev, name in zip(grads, ref, norms, evals, ("dhidden A", "dW A", "dhidden B", "dW B")):
        parity.check_gemm_grad(got, r, nm, f"{tag} {name}", ev, kappa=parity.KAPPA_JSD)


def test_linear_jsd_endpoints_frozen_teacher_and_invariance():
    N, V, Da, Db = 136, 1500, 128, 64
    ha, Wa, hb, Wb, g = (t.to(DEV) for t in _kl_case(N, V, Da, Db, seed=43))
    for beta, d in ((0.0, vp.KL_FORWARD), (1.0, vp.KL_REVERSE)):
        jsd, _, _ = vp.vp_linear_jsd_fwd(ha, Wa, hb, Wb, beta)
        kl, _, _ = vp.vp_linear_kl_fwd(ha, Wa, hb, Wb, d)
        torch.cuda.synchronize()
        assert torch.equal(jsd, kl), f"beta = {beta} is the KL call"
    jsd, sa, sb = vp.vp_linear_jsd_fwd(ha, Wa, hb, Wb, 0.5)
    full = vp.vp_linear_jsd_bwd(ha, Wa, hb, Wb, 0.5, sa, sb, g)
    student = vp.vp_linear_jsd_bwd(ha, Wa, hb, Wb, 0.5, sa, sb, g, want=(True, True, False, False))
    part, _, _ = vp.vp_linear_jsd_fwd(ha[64:128].contiguous(), Wa, hb[64:128].contiguous(), Wb, 0.5)
    same, _, _ = vp.vp_linear_jsd_fwd(ha, Wa, ha, Wa, 0.5)
    torch.cuda.synchronize()
    assert student[2] is None and torch.equal(student[0], full[0]) and torch.equal(student[1], full[1])
    assert torch.equal(jsd[64:128].view(torch.int32), part.view(torch.int32))
    assert float(same.abs().max()) < 1e-5          # a model against itself: mix = p up to rounding
    with pytest.raises(vp.VPError):
        vp.vp_linear_jsd_fwd(ha, Wa, hb, Wb, 1.5)


# ---------------------------------------------------------------------------
# Edge cases: the smallest problem, and a NaN row of hidden states
# ---------------------------------------------------------------------------
def test_linear_ops_smallest_problem():
    ha, Wa, hb, Wb, g = _kl_case(1, 1, 64, 64, seed=61)
    dev = [t.to(DEV) for t in (ha, Wa, hb, Wb, g)]
    t = torch.zeros(1, dtype=torch.int64, device=DEV)
    lp, _ = vp.vp_linear_logp_fwd(dev[0], dev[1], t)
    H, _ = vp.vp_linear_entropy_fwd(dev[0], dev[1])
    kl, _, _ = vp.vp_linear_kl_fwd(*dev[:4])
    jsd, sa, sb = vp.vp_linear_jsd_fwd(*dev[:4], 0.5)
    grads = vp.vp_linear_jsd_bwd(*dev[:4], 0.5, sa, sb, dev[4])
    torch.cuda.synchronize()
    # one vocabulary row: p = q = 1, so logp = H = KL = JSD = 0 and every gradient is 0
    for x in (lp, H, kl, jsd):
        assert float(x.abs().max()) == 0.0
    assert all(float(gr.abs().max()) == 0.0 for gr in grads)


def test_linear_ops_nan_hidden_row():
    N, V, D = 130, 1000, 128
    ha, Wa, hb, Wb, g = _kl_case(N, V, D, D, seed=62)
    ha = ha.clone()
    ha[7, 5] = float("nan")
    dev = [t.to(DEV) for t in (ha, Wa, hb, Wb, g)]
    H, st = vp.vp_linear_entropy_fwd(dev[0], dev[1])
    dh, dW = vp.vp_linear_entropy_bwd(dev[0], dev[1], st, dev[4])
    kl, sa, sb = vp.vp_linear_kl_fwd(*dev[:4])
    torch.cuda.synchronize()
    ha64, Wa64, hb64, Wb64 = (parity.to64(t) for t in (ha, Wa, hb, Wb))
    parity.check_out(H, oracle.linear_entropy_fwd(ha64, Wa64)[0], "NaN row: H")
    parity.check_out(kl, oracle.linear_kl_fwd(ha64, Wa64, hb64, Wb64)[0], "NaN row: KL")
    assert torch.isnan(H[7]) and torch.isnan(kl[7]) and torch.isfinite(H[:7]).all() and torch.isfinite(kl[8:]).all()
    assert torch.isnan(dh[7]).all() and torch.isfinite(dh[8]).all() and torch.isnan(dW).all()


def test_linear_two_model_nan_row_backward():
    """A NaN row of model A's hidden states: NaN KL / JSD and NaN gradient rows for both models (the
    dual epilogues' column-checked path), every other row finite."""
    N, V, D = 130, 1000, 128
    ha, Wa, hb, Wb, g = _kl_case(N, V, D, D, seed=63)
    ha = ha.clone()
    ha[9, 3] = float("nan")
    dev = [t.to(DEV) for t in (ha, Wa, hb, Wb, g)]
    for direction in (vp.KL_REVERSE, vp.KL_FORWARD):
        kl, sa, sb = vp.vp_linear_kl_fwd(*dev[:4], direction)
        dha, dwa, dhb, dwb = vp.vp_linear_kl_bwd(*dev[:4], direction, sa, sb, dev[4])
        torch.cuda.synchronize()
        assert torch.isnan(kl[9]) and torch.isfinite(kl[:9]).all() and torch.isfinite(kl[10:]).all()
        for dh in (dha, dhb):
            assert torch.isnan(dh[9]).all() and torch.isfinite(dh[:9]).all() and torch.isfinite(dh[10:]).all()
        assert torch.isnan(dwa).all() and torch.isnan(dwb).all()
    jsd, sa, sb = vp.vp_linear_jsd_fwd(*dev[:4], 0.5)
    dha, dwa, dhb, dwb = vp.vp_linear_jsd_bwd(*dev[:4], 0.5, sa, sb, dev[4])
    torch.cuda.synchronize()
    assert torch.isnan(jsd[9]) and torch.isfinite(jsd[:9]).all() and torch.isfinite(jsd[10:]).all()
    for dh in (dha, dhb):
        assert torch.isnan(dh[9]).all() and torch.isfinite(dh[:9]).all() and torch.isfinite(dh[10:]).all()


def test_linear_two_model_wide_logit_spread():
    """Heads scaled so that the logits of a row spread over several hundred units: most p and q
    underflow to 0, the JSD's mixture underflows where both do (log mix = -inf), and the dual
    epilogues redo those tiles and groups with the column checks. KL and JSD, forward and
    backward, against the oracle."""
    N, V, Da, Db = 136, 1300, 64, 128
    ha, Wa, g = _model(71, N, V, Da, scale=400.0)
    hb, Wb, _ = _model(72, N, V, Db, scale=300.0)
    ha64, Wa64, hb64, Wb64 = (parity.to64(t) for t in (ha, Wa, hb, Wb))
    za, zb = oracle.linear_logits(ha64, Wa64), oracle.linear_logits(hb64, Wb64)
    spread = np.minimum(za.max(1) - za.min(1), zb.max(1) - zb.min(1))
    assert spread.min() > 200.0, "the case must push exp(z - m) below the fp32 range"
    _check_kl(ha, Wa, hb, Wb, g, vp.KL_REVERSE, "wide spread")
    _check_kl(ha, Wa, hb, Wb, g, vp.KL_FORWARD, "wide spread")
    beta = 0.4
    dev = [t.to(DEV) for t in (ha, Wa, hb, Wb, g)]
    jsd, sa, sb = vp.vp_linear_jsd_fwd(*dev[:4], beta)
    grads = vp.vp_linear_jsd_bwd(*dev[:4], beta, sa, sb, dev[4])
    torch.cuda.synchronize()
    g64 = g.double().numpy()
    parity.check_out(jsd, oracle.linear_jsd_fwd(ha64, Wa64, hb64, Wb64, beta), "wide spread JSD")
    ref = oracle.linear_jsd_bwd(ha64, Wa64, hb64, Wb64, beta, g64)
    dza, dzb = (np.abs(x) for x in oracle.jsd_bwd(za, zb, beta, g64))
    Ma, Mb = _jsd_mags(za, zb, beta, g64)
    # p, q and the mixture (>= min(beta, 1 - beta) max(p, q)) flush below 2^-126
    below = parity.TINY / min(beta, 1.0 - beta)
    Fa, Fb = parity.flushed(Ma, _probs(za), below=below), parity.flushed(Mb, _probs(zb), below=below)
    lam = (1.0 + parity.logit_scale((ha64, Wa64), (hb64, Wb64)))[:, None]
    Ma, Mb = Ma * lam, Mb * lam
    norms = (parity.gemm_norms(dza, Wa64), parity.gemm_norms(dza.T, ha64), parity.gemm_norms(dzb, Wb64),
             parity.gemm_norms(dzb.T, hb64))
    evals = (Ma @ np.abs(Wa64), Ma.T @ np.abs(ha64), Mb @ np.abs(Wb64), Mb.T @ np.abs(hb64))
    flush = (Fa @ np.abs(Wa64), Fa.T @ np.abs(ha64), Fb @ np.abs(Wb64), Fb.T @ np.abs(hb64))
    for got, r, nm, ev, fl, name in zip(grads, ref, norms, evals, flush, ("dhidden A", "dW A", "dhidden B", "dW B")):
        parity.check_gemm_grad(got, r, nm, f"wide spread JSD {name}", ev, fl, kappa=parity.KAPPA_JSD)
