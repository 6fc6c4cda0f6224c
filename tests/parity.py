"""Comparison helpers for GPU-vs-oracle parity (test infrastructure).

Tolerances (stated in the design notes, derived from the target):
  * per-row outputs (logp, H, KL, logS):  |x - y| <= 2e-5 + 2e-5 |y|;
  * fp32 gradients:                       |g - g64| <= 1e-6 max(1, |g64|): 1e-6 absolute up to
    |g64| = 1 and relative above (an absolute 1e-6 is below half the spacing
    of fp32 values from |g64| = 16.8 on, so no fp32 result could meet it there);
  * bf16 gradients:                       |g - RNE_bf16(g64)| <= 1 ulp_bf16(RNE_bf16(g64))
                                                               + KAPPA_BF16 * 2^-24 * M_j,
    where M_j is the magnitude of the operands of the element's formula
    (dlogp: |g|(p + onehot); dH: |g| p (|log p| + |H| + 1);
    dP of KL: |g| p (|log p| + |log q| + |KL| + 1); dQ of KL: |g| (p + q)).
    KAPPA_BF16 = 4: the forward's exponentials run on the hardware base-2
    unit, whose relative error (measured on GB300 over dense argument sweeps)
    is at most 1.44e-7 = 2.4 2^-24 per term, with a mean of -5e-8 below -1
    and +3.3e-8 above +1 and a spread of 3e-8; over a row's largest terms
    this leaves the centred mean c = W / S with ~2^-23 relative error, which
    the gradient resolves only where it cancels (log p ~ -H, log p - log q ~
    KL); elsewhere the gradients are within one ulp. 4 covers the per-term
    error of p plus that of c (the differences q - p and 1 - p are formed
    without cancellation). The GPU tests record the smallest factor each
    check would have passed with (kappa_needed; tests/parity_errors.md).
    ORACLE_EPS = 2^-40 bounds the fp64 oracle's own rounding relative to those
    operands (its sums run over up to ~10^5 terms); it matters only where the
    exact gradient is 0 (a uniform row: log p = -H exactly), where the oracle
    returns rounding noise of ~1e-20 and one ulp of that noise is meaningless;
    ulp below 2^-126 is taken as 2^-126 (the bf16 path flushes fp32
    subnormals to zero);
  * the generalized JSD gradient (test_gpu_jsd) carries KAPPA_JSD = 8 in
    place of KAPPA_BF16 (its mixture logarithms run on the hardware base-2
    unit too, adding their own error to that of p and q);
  * NaN and +-inf in the same places, everywhere.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import vocab_wide_logprobs_gb300 as vp

OUT_ATOL = 2e-5
OUT_RTOL = 2e-5
F32_GRAD_ATOL = 1e-6
KAPPA_BF16 = 4          # logprobs, entropy, KL, top-k and the fused linear ops
KAPPA_JSD = 8           # the generalized JSD (mixture logarithms on the base-2 unit)
ORACLE_EPS = 2.0 ** -40
TINY = 2.0 ** -126
STATS = {}  # worst error / tolerance and the share of elements that needed the conditioning term


def to64(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 copy of a bf16 / fp32 tensor (any device)."""
    return t.detach().to("cpu", torch.float64).numpy()


def rne_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even, in one step."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0)
    _, e = np.frexp(x[fin])                      # x = f 2^e, f in [0.5, 1)
    scale = np.maximum(np.ldexp(1.0, e - 8), 2.0 ** -133)  # bf16 spacing, subnormals included
    y = np.rint(x[fin] / scale) * scale          # exact in fp64; rint is half-to-even
    y[np.abs(y) > 3.3895313892515355e38] = np.inf * np.sign(y[np.abs(y) > 3.3895313892515355e38])
    out[fin] = y
    return out


def ulp_bf16(y: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(np.asarray(y, dtype=np.float64)), TINY)
    _, e = np.frexp(a)
    return np.ldexp(1.0, e - 8)


def _record_ulp(what, err, ulp, rows=None):
    """Per check: elements, how many are beyond one bf16 ulp, the worst error in ulps and (given the
    row of each element) the first rows holding elements beyond one ulp."""
    STATS[what] = {"n": int(err.size), "beyond_1ulp": int((err > ulp).sum()),
                   "worst_err_over_ulp": float((err / ulp).max()) if err.size else 0.0}
    if rows is not None and STATS[what]["beyond_1ulp"]:
        STATS[what]["rows_beyond"] = sorted({int(x) for x in np.asarray(rows)[err > ulp]})[:8]


def _record_kappa(what, err, base, mag, kappa):
    """The smallest conditioning factor the check would have passed with: max over the elements of
    (err - base) / (2^-24 M), base being every other term of the tolerance; 0 where all are within base."""
    with np.errstate(invalid="ignore", divide="ignore"):
        need = np.where(err > base, (err - base) / (2.0 ** -24 * mag), 0.0)
    STATS[what]["kappa_needed"] = float(np.nanmax(need)) if need.size else 0.0
    STATS[what]["kappa"] = float(kappa)


def _placement(got, ref, what):
    gn, rn = np.isnan(got), np.isnan(ref)
    if not (gn == rn).all():
        idx = np.argwhere(gn != rn)[:5]
        raise AssertionError(f"{what}: NaN placement differs at {idx.tolist()} "
                             f"(got {[got[tuple(i)] for i in idx]}, ref {[ref[tuple(i)] for i in idx]})")
    gi, ri = np.isinf(got), np.isinf(ref)
    if not ((gi == ri).all() and (got[ri] == ref[ri]).all()):
        idx = np.argwhere((gi != ri) | (ri & (got != ref)))[:5]
        raise AssertionError(f"{what}: inf placement differs at {idx.tolist()}")


def as_fp32_output(ref):
    """The oracle's fp64 value as an fp32 output reads it: magnitudes past FLT_MAX are +-inf."""
    ref = np.asarray(ref, np.float64)
    with np.errstate(invalid="ignore"):
        return np.where(np.abs(ref) > 3.4028234663852886e38, np.sign(ref) * np.inf, ref)


def check_out(got, ref, what, atol=OUT_ATOL, rtol=OUT_RTOL):
    got = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = as_fp32_output(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    _placement(got, ref, what)
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin])
    tol = atol + rtol * np.abs(ref[fin])
    if err.size and not (err <= tol).all():
        i = np.argmax(err / tol)
        raise AssertionError(f"{what}: err {err[i]:.3e} > tol {tol[i]:.3e} (got {got[fin][i]!r}, "
                             f"ref {ref[fin][i]!r}); {int((err > tol).sum())} bad of {err.size}")
    return float((err / tol).max()) if err.size else 0.0


def check_grad(got: torch.Tensor, ref: np.ndarray, what: str, mag=None, oracle_mag=None, kappa=KAPPA_BF16):
    """Returns the worst error as a fraction of its tolerance. `mag` = M_j (bf16 conditioning term, fp32
    evaluation); `oracle_mag` = M_j for the fp64 oracle's own rounding (ORACLE_EPS M_j), which matters
    only where the exact gradient is 0 and the oracle's value is rounding noise."""
    g = to64(got)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    if got.dtype == torch.bfloat16:
        r = rne_bf16(ref)
        _placement(g, r, what)
        fin = np.isfinite(r)
        err = np.abs(g[fin] - r[fin])
        ulp = ulp_bf16(r[fin])
        tol = ulp + (kappa * 2.0 ** -24 * np.asarray(mag)[fin] if mag is not None else 0.0)
        if oracle_mag is not None:
            tol = tol + ORACLE_EPS * np.asarray(oracle_mag)[fin]
        _record_ulp(what, err, ulp, np.nonzero(fin)[0] if fin.ndim == 2 else None)
        if mag is not None:
            base = ulp + (ORACLE_EPS * np.asarray(oracle_mag)[fin] if oracle_mag is not None else 0.0)
            _record_kappa(what, err, base, np.asarray(mag)[fin], kappa)
    else:
        _placement(g, ref, what)
        fin = np.isfinite(ref)
        err = np.abs(g[fin] - ref[fin])
        tol = F32_GRAD_ATOL * np.maximum(1.0, np.abs(ref[fin]))
        STATS[what] = {"max_abs_err": float(err.max()) if err.size else 0.0, "n": int(err.size)}
    if err.size and not (err <= tol).all():
        i = np.argmax(err / tol)
        raise AssertionError(f"{what}: err {err[i]:.3e} > tol {tol[i]:.3e} (got {g[fin][i]!r}, "
                             f"ref {ref[fin][i]!r}); {int((err > tol).sum())} bad of {err.size}")
    worst = float((err / tol).max()) if err.size else 0.0
    STATS[what]["worst_over_tol"] = worst
    return worst


# ---------------------------------------------------------------------------
# Run every op on the GPU and on the oracle over the same inputs
# ---------------------------------------------------------------------------
def gpu_all(a, b, targets, grad, ops=("logprobs", "entropy", "kl_rev", "kl_fwd"), vocab_start=0):
    """a, b: CUDA logits views ([N, V] or [B, T, V]); targets int64 [N]; grad fp32 [N]."""
    out = {}
    t = targets.reshape(-1)
    g = grad.reshape(-1)
    if "logprobs" in ops:
        err = torch.zeros(1, dtype=torch.int32, device=a.device)
        lp, st = vp.vp_logprobs_fwd(a, t, vocab_start, err_word=err)
        out["logp"], out["logp_stats"] = lp, st
        out["dlogp"] = vp.vp_logprobs_bwd(a, t, st, g, vocab_start, err_word=err)
        out["err"] = err
    if "entropy" in ops:
        H, st = vp.vp_entropy_fwd(a)
        out["H"], out["H_stats"] = H, st
        out["dH"] = vp.vp_entropy_bwd(a, st, g)
    for name, d in (("kl_rev", vp.KL_REVERSE), ("kl_fwd", vp.KL_FORWARD)):
        if name in ops:
            kl, sa, sb = vp.vp_kl_fwd(a, b, d)
            out[name], out[name + "_sa"], out[name + "_sb"] = kl, sa, sb
            da, db = vp.vp_kl_bwd(a, b, d, sa, sb, g)
            out["d" + name + "_a"], out["d" + name + "_b"] = da, db
    torch.cuda.synchronize()
    return out


def rows2d(x: torch.Tensor) -> np.ndarray:
    """fp64 [N, V] copy of a [N, V] or [B, T, V] view."""
    return to64(x.reshape(-1, x.shape[-1]))


def _logp_rows(x64, m, logS):
    with np.errstate(invalid="ignore", over="ignore"):
        lp = (x64 - m[:, None]) - logS[:, None]
        return lp, np.exp(lp)


def oracle_all(a64, b64, targets, grad, ops=("logprobs", "entropy", "kl_rev", "kl_fwd"), vocab_start=0):
    """Oracle outputs and gradients, plus the saved statistics and the M_j magnitudes of the tolerance."""
    t = np.asarray(targets).reshape(-1)
    g = np.asarray(grad, np.float64).reshape(-1)
    ag = np.abs(g)[:, None]
    out, mag = {}, {}
    if "logprobs" in ops or "entropy" in ops or any(k in ops for k in ("kl_rev", "kl_fwd")):
        H, ma, lsa = oracle.entropy_fwd(a64)
        lpa, pa = _logp_rows(a64, ma, lsa)
    if "logprobs" in ops:
        lp, m, ls, err = oracle.logprobs_fwd(a64, t, vocab_start)
        out.update(logp=lp, logp_stats=(m, ls), err=err, dlogp=oracle.logprobs_bwd(a64, t, g, vocab_start))
        onehot = np.zeros_like(pa)
        loc = t - vocab_start
        ok = (t >= 0) & (loc >= 0) & (loc < a64.shape[1])
        onehot[np.nonzero(ok)[0], loc[ok]] = 1.0
        mag["dlogp"] = ag * (pa + onehot)
    if "entropy" in ops:
        out.update(H=H, H_stats=(ma, lsa), dH=oracle.entropy_bwd(a64, g))
        with np.errstate(invalid="ignore"):
            mag["dH"] = ag * pa * (np.abs(lpa) + np.abs(H)[:, None] + 1.0)
    kls = [k for k in ("kl_rev", "kl_fwd") if k in ops]
    if kls:
        Hb, mb, lsb = oracle.entropy_fwd(b64)
        lpb, pb = _logp_rows(b64, mb, lsb)
    for name in kls:
        d = oracle.REVERSE if name == "kl_rev" else oracle.FORWARD
        kl, ma_, lsa_, mb_, lsb_ = oracle.kl_fwd(a64, b64, d)
        out[name], out[name + "_sa"], out[name + "_sb"] = kl, (ma_, lsa_), (mb_, lsb_)
        da, db = oracle.kl_bwd(a64, b64, g, d)
        out["d" + name + "_a"], out["d" + name + "_b"] = da, db
        (lpP, pP), (lpQ, pQ) = ((lpa, pa), (lpb, pb)) if d == oracle.REVERSE else ((lpb, pb), (lpa, pa))
        with np.errstate(invalid="ignore"):
            mP = ag * pP * (np.abs(lpP) + np.abs(lpQ) + np.abs(kl)[:, None] + 1.0)
        mQ = ag * (pP + pQ)
        mag["d" + name + ("_a" if d == oracle.REVERSE else "_b")] = mP
        mag["d" + name + ("_b" if d == oracle.REVERSE else "_a")] = mQ
    # positions with p = 0 have zero operands (their |log p| is inf): no conditioning term there
    out["_mag"] = {k: np.nan_to_num(v, nan=0.0, posinf=0.0) for k, v in mag.items()}
    return out


def _record_centred_mean(got, ref, k, prim, st, rows, what):
    """Error of the record's centred mean c against the oracle's (informational):
    entropy c = log S - H; KL(P||Q) on P's record c = KL + log S_P - log S_Q."""
    if prim == "H" and k == "H_stats":
        c_ref = ref["H_stats"][1] - np.asarray(ref["H"], np.float64)
    elif prim in ("kl_rev", "kl_fwd"):
        p_key = prim + ("_sa" if prim == "kl_rev" else "_sb")
        q_key = prim + ("_sb" if prim == "kl_rev" else "_sa")
        if k != p_key:
            return
        c_ref = np.asarray(ref[prim], np.float64) + ref[p_key][1] - ref[q_key][1]
    else:
        return
    c = to64(st["c"])
    fin = np.isfinite(c_ref)
    if fin.any():
        e = np.abs(c[fin] - c_ref[fin])
        STATS[what + " c"] = {"n": int(fin.sum()), "max_abs_err": float(e.max()),
                              "max_rel_err": float((e / np.maximum(np.abs(c_ref[fin]), 1e-30)).max())}


def _primary(key):
    for p in ("kl_rev", "kl_fwd", "logp", "H"):
        if key.startswith(p + "_"):
            return p
    return None


def compare_all(got: dict, ref: dict, rows=None, tag=""):
    """Element-by-element parity on the given rows (all rows when None). Returns worst ratios.

    Saved statistics are compared on the rows whose output is not NaN: m must
    equal the exact row max wherever that max is finite, logS = hi + lo must
    match the oracle's log S to the output tolerance."""
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    worst = {}
    mag = ref.get("_mag", {})
    for k, r in ref.items():
        if k in ("err", "_mag") or k not in got:
            continue
        gk = got[k]
        prim = _primary(k)
        if k.startswith("d"):
            # logprobs, entropy and KL gradients: one bf16 ulp plus KAPPA_BF16 2^-24 M_j (and the
            # fp64 oracle's own rounding)
            worst[k] = check_grad(sel(gk), r, f"{tag}{k}", mag.get(k), oracle_mag=mag.get(k))
        elif prim is not None:
            m_ref, ls_ref = r
            st = vp.decode_rowstats(sel(gk))
            ok = ~np.isnan(np.asarray(ref[prim]))
            if k.endswith("_sb") and prim.startswith("kl"):
                ok = ok & np.isfinite(np.asarray(ref[prim]))  # Q's record on flagged rows may be empty
            m64 = to64(st["m"])
            fin = ok & np.isfinite(m_ref)
            assert (m64[fin] == m_ref[fin]).all(), f"{tag}{k}: row max differs"
            worst[k] = check_out(to64(st["logS"])[ok], ls_ref[ok], f"{tag}{k} logS")
            _record_centred_mean(got, ref, k, prim, st, rows, f"{tag}{k}")
        else:
            worst[k] = check_out(sel(gk), r, f"{tag}{k}")
    return worst


# ---------------------------------------------------------------------------
# Gradients of the fused linear ops: dhidden = dz . W and dW = dz^T . h, with dz
# formed in fp32 in the GEMM epilogue.
# Exact precision (VP_GRAD_EXACT, the default): dz reaches the bf16 tensor cores
# as the pair dz_hi + dz_lo, so each output is held to one bf16 ulp plus a
# rounding term in the root-sum-square of the dot product's terms,
# GEMM_RSS * sqrt(sum_k (dz_k op_k)^2) (gemm_norms).
# Fast precision (VP_GRAD_FAST): dz is rounded to bf16, so each output is held
# to one bf16 ulp plus the forward error bound of a dot product with
# bf16-rounded dz, 2^-8 sum_k |dz_k| |op_k|; where dz itself is a difference
# that can cancel (the entropy and KL gradients), the fp32 evaluation error of
# dz enters as well: KAPPA_BF16 2^-24 sum_k M_k |op_k| (eval_mag).
# For the entropy, KL and JSD of the fused linear ops, eval_mag takes M_k (1 + L_r)
# in place of M_k (both precisions), L_r = logit_scale(...) of the row: their dz
# is formed from the recomputed logits, fp32 accumulations of bf16 products
# whose error is ~2^-24 L_r, and where dz cancels (q ~ p, log p - log q ~ KL,
# log p ~ -H) that error is what remains.
# In both, the exponentials flush a probability below the fp32 normal range
# (2^-126) to 0, so an element of dz whose p (or q) is that small may be lost
# whole: its share M_j of the tolerance, carried through the same dot product,
# enters unscaled (flush_mag; flushed() selects it).
# ---------------------------------------------------------------------------
GEMM_KAPPA = 2.0 ** -8
GEMM_RSS = 2.0 ** -13


def logit_scale(*models):
    """Per row, the largest sum_k |h_rk| |w_jk| over the vocabulary (summed over the models given as
    (h, W) pairs): the magnitude that bounds the fp32 accumulation error of the recomputed logits."""
    total = None
    for h, W in models:
        L = np.abs(np.asarray(h, np.float64)) @ np.abs(np.asarray(W, np.float64)).T
        total = L if total is None else total + L
    return total.max(axis=1)


def gemm_norms(a, b):
    """(sum_k |a_ik| |b_kj|, sqrt(sum_k a_ik^2 b_kj^2)) for the product a . b."""
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.abs(a) @ np.abs(b), np.sqrt((a * a) @ (b * b))


def flushed(M, *probs, below=TINY):
    """M_j at the elements where one of the formula's probabilities is below `below`, else 0."""
    mask = np.zeros(np.shape(M), bool)
    for p in probs:
        with np.errstate(invalid="ignore"):
            mask |= np.asarray(p) < below
    return np.where(mask, M, 0.0)


def check_gemm_grad(got, ref, norms, what, eval_mag=None, flush_mag=None, fast=False, kappa=KAPPA_BF16):
    """norms: gemm_norms(dz, operand) of the output's dot products (l1, l2); eval_mag: sum_k M_k |op_k|."""
    l1, l2 = norms
    g = to64(got)
    r = rne_bf16(ref)
    _placement(g, r, what)
    fin = np.isfinite(r)
    err = np.abs(g[fin] - r[fin])
    ulp = ulp_bf16(r[fin])
    tol = ulp + (GEMM_KAPPA * l1[fin] if fast else GEMM_RSS * l2[fin])
    if eval_mag is not None:
        tol = tol + kappa * 2.0 ** -24 * eval_mag[fin]
    if flush_mag is not None:
        tol = tol + flush_mag[fin]
    _record_ulp(what, err, ulp)
    if eval_mag is not None:
        base = ulp + (GEMM_KAPPA * l1[fin] if fast else GEMM_RSS * l2[fin]) + (flush_mag[fin] if flush_mag is not None else 0.0)
        _record_kappa(what, err, base, eval_mag[fin], kappa)
    with np.errstate(invalid="ignore", divide="ignore"):
        over = np.where(l2[fin] > 0, np.maximum(err - ulp, 0.0) / l2[fin], 0.0)
    STATS[what]["worst_beyond_ulp_over_rss"] = float(over.max()) if err.size else 0.0
    STATS[what]["worst_over_tol"] = float((err / tol).max()) if err.size else 0.0
    STATS[what]["precision"] = "fast" if fast else "exact"
    if err.size:
        i = int(np.argmax(err / tol))
        idx = np.argwhere(fin)[i].tolist()
        STATS[what]["worst"] = {"index": idx, "got": float(g[fin][i]), "ref": float(ref[fin][i]),
                                "ulp": float(ulp[i]), "rss": float(l2[fin][i]),
                                "eval": float(eval_mag[fin][i]) if eval_mag is not None else None}
    assert (err <= tol).all(), f"{what}: worst err/tol {(err / tol).max():.3f}, {(err > tol).sum()} bad of {err.size}"
    return float((err / tol).max())
