"""Comparison helpers for GPU-vs-oracle parity (test infrastructure).

Tolerances (stated in the design notes, derived from the target):
  * per-row outputs (logp, H, KL, logS):  |x - y| <= 2e-5 + 2e-5 |y|;
  * fp32 gradients:                       |g - g64| <= 1e-6;
  * bf16 gradients:                       |g - RNE_bf16(g64)| <= 1 ulp_bf16(RNE_bf16(g64)),
    where ulp below 2^-126 is taken as 2^-126 because the bf16 path computes
    in fp32 with subnormal results flushed to zero;
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
TINY = 2.0 ** -126


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


def check_out(got, ref, what, atol=OUT_ATOL, rtol=OUT_RTOL):
    got = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
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


def check_grad(got: torch.Tensor, ref: np.ndarray, what: str):
    """Returns the worst error as a fraction of its tolerance."""
    g = to64(got)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    if got.dtype == torch.bfloat16:
        r = rne_bf16(ref)
        _placement(g, r, what)
        fin = np.isfinite(r)
        err = np.abs(g[fin] - r[fin])
        tol = ulp_bf16(r[fin])
    else:
        _placement(g, ref, what)
        fin = np.isfinite(ref)
        err = np.abs(g[fin] - ref[fin])
        tol = np.full(err.shape, F32_GRAD_ATOL)
    if err.size and not (err <= tol).all():
        i = np.argmax(err / tol)
        raise AssertionError(f"{what}: err {err[i]:.3e} > tol {tol[i]:.3e} (got {g[fin][i]!r}, "
                             f"ref {ref[fin][i]!r}); {int((err > tol).sum())} bad of {err.size}")
    return float((err / tol).max()) if err.size else 0.0


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
        lp, m, ls = vp.vp_logprobs_fwd(a, t, vocab_start, err_word=err)
        out["logp"], out["logp_m"], out["logp_logS"] = lp, m, ls
        out["dlogp"] = vp.vp_logprobs_bwd(a, t, m, ls, g, vocab_start, err_word=err)
        out["err"] = err
    if "entropy" in ops:
        H, m, ls = vp.vp_entropy_fwd(a)
        out["H"], out["H_m"], out["H_logS"] = H, m, ls
        out["dH"] = vp.vp_entropy_bwd(a, m, ls, H, g)
    for name, d in (("kl_rev", vp.KL_REVERSE), ("kl_fwd", vp.KL_FORWARD)):
        if name in ops:
            kl, ma, lsa, mb, lsb = vp.vp_kl_fwd(a, b, d)
            out[name] = kl
            out[name + "_ma"], out[name + "_lsa"], out[name + "_mb"], out[name + "_lsb"] = ma, lsa, mb, lsb
            da, db = vp.vp_kl_bwd(a, b, d, ma, lsa, mb, lsb, kl, g)
            out["d" + name + "_a"], out["d" + name + "_b"] = da, db
    torch.cuda.synchronize()
    return out


def rows2d(x: torch.Tensor) -> np.ndarray:
    """fp64 [N, V] copy of a [N, V] or [B, T, V] view."""
    return to64(x.reshape(-1, x.shape[-1]))


def oracle_all(a64, b64, targets, grad, ops=("logprobs", "entropy", "kl_rev", "kl_fwd"), vocab_start=0):
    t = np.asarray(targets).reshape(-1)
    g = np.asarray(grad, np.float64).reshape(-1)
    out = {}
    if "logprobs" in ops:
        lp, m, ls, err = oracle.logprobs_fwd(a64, t, vocab_start)
        out.update(logp=lp, logp_m=m, logp_logS=ls, err=err, dlogp=oracle.logprobs_bwd(a64, t, g, vocab_start))
    if "entropy" in ops:
        H, m, ls = oracle.entropy_fwd(a64)
        out.update(H=H, H_m=m, H_logS=ls, dH=oracle.entropy_bwd(a64, g))
    for name, d in (("kl_rev", oracle.REVERSE), ("kl_fwd", oracle.FORWARD)):
        if name in ops:
            kl, ma, lsa, mb, lsb = oracle.kl_fwd(a64, b64, d)
            out[name] = kl
            out[name + "_ma"], out[name + "_lsa"], out[name + "_mb"], out[name + "_lsb"] = ma, lsa, mb, lsb
            da, db = oracle.kl_bwd(a64, b64, g, d)
            out["d" + name + "_a"], out["d" + name + "_b"] = da, db
    return out


def _primary(key):
    for p in ("kl_rev", "kl_fwd", "logp", "H"):
        if key.startswith(p + "_"):
            return p
    return None


def compare_all(got: dict, ref: dict, rows=None, tag=""):
    """Element-by-element parity on the given rows (all rows when None). Returns worst ratios.

    Saved statistics (m, logS) are compared on the rows whose output is not NaN:
    the centre m must equal the exact row max wherever that max is finite."""
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    worst = {}
    for k, r in ref.items():
        if k == "err" or k not in got:
            continue
        gk = got[k]
        prim = _primary(k)
        if k.startswith("d"):
            worst[k] = check_grad(sel(gk), r, f"{tag}{k}")
        elif prim is not None:
            ok = ~np.isnan(np.asarray(ref[prim]))
            g64 = to64(sel(gk))
            if k.endswith(("_m", "_ma", "_mb")):
                fin = ok & np.isfinite(r)
                assert (g64[fin] == r[fin]).all(), f"{tag}{k}: row max differs"
            else:
                worst[k] = check_out(g64[ok], r[ok], f"{tag}{k}")
        else:
            worst[k] = check_out(sel(gk), r, f"{tag}{k}")
    return worst
