"""Pins for the fp64 oracle: checks against facts that do not come from the oracle.

Each ``pin_*`` function takes an oracle library handle (``None`` = the default
build) and raises AssertionError when the oracle disagrees with:

* brute force in Python ``decimal`` at 60+ digits on tiny rows, computing the
  softmax without any max-centring (so the oracle's centring is checked too),
  and gradients by Decimal central differences (so no gradient formula is
  restated here);
* closed forms: the uniform row (H = log V, logp = -log V, KL(A||A) = 0), the
  two-token row (binary entropy and binary KL), the one-hot row spanning
  +-3e38 (H = 0 and KL(p||p) = 0 with zero gradients, page "Add Triton kernels
  for vocab-parallel logprobs, entropy and KL", Codex thread "Guard zero
  rescaling before applying infinite shifts");
* invariants: 0 <= H <= log V, KL >= 0, logp <= 0, sum_t exp(logp_t) = 1,
  H = -sum_t p_t logp_t, every gradient row sums to 0, shift invariance at
  offsets 1e4 and 2^20 (same page, second commit message: large common offsets);
* fp64 central differences on V = 64 rows;
* the re-centring merge over 2, 3 and 7 host shards, with empty and all -inf
  shards, equal to the direct form;
* the per-shard records (max, sum-exp, centred weighted sum, flags) against
  Decimal sums over each shard;
* hand-built rows for every NaN / inf precedence rule and target rule;
* several target ids per row: Decimal brute force with duplicate and ignored
  ids and a fully ignored row, K = 1 against the single-id definition,
  duplicated ids against one id carrying the summed gradient;
* the generalized JSD: Decimal brute force of the value and of both gradients,
  JSD(A, A) = 0, disjoint supports giving the entropy of the mixing weights,
  symmetry at beta = 1/2, bounds, and the limits JSD_beta / beta -> KL(B||A)
  and JSD_beta / (1 - beta) -> KL(A||B) that tie it to the KL endpoints.

``tests/test_oracle_mutants.py`` plants plausible mistakes in copies of the
oracle source and checks that at least one pin fails for each.
"""
from __future__ import annotations

import math
from decimal import Decimal, localcontext

import numpy as np

import oracle

INF = float("inf")
NAN = float("nan")


# ----------------------------------------------------------------------------
# Decimal brute force (no max-centring, no library softmax)
# ----------------------------------------------------------------------------
def _dexp(v):
    if isinstance(v, Decimal):
        return v.exp()
    if v == -INF:
        return Decimal(0)
    return Decimal(v).exp()


def _dprobs(z):
    e = [_dexp(v) for v in z]
    S = sum(e)
    return [x / S for x in e]


def _dentropy(z):
    return -sum((p * p.ln() for p in _dprobs(z) if p > 0), Decimal(0))


def _dlogp(z, t):
    p = _dprobs(z)[t]
    return p.ln() if p > 0 else Decimal("-Infinity")


def _dkl(P, Q):
    p, q = _dprobs(P), _dprobs(Q)
    return sum((pi * (pi.ln() - qi.ln()) for pi, qi in zip(p, q) if pi > 0), Decimal(0))


def _dgrad(f, z, h=Decimal("1e-25")):
    """Central differences of a Decimal function of a row (entries may be -inf)."""
    out = []
    for j in range(len(z)):
        if z[j] == -INF:
            out.append(Decimal(0))
            continue
        zp = [Decimal(v) if v != -INF else -INF for v in z]
        zm = list(zp)
        zp[j] = Decimal(z[j]) + h
        zm[j] = Decimal(z[j]) - h
        out.append((f(zp) - f(zm)) / (2 * h))
    return out


def _close(a, b, atol, rtol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    same_nan = np.isnan(a) == np.isnan(b)
    assert same_nan.all(), f"{what}: NaN placement differs\n{a}\n{b}"
    fin = np.isfinite(b)
    assert (np.isinf(a) == np.isinf(b)).all() and (a[np.isinf(b)] == b[np.isinf(b)]).all(), \
        f"{what}: inf placement differs\n{a}\n{b}"
    err = np.abs(a[fin] - b[fin])
    tol = atol + rtol * np.abs(b[fin])
    assert (err <= tol).all(), f"{what}: max err {err.max():.3e} (tol {tol[np.argmax(err - tol)]:.3e})"


def _tiny_rows(seed, V, n, mask_frac=0.0):
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 2.5, size=(n, V))
    if mask_frac:
        m = rng.random((n, V)) < mask_frac
        m[:, 0] = False  # keep each row supported somewhere
        x[m] = -INF
    return x


# ----------------------------------------------------------------------------
# Brute force pins
# ----------------------------------------------------------------------------
def pin_brute_force_fwd(lib=None):
    with localcontext() as ctx:
        ctx.prec = 60
        for V in (1, 2, 3, 5, 8, 16):
            a = _tiny_rows(V, V, 6, mask_frac=0.2 if V > 2 else 0.0)
            b = _tiny_rows(100 + V, V, 6)
            b[:, :] += 3.0  # a different offset per tensor
            tg = np.arange(6) % V
            H, _, _ = oracle.entropy_fwd(a, lib=lib)
            lp, _, _, _ = oracle.logprobs_fwd(a, tg, lib=lib)
            klr = oracle.kl_fwd(a, b, oracle.REVERSE, lib=lib)[0]
            klf = oracle.kl_fwd(a, b, oracle.FORWARD, lib=lib)[0]
            for r in range(6):
                _close(H[r], float(_dentropy(list(a[r]))), 1e-14, 1e-14, f"H V={V}")
                _close(lp[r], float(_dlogp(list(a[r]), tg[r])), 1e-14, 1e-14, f"logp V={V}")
                _close(klr[r], float(_dkl(list(a[r]), list(b[r]))), 1e-14, 1e-13, f"KL(A||B) V={V}")
                # forward KL(B||A): A has -inf where B does not -> +inf (mismatch)
                expect = INF if np.any(np.isneginf(a[r]) & ~np.isneginf(b[r])) \
                    else float(_dkl(list(b[r]), list(a[r])))
                _close(klf[r], expect, 1e-14, 1e-13, f"KL(B||A) V={V}")


def pin_brute_force_grads(lib=None):
    with localcontext() as ctx:
        ctx.prec = 80
        for V in (2, 3, 5, 8):
            a = _tiny_rows(7 * V, V, 3, mask_frac=0.25 if V > 2 else 0.0)
            b = _tiny_rows(9 * V, V, 3)
            tg = (np.arange(3) * 2 + 1) % V
            a[np.arange(3), tg] = 0.5  # the target itself is never masked here
            g = np.array([0.7, -1.3, 2.1])
            dlog = oracle.logprobs_bwd(a, tg, g, lib=lib)
            dent = oracle.entropy_bwd(a, g, lib=lib)
            da_r, db_r = oracle.kl_bwd(a, b, g, oracle.REVERSE, lib=lib)
            db_f, da_f = oracle.kl_bwd(b, a, g, oracle.FORWARD, lib=lib)  # KL(A||B) again, args swapped
            for r in range(3):
                gr = Decimal(g[r])
                A, B = list(a[r]), list(b[r])
                ref_lp = [gr * d for d in _dgrad(lambda z: _dlogp(z, tg[r]), A)]
                ref_h = [gr * d for d in _dgrad(_dentropy, A)]
                ref_da = [gr * d for d in _dgrad(lambda z: _dkl(z, B), A)]
                ref_db = [gr * d for d in _dgrad(lambda z: _dkl(A, z), B)]
                f = lambda L: [float(v) for v in L]
                _close(dlog[r], f(ref_lp), 1e-13, 1e-12, f"dlogp V={V}")
                _close(dent[r], f(ref_h), 1e-13, 1e-12, f"dH V={V}")
                _close(da_r[r], f(ref_da), 1e-13, 1e-12, f"dKL/dA V={V}")
                _close(db_r[r], f(ref_db), 1e-13, 1e-12, f"dKL/dB V={V}")
                _close(da_f[r], f(ref_da), 1e-13, 1e-12, f"dKL/dA (forward, swapped) V={V}")
                _close(db_f[r], f(ref_db), 1e-13, 1e-12, f"dKL/dB (forward, swapped) V={V}")


def pin_topk_targets(lib=None):
    """Several ids per row: Decimal brute force, the single-id oracle at K = 1, duplicates add up."""
    with localcontext() as ctx:
        ctx.prec = 80
        for V in (3, 5, 8):
            x = _tiny_rows(500 + V, V, 4, mask_frac=0.2)
            t = np.array([[0, 0, -1], [V - 1, 1 % V, 2 % V], [-1, -1, -1], [2 % V, -5, 0]])
            x[np.arange(4)[:, None], np.maximum(t, 0)] = 0.25      # ids never sit on a masked logit
            g = np.array([[0.5, -1.5, 9.0], [1.0, 2.0, -0.5], [3.0, 3.0, 3.0], [0.7, 4.0, -1.1]])
            lp, err = oracle.logprobs_topk_fwd(x, t, lib=lib)
            dx = oracle.logprobs_topk_bwd(x, t, g, lib=lib)
            assert err == 0
            for r in range(4):
                row = list(x[r])
                for k in range(3):
                    ref = 0.0 if t[r, k] < 0 else float(_dlogp(row, t[r, k]))
                    _close(lp[r, k], ref, 1e-14, 1e-14, f"top-k logp V={V}")
                used = [(Decimal(g[r, k]), t[r, k]) for k in range(3) if t[r, k] >= 0]
                f = lambda z: sum((gk * _dlogp(z, tk) for gk, tk in used), Decimal(0))
                ref = [float(d) for d in _dgrad(f, row)] if used else [0.0] * V
                _close(dx[r], ref, 1e-13, 1e-12, f"top-k gradient V={V} row {r}")
    # K = 1 is the single-id oracle; a duplicated id carries the sum of its gradients
    N, V = 6, 300
    x = _rand(81, N, V)
    t1 = np.random.default_rng(82).integers(0, V, N)
    t1[2] = -1
    g1 = np.linspace(-1, 2, N)
    assert np.array_equal(oracle.logprobs_topk_fwd(x, t1[:, None], lib=lib)[0][:, 0],
                          oracle.logprobs_fwd(x, t1, lib=lib)[0])
    _close(oracle.logprobs_topk_bwd(x, t1[:, None], g1[:, None], lib=lib), oracle.logprobs_bwd(x, t1, g1, lib=lib),
           1e-15, 0, "top-k K = 1")
    g2 = np.stack([0.25 * g1, 0.75 * g1], 1)
    _close(oracle.logprobs_topk_bwd(x, np.stack([t1, t1], 1), g2, lib=lib), oracle.logprobs_bwd(x, t1, g1, lib=lib),
           1e-15, 1e-14, "duplicated ids")
    # an id outside the shard: NaN for that id, the error bit, a NaN gradient row
    t = np.stack([t1, t1], 1)
    t[4, 1] = V + 7
    lp, err = oracle.logprobs_topk_fwd(x, t, lib=lib)
    assert err == 1 and np.isnan(lp[4, 1]) and np.isfinite(lp[4, 0])
    assert np.isnan(oracle.logprobs_topk_bwd(x, t, g2, lib=lib)[4]).all()


# ----------------------------------------------------------------------------
# Closed forms
# ----------------------------------------------------------------------------
def pin_uniform_row(lib=None):
    for V in (1, 7, 4096, 75968):
        x = np.full((3, V), 1.25)
        x[1] = -40.0
        x[2] = 1e4
        H = oracle.entropy_fwd(x, lib=lib)[0]
        _close(H, np.full(3, math.log(V)), 1e-12, 1e-11, f"uniform H V={V}")  # fp64 sum of V terms
        tg = np.array([0, V // 2, V - 1])
        lp = oracle.logprobs_fwd(x, tg, lib=lib)[0]
        _close(lp, np.full(3, -math.log(V)), 1e-12, 1e-12, f"uniform logp V={V}")
        kl = oracle.kl_fwd(x, x + 3.0, lib=lib)[0]
        _close(kl, np.zeros(3), 1e-13, 0, f"uniform KL V={V}")
        if V <= 4096:
            g = np.array([1.0, -2.0, 0.5])
            dH = oracle.entropy_bwd(x, g, lib=lib)
            _close(dH, np.zeros_like(x), 1e-14, 0, "uniform dH")
            dl = oracle.logprobs_bwd(x, tg, g, lib=lib)
            ref = -g[:, None] * np.full_like(x, 1.0 / V)
            ref[np.arange(3), tg] += g
            _close(dl, ref, 1e-14, 1e-13, "uniform dlogp")


def pin_two_token_closed_form(lib=None):
    rng = np.random.default_rng(3)
    a = rng.normal(0, 3, size=(16, 2))
    b = rng.normal(0, 3, size=(16, 2))
    p = 1.0 / (1.0 + np.exp(-(a[:, 0] - a[:, 1])))
    q = 1.0 / (1.0 + np.exp(-(b[:, 0] - b[:, 1])))
    Hc = -(p * np.log(p) + (1 - p) * np.log1p(-p))
    klc = p * np.log(p / q) + (1 - p) * np.log((1 - p) / (1 - q))
    _close(oracle.entropy_fwd(a, lib=lib)[0], Hc, 1e-13, 1e-12, "binary entropy")
    _close(oracle.kl_fwd(a, b, lib=lib)[0], klc, 1e-13, 1e-11, "binary KL")
    lp = oracle.logprobs_fwd(a, np.zeros(16, dtype=np.int64), lib=lib)[0]
    _close(lp, np.log(p), 1e-13, 1e-12, "binary logp")


def pin_one_hot_extremes(lib=None):
    for big in (3e38, 1e308):
        x = np.array([[-big, big, -big, -big], [big, -big, -big, -big], [-big, -big, -big, big]])
        g = np.array([1.5, -0.5, 2.0])
        H = oracle.entropy_fwd(x, lib=lib)[0]
        assert (H == 0.0).all(), f"one-hot H {H}"
        kl = oracle.kl_fwd(x, x, lib=lib)[0]
        assert (kl == 0.0).all(), f"one-hot KL(p||p) {kl}"
        dH = oracle.entropy_bwd(x, g, lib=lib)
        assert (dH == 0.0).all(), f"one-hot dH {dH}"
        da, db = oracle.kl_bwd(x, x, g, lib=lib)
        assert (da == 0.0).all() and (db == 0.0).all(), "one-hot dKL"
        tg = np.array([1, 0, 3])
        lp = oracle.logprobs_fwd(x, tg, lib=lib)[0]
        assert (lp == 0.0).all(), f"one-hot logp {lp}"
        assert (oracle.logprobs_bwd(x, tg, g, lib=lib) == 0.0).all(), "one-hot dlogp"


# ----------------------------------------------------------------------------
# Invariants on random rows
# ----------------------------------------------------------------------------
def _rand(seed, N, V, sigma=3.0, offset=5.0):
    rng = np.random.default_rng(seed)
    return rng.normal(0, sigma, (N, V)) + rng.uniform(-offset, offset, (N, 1))


def pin_invariants(lib=None):
    N, V = 24, 1000
    a, b = _rand(11, N, V), _rand(12, N, V)
    g = np.random.default_rng(13).normal(size=N)
    H = oracle.entropy_fwd(a, lib=lib)[0]
    assert (H >= -1e-12).all() and (H <= math.log(V) + 1e-12).all(), "0 <= H <= log V"
    for d in (oracle.REVERSE, oracle.FORWARD):
        kl = oracle.kl_fwd(a, b, d, lib=lib)[0]
        assert (kl >= -1e-12).all(), "KL >= 0"
    assert (oracle.kl_fwd(a, a, lib=lib)[0] == 0.0).all(), "KL(P||P) = 0 exactly"
    # logprobs of every token of a row: normalisation and the entropy identity
    rows = np.repeat(a[:4], V, axis=0)
    tg = np.tile(np.arange(V), 4)
    lp = oracle.logprobs_fwd(rows, tg, lib=lib)[0].reshape(4, V)
    assert (lp <= 0).all(), "logp <= 0"
    _close(np.exp(lp).sum(1), np.ones(4), 1e-13, 0, "sum_t p_t = 1")
    _close(-(np.exp(lp) * lp).sum(1), H[:4], 1e-12, 1e-12, "H = -sum p logp")
    rows_b = np.repeat(b[:4], V, axis=0)
    lpb = oracle.logprobs_fwd(rows_b, tg, lib=lib)[0].reshape(4, V)
    klr = oracle.kl_fwd(a[:4], b[:4], oracle.REVERSE, lib=lib)[0]
    klf = oracle.kl_fwd(a[:4], b[:4], oracle.FORWARD, lib=lib)[0]
    _close((np.exp(lp) * (lp - lpb)).sum(1), klr, 1e-12, 1e-12, "KL(A||B) = E_a[logp_a - logp_b]")
    _close((np.exp(lpb) * (lpb - lp)).sum(1), klf, 1e-12, 1e-12, "KL(B||A) = E_b[logp_b - logp_a]")
    # gradients sum to zero along the row (shift invariance of every output)
    tg1 = np.random.default_rng(14).integers(0, V, N)
    for name, d in (("dlogp", oracle.logprobs_bwd(a, tg1, g, lib=lib)),
                    ("dH", oracle.entropy_bwd(a, g, lib=lib)),
                    *zip(("dA", "dB"), oracle.kl_bwd(a, b, g, oracle.REVERSE, lib=lib)),
                    *zip(("dA fwd", "dB fwd"), oracle.kl_bwd(a, b, g, oracle.FORWARD, lib=lib))):
        s = np.abs(d.sum(1))
        assert (s <= 1e-12 * (1 + np.abs(d).sum(1))).all(), f"{name} rows sum to 0"


def pin_shift_invariance(lib=None):
    N, V = 8, 513
    rng = np.random.default_rng(21)
    # multiples of 2^-20 so that x + c is exact in fp64
    a = np.round(rng.normal(0, 3, (N, V)) * 2**20) / 2**20
    b = np.round(rng.normal(0, 3, (N, V)) * 2**20) / 2**20
    b[0, 5] = -INF
    a[1, 7] = -INF
    tg = rng.integers(0, V, N)
    g = rng.normal(size=N)
    base = (oracle.entropy_fwd(a, lib=lib)[0], oracle.logprobs_fwd(a, tg, lib=lib)[0],
            oracle.kl_fwd(a, b, oracle.FORWARD, lib=lib)[0],
            oracle.entropy_bwd(a, g, lib=lib), oracle.logprobs_bwd(a, tg, g, lib=lib),
            *oracle.kl_bwd(a, b, g, oracle.FORWARD, lib=lib))
    for c in (1e4, 2.0**20, -1e4):
        a2, b2 = a + c, b - 0.5 * c
        got = (oracle.entropy_fwd(a2, lib=lib)[0], oracle.logprobs_fwd(a2, tg, lib=lib)[0],
               oracle.kl_fwd(a2, b2, oracle.FORWARD, lib=lib)[0],
               oracle.entropy_bwd(a2, g, lib=lib), oracle.logprobs_bwd(a2, tg, g, lib=lib),
               *oracle.kl_bwd(a2, b2, g, oracle.FORWARD, lib=lib))
        for i, (x, y) in enumerate(zip(got, base)):
            _close(x, y, 1e-12, 1e-12, f"shift {c} output {i}")


def pin_finite_differences(lib=None):
    V = 64
    a, b = _rand(31, 3, V, offset=2.0), _rand(32, 3, V, offset=2.0)
    g = np.array([1.0, -0.7, 0.3])
    tg = np.array([3, 17, 63])
    h = 1e-6

    def fd(f, x):
        out = np.empty_like(x)
        for j in range(V):
            xp, xm = x.copy(), x.copy()
            xp[:, j] += h
            xm[:, j] -= h
            out[:, j] = (f(xp) - f(xm)) / (2 * h)
        return out * g[:, None]

    checks = [
        ("dlogp", oracle.logprobs_bwd(a, tg, g, lib=lib), fd(lambda x: oracle.logprobs_fwd(x, tg, lib=lib)[0], a)),
        ("dH", oracle.entropy_bwd(a, g, lib=lib), fd(lambda x: oracle.entropy_fwd(x, lib=lib)[0], a)),
    ]
    for d in (oracle.REVERSE, oracle.FORWARD):
        da, db = oracle.kl_bwd(a, b, g, d, lib=lib)
        checks.append((f"dA dir{d}", da, fd(lambda x: oracle.kl_fwd(x, b, d, lib=lib)[0], a)))
        checks.append((f"dB dir{d}", db, fd(lambda x: oracle.kl_fwd(a, x, d, lib=lib)[0], b)))
    for name, got, ref in checks:
        _close(got, ref, 1e-8, 1e-6, f"finite differences {name}")


# ----------------------------------------------------------------------------
# Generalized JSD (reading R13: mix = beta q + (1 - beta) p,
# JSD = beta KL(q || mix) + (1 - beta) KL(p || mix); beta = 0 / 1 are the KL endpoints)
# ----------------------------------------------------------------------------
def _djsd(A, B, beta):
    beta = Decimal(beta)
    p, q = _dprobs(A), _dprobs(B)
    out = Decimal(0)
    for pi, qi in zip(p, q):
        mix = beta * qi + (1 - beta) * pi
        if qi > 0:
            out += beta * qi * (qi / mix).ln()
        if pi > 0:
            out += (1 - beta) * pi * (pi / mix).ln()
    return out


def pin_jsd_brute_force(lib=None):
    """Interior JSD and both gradients against Decimal, on rows with -inf entries."""
    with localcontext() as ctx:
        ctx.prec = 80
        for V in (2, 3, 6, 11):
            a = _tiny_rows(300 + V, V, 3, mask_frac=0.2 if V > 2 else 0.0)
            b = _tiny_rows(400 + V, V, 3, mask_frac=0.2 if V > 2 else 0.0)
            b += 1.5
            g = np.array([1.0, -0.6, 2.2])
            for beta in (0.2, 0.5, 0.83):
                J = oracle.jsd_fwd(a, b, beta, lib=lib)
                da, db = oracle.jsd_bwd(a, b, beta, g, lib=lib)
                for r in range(3):
                    A, B = list(a[r]), list(b[r])
                    _close(J[r], float(_djsd(A, B, beta)), 1e-14, 1e-13, f"JSD V={V} beta={beta}")
                    gr = Decimal(g[r])
                    ref_a = [float(gr * d) for d in _dgrad(lambda z: _djsd(z, B, beta), A)]
                    ref_b = [float(gr * d) for d in _dgrad(lambda z: _djsd(A, z, beta), B)]
                    _close(da[r], ref_a, 1e-13, 1e-12, f"dJSD/dA V={V} beta={beta}")
                    _close(db[r], ref_b, 1e-13, 1e-12, f"dJSD/dB V={V} beta={beta}")


def pin_jsd_closed_forms(lib=None):
    N, V = 6, 300
    a, b = _rand(61, N, V), _rand(62, N, V)
    g = np.linspace(-1.0, 1.5, N)
    for beta in (0.1, 0.5, 0.9):
        # identical inputs: 0, with zero gradients
        _close(oracle.jsd_fwd(a, a, beta, lib=lib), np.zeros(N), 1e-14, 0, f"JSD(A, A) beta={beta}")
        for d in oracle.jsd_bwd(a, a, beta, g, lib=lib):
            _close(d, np.zeros_like(d), 1e-15, 0, f"dJSD(A, A) beta={beta}")
        # disjoint supports: the entropy of the mixing weights, with zero gradients
        p, q = a.copy(), b.copy()
        p[:, V // 2:] = -INF
        q[:, :V // 2] = -INF
        hb = -beta * math.log(beta) - (1 - beta) * math.log(1 - beta)
        _close(oracle.jsd_fwd(p, q, beta, lib=lib), np.full(N, hb), 1e-14, 1e-14, f"disjoint beta={beta}")
        for d in oracle.jsd_bwd(p, q, beta, g, lib=lib):
            _close(d, np.zeros_like(d), 1e-14, 0, f"dJSD disjoint beta={beta}")
        # bounds and gradient rows summing to zero
        J = oracle.jsd_fwd(a, b, beta, lib=lib)
        assert (J >= 0).all() and (J <= hb + 1e-15).all(), "0 <= JSD <= H(beta)"
        for d in oracle.jsd_bwd(a, b, beta, g, lib=lib):
            assert (np.abs(d.sum(1)) <= 1e-13 * (1 + np.abs(d).sum(1))).all(), "dJSD rows sum to 0"
    # beta = 1/2 is symmetric in its arguments
    _close(oracle.jsd_fwd(a, b, 0.5, lib=lib), oracle.jsd_fwd(b, a, 0.5, lib=lib), 1e-15, 1e-14, "symmetry")
    da, db = oracle.jsd_bwd(a, b, 0.5, g, lib=lib)
    db2, da2 = oracle.jsd_bwd(b, a, 0.5, g, lib=lib)
    _close(da, da2, 1e-15, 1e-13, "symmetric dA")
    _close(db, db2, 1e-15, 1e-13, "symmetric dB")


def pin_jsd_endpoints(lib=None):
    """beta = 0 / 1 are the KL branches exactly; the interior tends to them at rate beta (1 - beta)."""
    N, V = 5, 257
    a, b = _rand(71, N, V, sigma=1.0, offset=0.5), _rand(72, N, V, sigma=1.0, offset=0.5)
    g = np.array([1.0, -2.0, 0.5, 0.3, -0.7])
    klf = oracle.kl_fwd(a, b, oracle.FORWARD, lib=lib)[0]      # KL(B || A)
    klr = oracle.kl_fwd(a, b, oracle.REVERSE, lib=lib)[0]      # KL(A || B)
    assert np.array_equal(oracle.jsd_fwd(a, b, 0.0, lib=lib), klf)
    assert np.array_equal(oracle.jsd_fwd(a, b, 1.0, lib=lib), klr)
    for got, ref in zip(oracle.jsd_bwd(a, b, 0.0, g, lib=lib), oracle.kl_bwd(a, b, g, oracle.FORWARD, lib=lib)):
        assert np.array_equal(got, ref)
    for got, ref in zip(oracle.jsd_bwd(a, b, 1.0, g, lib=lib), oracle.kl_bwd(a, b, g, oracle.REVERSE, lib=lib)):
        assert np.array_equal(got, ref)
    # the ratio's error is first order in beta (about 4.4 beta on these rows): take two steps
    for eps in (1e-6, 1e-7):
        _close(oracle.jsd_fwd(a, b, eps, lib=lib) / eps, klf, 0, 10 * eps, "JSD_beta / beta -> KL(B||A)")
        _close(oracle.jsd_fwd(a, b, 1 - eps, lib=lib) / eps, klr, 0, 10 * eps, "JSD_beta / (1 - beta) -> KL(A||B)")


def pin_jsd_special_rows(lib=None):
    V = 8
    base = np.linspace(-2.0, 1.5, V)
    a = np.tile(base, (4, 1))
    b = np.tile(base[::-1], (4, 1))
    a[0, 3] = NAN            # NaN in A
    b[1, 5] = INF            # +inf in B
    a[2, :] = -INF           # no finite logit in A
    b[3, :6] = -INF          # B supported on two entries only: finite JSD
    J = oracle.jsd_fwd(a, b, 0.4, lib=lib)
    da, db = oracle.jsd_bwd(a, b, 0.4, np.ones(4), lib=lib)
    assert np.isnan(J[:3]).all() and np.isfinite(J[3])
    assert np.isnan(da[:3]).all() and np.isnan(db[:3]).all()
    assert np.isfinite(da[3]).all() and (db[3, :6] == 0).all()


# ----------------------------------------------------------------------------
# Re-centring merge over host shards
# ----------------------------------------------------------------------------
def pin_shard_merge(lib=None):
    N, V = 12, 700
    a, b = _rand(41, N, V), _rand(42, N, V)
    a[0, 0:100] = -INF           # an all -inf first shard for row 0
    b[1, 350:] = -INF            # a masked tail in B
    a[1, 350:] = -INF            # ... that A also masks (no mismatch)
    a[2, :] += 1e4               # a large common offset
    b[2, :] -= 1e4
    a[3, 5] = 3e38               # extreme spread inside one row
    a[3, 6] = -3e38
    rng = np.random.default_rng(43)
    for k in (2, 3, 7):
        inner = np.sort(rng.integers(0, V, k - 1))
        if k == 7:
            inner[2] = inner[1]  # an empty shard
        cuts = np.concatenate([[0], inner, [V]])
        if k == 2:
            cuts = np.array([0, 100, V])  # row 0: first shard all -inf
        _close(oracle.entropy_sharded(a, cuts, lib=lib), oracle.entropy_fwd(a, lib=lib)[0],
               1e-13, 1e-13, f"entropy merge k={k}")
        recs = np.stack([oracle.shard_stats(a, cuts[s], cuts[s + 1], lib=lib) for s in range(k)])
        _close(oracle.merge_entropy_records(recs, lib=lib), oracle.entropy_fwd(a, lib=lib)[0],
               1e-13, 1e-13, f"entropy merge of gathered records k={k}")
        for d in (oracle.REVERSE, oracle.FORWARD):
            _close(oracle.kl_sharded(a, b, cuts, d, lib=lib), oracle.kl_fwd(a, b, d, lib=lib)[0],
                   1e-12, 1e-12, f"KL merge k={k} dir {d}")
            recs = np.stack([oracle.shard_kl_stats(a, b, cuts[s], cuts[s + 1], d, lib=lib) for s in range(k)])
            _close(oracle.merge_kl_records(recs, lib=lib), oracle.kl_fwd(a, b, d, lib=lib)[0],
                   1e-12, 1e-12, f"KL merge of gathered records k={k} dir {d}")


def pin_shard_records(lib=None):
    """Per-shard records (m, S, W, flags) against Decimal sums over the shard."""
    V = 13
    rng = np.random.default_rng(51)
    a, b = rng.normal(0, 3, (4, V)), rng.normal(0, 3, (4, V))
    a[1, 0:4] = -INF      # an all -inf shard [0, 4) in row 1
    b[2, 6] = -INF        # B masked where A is finite: a mismatch for KL(A||B)
    a[3, 9] = NAN         # a NaN in row 3

    def dsum(z, m, w=None):
        with localcontext() as ctx:
            ctx.prec = 60
            e = [Decimal(0) if v == -INF else (Decimal(v) - Decimal(m)).exp() for v in z]
            S = sum(e, Decimal(0))
            if w is None:
                return float(S), None
            W = sum((ei * wi for ei, wi in zip(e, w) if ei > 0), Decimal(0))
            return float(S), float(W)

    for lo, hi in ((0, 4), (4, 11), (11, 13), (0, 13)):
        got = oracle.shard_stats(a, lo, hi, lib=lib)
        for r in range(a.shape[0]):
            z = [float(v) for v in a[r, lo:hi]]
            bad = any(math.isnan(v) or v == INF for v in z)
            assert got[r, 3] == bad, f"shard [{lo},{hi}) row {r} bad flag"
            if bad:
                continue
            m = max(z)
            assert got[r, 0] == m, f"shard [{lo},{hi}) row {r} max"
            if m == -INF:
                assert got[r, 1] == 0 and got[r, 2] == 0, "all -inf shard has S = W = 0"
                continue
            S, W = dsum(z, m, [Decimal(v) - Decimal(m) if v != -INF else 0 for v in z])
            _close(got[r, 1], S, 0, 1e-14, f"shard [{lo},{hi}) row {r} S")
            _close(got[r, 2], W, 1e-14, 1e-13, f"shard [{lo},{hi}) row {r} W")
        for d in (oracle.REVERSE, oracle.FORWARD):
            got = oracle.shard_kl_stats(a, b, lo, hi, d, lib=lib)
            P, Q = (a, b) if d == oracle.REVERSE else (b, a)
            for r in range(a.shape[0]):
                p = [float(v) for v in P[r, lo:hi]]
                q = [float(v) for v in Q[r, lo:hi]]
                bad = any(math.isnan(v) or v == INF for v in p + q)
                flag = any(pj > -INF and qj == -INF for pj, qj in zip(p, q))
                what = f"KL dir {d} shard [{lo},{hi}) row {r}"
                assert got[r, 5] == bad and got[r, 6] == flag, what + " flags"
                if bad:
                    continue
                mp, mq = max(p), max(q)
                assert got[r, 0] == mp and got[r, 2] == mq, what + " maxima"
                if mp > -INF:
                    w = None if flag else [(Decimal(pj) - Decimal(mp)) - (Decimal(qj) - Decimal(mq))
                                           if pj != -INF else 0 for pj, qj in zip(p, q)]
                    Sp, W = dsum(p, mp, w)
                    _close(got[r, 1], Sp, 0, 1e-14, what + " S_P")
                    if W is not None:
                        _close(got[r, 4], W, 1e-14, 1e-13, what + " W")
                if mq > -INF:
                    _close(got[r, 3], dsum(q, mq)[0], 0, 1e-14, what + " S_Q")


# ----------------------------------------------------------------------------
# NaN / inf precedence and target rules (readings R2-R5 of the oracle header)
# ----------------------------------------------------------------------------
def pin_special_rows(lib=None):
    V = 6
    base = np.array([0.5, -1.0, 2.0, 0.0, -3.0, 1.0])
    rows = np.tile(base, (8, 1))
    rows[1, 2] = NAN              # NaN in the row
    rows[2, 4] = INF              # +inf in the row
    rows[3, :] = -INF             # all -inf
    rows[4, 1] = -INF             # a masked entry: finite result
    rows[5, :] = [-INF, -INF, 7.0, -INF, -INF, -INF]  # one-hot by masking
    rows[6, 0] = -1000.0          # an entry whose probability underflows in fp64
    H = oracle.entropy_fwd(rows, lib=lib)[0]
    assert np.isnan(H[1]) and np.isnan(H[2]) and np.isnan(H[3]), f"NaN rows {H}"
    assert np.isfinite(H[[0, 4, 5, 6, 7]]).all() and H[5] == 0.0, f"finite rows {H}"
    g = np.ones(8)
    dH = oracle.entropy_bwd(rows, g, lib=lib)
    assert np.isnan(dH[1:4]).all(), "NaN rows -> NaN gradient rows"
    assert np.isfinite(dH[[0, 4, 5, 6, 7]]).all() and dH[4, 1] == 0.0 and dH[6, 0] == 0.0, \
        "p_j = 0 positions get exactly 0"

    # logprobs targets: ignored, out of range, -inf target, NaN row, all -inf row
    vs = 100
    tg = np.array([vs + 2, vs + 0, vs + 1, vs + 1, vs + 1, -1, vs + V, vs - 1])
    lp, _, _, err = oracle.logprobs_fwd(rows, tg, vocab_start=vs, lib=lib)
    assert np.isfinite(lp[0]) and np.isnan(lp[1]) and np.isnan(lp[2]) and np.isnan(lp[3])
    assert lp[4] == -INF, "target on a -inf logit gives -inf"
    assert lp[5] == 0.0, "ignored target gives 0"
    assert np.isnan(lp[6]) and np.isnan(lp[7]) and err == oracle.ERR_TARGET, "out-of-range targets"
    lp_ok, _, _, err_ok = oracle.logprobs_fwd(rows[[0]], [vs + 2], vocab_start=vs, lib=lib)
    assert err_ok == 0 and lp_ok[0] == lp[0]
    dl = oracle.logprobs_bwd(rows, tg, g, vocab_start=vs, lib=lib)
    assert (dl[5] == 0).all(), "ignored target: zero gradient row"
    assert np.isnan(dl[[1, 2, 3, 6, 7]]).all(), "NaN / error rows: NaN gradient rows"
    assert np.isfinite(dl[[0, 4]]).all() and dl[4, 1] == 1.0, "-inf target: gradient g at the target"

    # KL precedence: NaN beats mismatch, all -inf P is NaN, mismatch beats the formula
    P = np.tile(base, (7, 1))
    Q = np.tile(base[::-1], (7, 1))
    Q[1, 3] = -INF                 # mismatch: P supports j=3
    Q[2, 3] = -INF
    P[2, 0] = NAN                  # ... but P has a NaN -> NaN
    P[3, :] = -INF                 # all -inf P -> NaN (Q finite)
    Q[4, :] = -INF                 # all -inf Q, finite P -> mismatch -> +inf
    P[5, 0] = -1000.0              # p underflows, Q masks it -> still a mismatch
    Q[5, 0] = -INF
    P[6, 2] = -INF                 # both masked at the same place -> finite
    Q[6, 2] = -INF
    kl = oracle.kl_fwd(P, Q, oracle.REVERSE, lib=lib)[0]
    assert np.isfinite(kl[0]) and kl[1] == INF and np.isnan(kl[2]) and np.isnan(kl[3])
    assert kl[4] == INF and kl[5] == INF and np.isfinite(kl[6]), f"KL precedence {kl}"
    kl_swapped = oracle.kl_fwd(Q, P, oracle.FORWARD, lib=lib)[0]
    _close(kl_swapped, kl, 0, 0, "forward with swapped arguments = reverse")
    dP, dQ = oracle.kl_bwd(P, Q, np.ones(7), oracle.REVERSE, lib=lib)
    assert np.isnan(dP[[1, 2, 3, 4, 5]]).all(), "flagged / NaN rows: NaN dP"
    assert np.isfinite(dQ[[1, 5]]).all(), "flagged rows: finite dQ"
    assert np.isnan(dQ[[2, 3, 4]]).all(), "NaN rows and an undefined q: NaN dQ"
    assert np.isfinite(dP[[0, 6]]).all() and dP[6, 2] == 0.0 and dQ[6, 2] == 0.0


# ----------------------------------------------------------------------------
# Fused linear logp
# ----------------------------------------------------------------------------
def _linear_case(seed, N, V, D):
    rng = np.random.default_rng(seed)
    h = rng.normal(0, 1, (N, D))
    W = rng.normal(0, 0.5, (V, D))
    tg = rng.integers(0, V, N)
    g = rng.normal(size=N)
    return h, W, tg, g


def pin_linear_logp_brute_force(lib=None):
    h, W, tg, g = _linear_case(51, 3, 5, 4)
    lp = oracle.linear_logp_fwd(h, W, tg + 10, vocab_start=10, lib=lib)[0]
    with localcontext() as ctx:
        ctx.prec = 60
        for r in range(3):
            z = [sum((Decimal(h[r, k]) * Decimal(W[j, k]) for k in range(4)), Decimal(0)) for j in range(5)]
            _close(lp[r], float(_dlogp(z, tg[r])), 1e-14, 1e-14, "linear logp brute force")
    logits = oracle.linear_logits(h, W, lib=lib)
    ref = np.array([[float(sum(Decimal(h[r, k]) * Decimal(W[j, k]) for k in range(4))) for j in range(5)]
                    for r in range(3)])
    _close(logits, ref, 1e-14, 1e-14, "linear logits")


def pin_linear_logp_finite_differences(lib=None):
    N, V, D = 3, 5, 4
    h, W, tg, g = _linear_case(52, N, V, D)
    dh, dW = oracle.linear_logp_bwd(h, W, tg, g, lib=lib)
    f = lambda hh, WW: float(np.dot(g, oracle.linear_logp_fwd(hh, WW, tg, lib=lib)[0]))
    eps = 1e-6
    ref_dh = np.empty_like(h)
    for r in range(N):
        for k in range(D):
            hp, hm = h.copy(), h.copy()
            hp[r, k] += eps
            hm[r, k] -= eps
            ref_dh[r, k] = (f(hp, W) - f(hm, W)) / (2 * eps)
    ref_dW = np.empty_like(W)
    for j in range(V):
        for k in range(D):
            Wp, Wm = W.copy(), W.copy()
            Wp[j, k] += eps
            Wm[j, k] -= eps
            ref_dW[j, k] = (f(h, Wp) - f(h, Wm)) / (2 * eps)
    _close(dh, ref_dh, 1e-8, 1e-6, "linear dhidden FD")
    _close(dW, ref_dW, 1e-8, 1e-6, "linear dW FD")
    # the materialise-then-logprobs path agrees (wiring of the fused oracle)
    logits = oracle.linear_logits(h, W, lib=lib)
    _close(oracle.linear_logp_fwd(h, W, tg, lib=lib)[0], oracle.logprobs_fwd(logits, tg, lib=lib)[0],
           1e-14, 1e-14, "linear logp = logprobs(logits)")


def pin_linear_row_stats(lib=None):
    """The block-wise normalisers (row max and log-sum-exp of h . W^T) against Decimal sums, with
    blocks of 2 rows over 5 rows (a ragged last block), and against the per-row oracle."""
    N, V, D = 5, 7, 4
    h, W, _, _ = _linear_case(53, N, V, D)
    h[3] += 40.0                                     # one row with a large spread
    m, ls = oracle.linear_row_stats(h, W, rows_per_block=2)
    with localcontext() as ctx:
        ctx.prec = 60
        for r in range(N):
            z = [sum((Decimal(h[r, k]) * Decimal(W[j, k]) for k in range(D)), Decimal(0)) for j in range(V)]
            zm = max(z)
            _close(m[r], float(zm), 1e-14, 1e-14, "linear row max")
            _close(ls[r], float(sum(_dexp(x - zm) for x in z).ln()), 1e-14, 1e-14, "linear row log S")
    tg = np.arange(N) % V
    _, m2, ls2, _ = oracle.linear_logp_fwd(h, W, tg, lib=lib)
    _close(m, m2, 1e-13, 1e-13, "row stats vs per-row oracle (max)")
    _close(ls, ls2, 1e-13, 1e-13, "row stats vs per-row oracle (log S)")
    # selected rows of dW equal those of the full backward (finite-difference pinned), an
    # ignored target included; the shard starts at vocab_start
    tg[2] = -1
    g = np.linspace(-1.0, 2.0, N)
    _, dW = oracle.linear_logp_bwd(h, W, tg + 100 * (tg >= 0), g, vocab_start=100, lib=lib)
    ids = [0, 3, 6]
    rows, _ = oracle.linear_logp_dW_rows(h, W, tg + 100 * (tg >= 0), g, ids, vocab_start=100)
    _close(rows, dW[ids], 1e-13, 1e-12, "selected dW rows")


# ----------------------------------------------------------------------------
# Fused linear entropy and KL (two models with their own hidden size)
# ----------------------------------------------------------------------------
def _two_models(seed, N, V, Da, Db):
    rng = np.random.default_rng(seed)
    return (rng.normal(0, 1, (N, Da)), rng.normal(0, 0.6, (V, Da)), rng.normal(0, 1, (N, Db)),
            rng.normal(0, 0.6, (V, Db)), rng.normal(size=N))


def _dlogits(h, W):
    return [[sum((Decimal(h[r, k]) * Decimal(W[j, k]) for k in range(h.shape[1])), Decimal(0))
             for j in range(W.shape[0])] for r in range(h.shape[0])]


def pin_linear_entropy_kl_brute_force(lib=None):
    ha, Wa, hb, Wb, _ = _two_models(61, 3, 5, 4, 6)
    H = oracle.linear_entropy_fwd(ha, Wa, lib=lib)[0]
    rev = oracle.linear_kl_fwd(ha, Wa, hb, Wb, oracle.REVERSE, lib=lib)[0]
    fwd = oracle.linear_kl_fwd(ha, Wa, hb, Wb, oracle.FORWARD, lib=lib)[0]
    with localcontext() as ctx:
        ctx.prec = 60
        za, zb = _dlogits(ha, Wa), _dlogits(hb, Wb)
        for r in range(3):
            _close(H[r], float(_dentropy(za[r])), 1e-14, 1e-14, "linear entropy brute force")
            _close(rev[r], float(_dkl(za[r], zb[r])), 1e-14, 1e-13, "linear KL(A||B) brute force")
            _close(fwd[r], float(_dkl(zb[r], za[r])), 1e-14, 1e-13, "linear KL(B||A) brute force")


def _fd(f, x, eps=1e-6):
    out = np.empty_like(x)
    for i in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[i] += eps
        xm[i] -= eps
        out[i] = (f(xp) - f(xm)) / (2 * eps)
    return out


def pin_linear_entropy_kl_finite_differences(lib=None):
    ha, Wa, hb, Wb, g = _two_models(62, 3, 5, 3, 4)
    dh, dW = oracle.linear_entropy_bwd(ha, Wa, g, lib=lib)
    H = lambda h, W: float(np.dot(g, oracle.linear_entropy_fwd(h, W, lib=lib)[0]))
    _close(dh, _fd(lambda x: H(x, Wa), ha), 1e-8, 1e-6, "linear entropy dhidden FD")
    _close(dW, _fd(lambda x: H(ha, x), Wa), 1e-8, 1e-6, "linear entropy dW FD")
    for d in (oracle.REVERSE, oracle.FORWARD):
        dha, dWa, dhb, dWb = oracle.linear_kl_bwd(ha, Wa, hb, Wb, g, d, lib=lib)
        K = lambda a, b, c, e: float(np.dot(g, oracle.linear_kl_fwd(a, b, c, e, d, lib=lib)[0]))
        _close(dha, _fd(lambda x: K(x, Wa, hb, Wb), ha), 1e-8, 1e-6, f"linear KL dir {d} dha FD")
        _close(dWa, _fd(lambda x: K(ha, x, hb, Wb), Wa), 1e-8, 1e-6, f"linear KL dir {d} dWa FD")
        _close(dhb, _fd(lambda x: K(ha, Wa, x, Wb), hb), 1e-8, 1e-6, f"linear KL dir {d} dhb FD")
        _close(dWb, _fd(lambda x: K(ha, Wa, hb, x), Wb), 1e-8, 1e-6, f"linear KL dir {d} dWb FD")


def pin_linear_entropy_kl_closed_forms(lib=None):
    N, V, D = 4, 7, 5
    ha, Wa, hb, Wb, g = _two_models(63, N, V, D, D + 2)
    # a zero LM head: uniform distribution, H = log V, zero gradients
    H = oracle.linear_entropy_fwd(ha, np.zeros((V, D)), lib=lib)[0]
    _close(H, np.full(N, math.log(V)), 1e-15, 1e-15, "linear entropy of a zero head")
    dh, dW = oracle.linear_entropy_bwd(ha, np.zeros((V, D)), g, lib=lib)
    _close(dh, np.zeros_like(dh), 1e-15, 0, "zero-head entropy dhidden")
    _close(dW, np.zeros_like(dW), 1e-15, 0, "zero-head entropy dW")
    # model B = model A with two extra hidden units that its head ignores: KL = 0, gradients 0
    hpad = np.concatenate([ha, hb[:, :2]], 1)
    Wpad = np.concatenate([Wa, np.zeros((V, 2))], 1)
    for d in (oracle.REVERSE, oracle.FORWARD):
        assert (oracle.linear_kl_fwd(ha, Wa, hpad, Wpad, d, lib=lib)[0] == 0).all(), "KL of a model with itself"
        for o in oracle.linear_kl_bwd(ha, Wa, hpad, Wpad, g, d, lib=lib):
            assert (o == 0).all(), "gradients of KL of a model with itself"
    # forward KL of (A, B) is reverse KL of (B, A)
    _close(oracle.linear_kl_fwd(ha, Wa, hb, Wb, oracle.FORWARD, lib=lib)[0],
           oracle.linear_kl_fwd(hb, Wb, ha, Wa, oracle.REVERSE, lib=lib)[0], 1e-15, 1e-15, "KL direction swap")


def pin_linear_jsd(lib=None):
    """Fused linear JSD: Decimal brute force, finite differences of all four gradients, the
    endpoints as the linear KL calls, and a model against itself."""
    ha, Wa, hb, Wb, g = _two_models(64, 3, 5, 3, 4)
    with localcontext() as ctx:
        ctx.prec = 60
        za, zb = _dlogits(ha, Wa), _dlogits(hb, Wb)
        for beta in (0.25, 0.7):
            got = oracle.linear_jsd_fwd(ha, Wa, hb, Wb, beta, lib=lib)
            for r in range(3):
                _close(got[r], float(_djsd(za[r], zb[r], beta)), 1e-14, 1e-12, f"linear JSD brute force beta={beta}")
    beta = 0.4
    grads = oracle.linear_jsd_bwd(ha, Wa, hb, Wb, beta, g, lib=lib)
    J = lambda a, b, c, e: float(np.dot(g, oracle.linear_jsd_fwd(a, b, c, e, beta, lib=lib)))
    refs = (_fd(lambda x: J(x, Wa, hb, Wb), ha), _fd(lambda x: J(ha, x, hb, Wb), Wa),
            _fd(lambda x: J(ha, Wa, x, Wb), hb), _fd(lambda x: J(ha, Wa, hb, x), Wb))
    for got, ref, name in zip(grads, refs, ("dha", "dWa", "dhb", "dWb")):
        _close(got, ref, 1e-8, 1e-6, f"linear JSD {name} FD")
    # the endpoints are the KL calls: beta = 0 is KL(B || A), beta = 1 is KL(A || B)
    _close(oracle.linear_jsd_fwd(ha, Wa, hb, Wb, 0.0, lib=lib),
           oracle.linear_kl_fwd(ha, Wa, hb, Wb, oracle.FORWARD, lib=lib)[0], 1e-15, 1e-15, "linear JSD beta = 0")
    _close(oracle.linear_jsd_fwd(ha, Wa, hb, Wb, 1.0, lib=lib),
           oracle.linear_kl_fwd(ha, Wa, hb, Wb, oracle.REVERSE, lib=lib)[0], 1e-15, 1e-15, "linear JSD beta = 1")
    # a model against itself: JSD = 0 and zero gradients
    _close(oracle.linear_jsd_fwd(ha, Wa, ha, Wa, 0.5, lib=lib), np.zeros(3), 1e-15, 0,
           "linear JSD of a model with itself")   # mix = p up to one rounding
    for o in oracle.linear_jsd_bwd(ha, Wa, ha, Wa, 0.5, g, lib=lib):
        _close(o, np.zeros_like(o), 1e-15, 0, "linear JSD gradients of a model with itself")


ALL_PINS = [
    pin_brute_force_fwd,
    pin_brute_force_grads,
    pin_topk_targets,
    pin_uniform_row,
    pin_two_token_closed_form,
    pin_one_hot_extremes,
    pin_invariants,
    pin_shift_invariance,
    pin_finite_differences,
    pin_shard_merge,
    pin_shard_records,
    pin_special_rows,
    pin_jsd_brute_force,
    pin_jsd_closed_forms,
    pin_jsd_endpoints,
    pin_jsd_special_rows,
    pin_linear_logp_brute_force,
    pin_linear_logp_finite_differences,
    pin_linear_row_stats,
    pin_linear_entropy_kl_brute_force,
    pin_linear_entropy_kl_finite_differences,
    pin_linear_entropy_kl_closed_forms,
    pin_linear_jsd,
]
