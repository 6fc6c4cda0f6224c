"""GPU parity of the vocabulary-sharded fused linear ops against the fp64 oracle of
the unsharded rows.

K shards of the head's rows (boundaries off every tile edge) each write their
records (vp_linear_*_partial); vp_*_merge turns the gathered records into the
outputs and row statistics, which must match the unsharded oracle at the
output tolerance. Each shard's backward with the merged records must give its
rows of dW and its term dz_k . W_k of dhidden (the caller adds the terms), both
at the fused-linear gradient tolerance (parity.check_gemm_grad).
"""
import numpy as np
import pytest
import torch

import oracle
import vocab_wide_logprobs_gb300 as vp
from tests import parity
from tests.test_gpu_linear_ent_kl import _model, _probs

pytestmark = pytest.mark.gpu
DEV = "cuda"
N, V = 200, 1000
CUTS = [(0, 300), (300, 777), (777, 1000)]   # 3 shards, none on a 64- or 256-column edge


def _targets(seed):
    rng = np.random.default_rng(seed)
    t = rng.integers(0, V, N).astype(np.int64)
    t[::17] = -1                                   # ignored
    t[1:6] = [299, 300, 776, 777, 999]             # shard edges
    return torch.from_numpy(t)


def _check_terms(dh_k, dW_k, dz, Mz, h64, W64, v0, v1, tag):
    """dW rows [v0, v1) and the shard's dhidden term dz[:, v0:v1] . W[v0:v1]."""
    dzk, Mk, Wk = dz[:, v0:v1], Mz[:, v0:v1], W64[v0:v1]
    adz = np.abs(dzk)
    parity.check_gemm_grad(dh_k, dzk @ Wk, parity.gemm_norms(adz, Wk), f"{tag} dhidden term", Mk @ np.abs(Wk))
    parity.check_gemm_grad(dW_k, dzk.T @ h64, parity.gemm_norms(adz.T, h64), f"{tag} dW rows", Mk.T @ np.abs(h64))


def test_linear_logp_sharded():
    D = 128
    h, W, g = _model(81, N, V, D)
    t = _targets(82)
    hd, Wd, td, gd = h.to(DEV), W.to(DEV), t.to(DEV), g.to(DEV)
    parts = vp.partials(N, DEV, K=len(CUTS))
    for k, (v0, v1) in enumerate(CUTS):
        vp.vp_linear_logp_partial(hd, Wd[v0:v1], td, vocab_start=v0, parts=parts[k])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    logp, st = vp.vp_logprobs_merge(parts, err_word=err)
    grads = [vp.vp_linear_logp_bwd(hd, Wd[v0:v1], td, st, gd, vocab_start=v0) for v0, v1 in CUTS]
    torch.cuda.synchronize()
    h64, W64, g64 = parity.to64(h), parity.to64(W), g.double().numpy()
    rlp, rm, rls, rerr = oracle.linear_logp_fwd(h64, W64, t.numpy())
    parity.check_out(logp, rlp, "sharded linear logp")
    d = vp.decode_rowstats(st)
    parity.check_out(d["m"], rm, "sharded max logit")
    parity.check_out(d["logS"], rls, "sharded logS")
    assert int(err.item()) == 0 and not rerr
    z = oracle.linear_logits(h64, W64)
    dz = oracle.logprobs_bwd(z, t.numpy(), g64)
    Mz = parity.oracle_all(z, z, t.numpy(), g64, ops=("logprobs",))["_mag"]["dlogp"]
    for (dh_k, dW_k), (v0, v1) in zip(grads, CUTS):
        _check_terms(dh_k, dW_k, dz, Mz, h64, W64, v0, v1, f"logp shard [{v0}, {v1})")


def test_linear_logp_sharded_target_in_no_shard():
    """A target >= 0 that no shard holds: NaN logp, the error bit, NaN gradient rows in every shard."""
    D = 64
    h, W, g = _model(83, N, V, D)
    t = _targets(84)
    t[11] = V + 5
    hd, Wd, td, gd = h.to(DEV), W.to(DEV), t.to(DEV), g.to(DEV)
    parts = vp.partials(N, DEV, K=len(CUTS))
    for k, (v0, v1) in enumerate(CUTS):
        vp.vp_linear_logp_partial(hd, Wd[v0:v1], td, vocab_start=v0, parts=parts[k])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    logp, st = vp.vp_logprobs_merge(parts, err_word=err)
    grads = [vp.vp_linear_logp_bwd(hd, Wd[v0:v1], td, st, gd, vocab_start=v0) for v0, v1 in CUTS]
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    assert torch.isnan(logp[11]) and torch.isfinite(logp[:11]).all() and torch.isfinite(logp[12:]).all()
    assert vp.decode_rowstats(st)["flags"][11] & vp.ROW_BADTARGET
    for dh_k, dW_k in grads:
        assert torch.isnan(dh_k[11]).all() and torch.isfinite(dh_k[:11]).all() and torch.isnan(dW_k).all()


def test_linear_entropy_sharded():
    D = 128
    h, W, g = _model(85, N, V, D)
    hd, Wd, gd = h.to(DEV), W.to(DEV), g.to(DEV)
    parts = vp.partials(N, DEV, K=len(CUTS))
    for k, (v0, v1) in enumerate(CUTS):
        vp.vp_linear_entropy_partial(hd, Wd[v0:v1], parts=parts[k])
    H, st = vp.vp_entropy_merge(parts)
    grads = [vp.vp_linear_entropy_bwd(hd, Wd[v0:v1], st, gd) for v0, v1 in CUTS]
    torch.cuda.synchronize()
    h64, W64, g64 = parity.to64(h), parity.to64(W), g.double().numpy()
    rH, rm, rls = oracle.linear_entropy_fwd(h64, W64)
    parity.check_out(H, rH, "sharded linear H")
    d = vp.decode_rowstats(st)
    parity.check_out(d["m"], rm, "sharded max logit")
    parity.check_out(d["logS"], rls, "sharded logS")
    z = oracle.linear_logits(h64, W64)
    dz = oracle.entropy_bwd(z, g64)
    Mz = parity.oracle_all(z, z, np.zeros(N, np.int64), g64, ops=("entropy",))["_mag"]["dH"]
    Mz = Mz * (1.0 + parity.logit_scale((h64, W64)))[:, None]
    for (dh_k, dW_k), (v0, v1) in zip(grads, CUTS):
        _check_terms(dh_k, dW_k, dz, Mz, h64, W64, v0, v1, f"entropy shard [{v0}, {v1})")


@pytest.mark.parametrize("direction", [vp.KL_REVERSE, vp.KL_FORWARD], ids=["reverse", "forward"])
def test_linear_kl_sharded(direction):
    Da, Db = 128, 64
    ha, Wa, g = _model(87, N, V, Da)
    hb, Wb, _ = _model(88, N, V, Db, scale=20.0)
    dev = [x.to(DEV) for x in (ha, Wa, hb, Wb, g)]
    parts = vp.partials(N, DEV, K=len(CUTS))
    for k, (v0, v1) in enumerate(CUTS):
        vp.vp_linear_kl_partial(dev[0], dev[1][v0:v1], dev[2], dev[3][v0:v1], direction, parts=parts[k])
    kl, sa, sb = vp.vp_kl_merge(parts, direction)
    grads = [vp.vp_linear_kl_bwd(dev[0], dev[1][v0:v1], dev[2], dev[3][v0:v1], direction, sa, sb, dev[4])
             for v0, v1 in CUTS]
    torch.cuda.synchronize()
    ha64, Wa64, hb64, Wb64 = (parity.to64(x) for x in (ha, Wa, hb, Wb))
    g64 = g.double().numpy()
    rkl, rma, rla, rmb, rlb = oracle.linear_kl_fwd(ha64, Wa64, hb64, Wb64, direction)
    parity.check_out(kl, rkl, f"sharded linear KL dir={direction}")
    for st, rm, rl, name in ((sa, rma, rla, "A"), (sb, rmb, rlb, "B")):
        d = vp.decode_rowstats(st)
        parity.check_out(d["m"], rm, f"sharded max logit of {name}")
        parity.check_out(d["logS"], rl, f"sharded logS of {name}")
    za, zb = oracle.linear_logits(ha64, Wa64), oracle.linear_logits(hb64, Wb64)
    dza, dzb = oracle.kl_bwd(za, zb, g64, direction)
    op = "kl_rev" if direction == vp.KL_REVERSE else "kl_fwd"
    M = parity.oracle_all(za, zb, np.zeros(N, np.int64), g64, ops=(op,))["_mag"]
    lam = (1.0 + parity.logit_scale((ha64, Wa64), (hb64, Wb64)))[:, None]
    M = {k: v * lam for k, v in M.items()}
    pa, pb = _probs(za), _probs(zb)
    assert min(pa.min(), pb.min()) > parity.TINY, "no probability of this case is flushed"
    for (dha, dwa, dhb, dwb), (v0, v1) in zip(grads, CUTS):
        tag = f"KL dir={direction} shard [{v0}, {v1})"
        _check_terms(dha, dwa, dza, M["d" + op + "_a"], ha64, Wa64, v0, v1, tag + " model A")
        _check_terms(dhb, dwb, dzb, M["d" + op + "_b"], hb64, Wb64, v0, v1, tag + " model B")


def test_linear_sharded_single_shard_equals_unsharded():
    """K = 1: the partial-merge path gives the unsharded forward's outputs and records."""
    D = 64
    h, W, _ = _model(89, N, V, D)
    t = _targets(90)
    hd, Wd, td = h.to(DEV), W.to(DEV), t.to(DEV)
    parts = vp.vp_linear_logp_partial(hd, Wd, td).unsqueeze(0)
    logp, st = vp.vp_logprobs_merge(parts)
    ref, rst = vp.vp_linear_logp_fwd(hd, Wd, td)
    eparts = vp.vp_linear_entropy_partial(hd, Wd).unsqueeze(0)
    H, _ = vp.vp_entropy_merge(eparts)
    rH, _ = vp.vp_linear_entropy_fwd(hd, Wd)
    torch.cuda.synchronize()
    parity.check_out(logp, ref.double().cpu().numpy(), "K = 1 logp")
    parity.check_out(H, rH.double().cpu().numpy(), "K = 1 H")
    d, rd = vp.decode_rowstats(st), vp.decode_rowstats(rst)
    assert torch.equal(d["m"], rd["m"])


def test_linear_partial_records_match_the_oracle_shard_sums():
    """Each shard's records field by field against the oracle's sums over the same columns of the
    fp64 logits: maxima and target logits at the output tolerance, S and W to 5e-5 (the GEMM's
    logits are fp32 accumulations, so the records are not bitwise the fp64 ones)."""
    D = 128
    h, W, _ = _model(91, N, V, D)
    t = _targets(92)
    hd, Wd, td = h.to(DEV), W.to(DEV), t.to(DEV)
    z = oracle.linear_logits(parity.to64(h), parity.to64(W))
    tt = t.numpy()
    for v0, v1 in CUTS:
        lrec = vp.decode_partials(vp.vp_linear_logp_partial(hd, Wd[v0:v1], td, vocab_start=v0))
        erec = vp.decode_partials(vp.vp_linear_entropy_partial(hd, Wd[v0:v1]))
        torch.cuda.synchronize()
        ref = oracle.shard_stats(z, v0, v1)                       # m, S, W, bad
        assert not ref[:, 3].any()
        for rec, name in ((lrec, "logp"), (erec, "entropy")):
            tag = f"{name} shard [{v0}, {v1})"
            parity.check_out(rec["m"], ref[:, 0], f"{tag} max")
            assert np.allclose(rec["S"].cpu().numpy(), ref[:, 1], rtol=5e-5, atol=0), f"{tag} S"
            assert (rec["flags"].cpu().numpy() & vp.PART_NANINF == 0).all()
        Wg = erec["W"].cpu().numpy()
        assert (np.abs(Wg - ref[:, 2]) <= 5e-5 * (np.abs(ref[:, 2]) + ref[:, 1])).all(), "shard W"
        assert (lrec["W"].cpu().numpy() == 0).all()
        has = (tt >= v0) & (tt < v1)
        lfl = lrec["flags"].cpu().numpy()
        assert (((lfl & vp.PART_HAS_TARGET) != 0) == has).all()
        assert (((lfl & vp.PART_IGNORED) != 0) == (tt < 0)).all()
        rows = np.nonzero(has)[0]
        parity.check_out(lrec["z_t"][torch.from_numpy(rows).to(DEV)], z[rows, tt[rows]], "target logit")
