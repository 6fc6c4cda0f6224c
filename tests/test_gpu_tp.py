"""GPU parity of the vocabulary-sharded forms: per-shard records, merge, and the
ordinary backward on each shard with the merged records, against the fp64
oracle of the whole (unsharded) rows, element by element.

Shards are column slices of the same logits read in place (so a shard's rows
start off the 16-byte grid: the scalar head and tail paths run), with empty
-inf shards, NaN and +-3e38 rows, large offsets, support mismatches, ignored,
out-of-range and boundary targets.
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


def _inputs(N, V, dtype, seed, cuts):
    w = workloads.pages_shape(seed=seed, N=N, V=V, dtype=torch.float32)
    a, b, t, g = w["a"], w["b"], w["targets"].clone(), w["grad"]
    c1 = cuts[1]
    a[0, :c1] = float("-inf")                  # shard 0 of row 0 has no finite logit
    b[0, :c1] = float("-inf")
    a[1, V // 2] = float("nan")                # a NaN row
    a[2] += 1e4 if dtype == torch.float32 else 200.0   # a large common offset
    b[2] += 1e4 if dtype == torch.float32 else 200.0
    b[3, min(c1 + 1, V - 1)] = float("-inf")   # B masked where A is finite: KL(A||B) = +inf
    a[4] = -3e38                               # one-hot row spanning +-3e38
    a[4, 5] = 3e38
    b[4] = a[4]
    t[5] = -1                                  # ignored target
    t[6] = V + 3                               # target in no shard: data error
    t[7] = c1 - 1                              # targets on both sides of a shard boundary
    t[8] = c1 if c1 < V else 0
    return a.to(dtype), b.to(dtype), t, g


def _sharded(a, b, t, g, cuts):
    """The sharded flow on one GPU: partial per shard, gather (stack), merge, backward per shard."""
    K = len(cuts) - 1
    sl = [slice(cuts[k], cuts[k + 1]) for k in range(K)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = {}
    parts = torch.stack([vp.vp_logprobs_partial(a[:, s], t, s.start) for s in sl])
    lp, st = vp.vp_logprobs_merge(parts, err_word=err)
    out.update(logp=lp, logp_stats=st, err=err, _lp_parts=parts)
    out["dlogp"] = torch.cat([vp.vp_logprobs_bwd(a[:, s], t, st, g, s.start, err_word=err) for s in sl], 1)
    parts = torch.stack([vp.vp_entropy_partial(a[:, s]) for s in sl])
    H, st = vp.vp_entropy_merge(parts)
    out.update(H=H, H_stats=st, _H_parts=parts)
    out["dH"] = torch.cat([vp.vp_entropy_bwd(a[:, s], st, g) for s in sl], 1)
    for name, d in (("kl_rev", vp.KL_REVERSE), ("kl_fwd", vp.KL_FORWARD)):
        parts = torch.stack([vp.vp_kl_partial(a[:, s], b[:, s], d) for s in sl])
        kl, sa, sb = vp.vp_kl_merge(parts, d)
        out[name], out[name + "_sa"], out[name + "_sb"], out["_" + name + "_parts"] = kl, sa, sb, parts
        grads = [vp.vp_kl_bwd(a[:, s], b[:, s], d, sa, sb, g) for s in sl]
        out["d" + name + "_a"] = torch.cat([x[0] for x in grads], 1)
        out["d" + name + "_b"] = torch.cat([x[1] for x in grads], 1)
    torch.cuda.synchronize()
    return out


CASES = [
    (40, 20011, torch.bfloat16, (0, 7001, 13003, 20011)),
    (40, 20011, torch.float32, (0, 7001, 13003, 20011)),
    (24, 75968, torch.bfloat16, (0, 37984, 75968)),
    (16, 9000, torch.bfloat16, (0, 1, 4000, 4001, 9000)),   # one-column shards
    (12, 5003, torch.float32, (0, 5003)),                   # K = 1
]


@pytest.mark.parametrize("N,V,dtype,cuts", CASES, ids=[f"{n}x{v}-{str(d)[6:]}-K{len(c) - 1}" for n, v, d, c in CASES])
def test_sharded_flow_matches_unsharded_oracle(N, V, dtype, cuts):
    a, b, t, g = _inputs(N, V, dtype, seed=N + V, cuts=cuts)
    a, b, t, g = a.to(DEV), b.to(DEV), t.to(DEV), g.to(DEV)
    got = _sharded(a, b, t, g, list(cuts))
    a64, b64 = parity.to64(a), parity.to64(b)
    ref = parity.oracle_all(a64, b64, t.cpu().numpy(), g.cpu().numpy())
    worst = parity.compare_all(got, ref, tag=f"sharded {N}x{V} K={len(cuts) - 1} ")
    assert int(got["err"].item()) == ref["err"] == 1
    flags = vp.decode_rowstats(got["logp_stats"])["flags"].cpu().numpy()
    assert (flags & vp.ROW_SHARDED).all() and flags[6] & vp.ROW_BADTARGET
    assert not (np.delete(flags, 6) & vp.ROW_BADTARGET).any()
    print("sharded worst/tol:", {k: round(v, 3) for k, v in worst.items()})


def test_partial_records_match_their_definition():
    """Each shard's record (max, sum-exp, centred weighted sum, flags) against the oracle's shard sums."""
    N, V, cuts = 40, 20011, (0, 7001, 13003, 20011)
    for dtype in (torch.bfloat16, torch.float32):
        a, b, t, g = _inputs(N, V, dtype, seed=5, cuts=cuts)
        a64, b64 = parity.to64(a), parity.to64(b)
        a, b, t = a.to(DEV), b.to(DEV), t.to(DEV)
        rtol = 2e-5 if dtype == torch.bfloat16 else 2e-6
        for k in range(len(cuts) - 1):
            lo, hi = cuts[k], cuts[k + 1]
            rec = vp.decode_partials(vp.vp_entropy_partial(a[:, lo:hi]))
            ref = oracle.shard_stats(a64, lo, hi)
            fl = rec["flags"].cpu().numpy()
            bad = ref[:, 3] != 0
            assert ((fl & vp.PART_NANINF) != 0).tolist() == bad.tolist()
            m = rec["m"].double().cpu().numpy()
            fin = ~bad & np.isfinite(ref[:, 0])
            assert (m[fin] == ref[fin, 0]).all(), "shard max"
            assert (m[~bad & ~np.isfinite(ref[:, 0])] == -np.finfo(np.float32).max).all()
            S, W = rec["S"].cpu().numpy(), rec["W"].cpu().numpy()
            assert np.allclose(S[fin], ref[fin, 1], rtol=rtol, atol=0), "shard sum-exp"
            # W against S (|W| / S is the mean |centred logit|, a few units)
            assert (np.abs(W[fin] - ref[fin, 2]) <= rtol * (np.abs(ref[fin, 2]) + ref[fin, 1])).all(), "shard W"
            lrec = vp.decode_partials(vp.vp_logprobs_partial(a[:, lo:hi], t, lo))
            tt = t.cpu().numpy()
            has = (tt >= lo) & (tt < hi)
            lfl = lrec["flags"].cpu().numpy()
            assert (((lfl & vp.PART_HAS_TARGET) != 0) == has).all()
            assert (((lfl & vp.PART_IGNORED) != 0) == (tt < 0)).all()
            zt = lrec["z_t"].double().cpu().numpy()
            rows = np.nonzero(has)[0]
            assert (zt[rows] == a64[rows, tt[rows]]).all(), "target logit"
            for d in (vp.KL_REVERSE, vp.KL_FORWARD):
                krec = vp.decode_partials(vp.vp_kl_partial(a[:, lo:hi], b[:, lo:hi], d))
                kref = oracle.shard_kl_stats(a64, b64, lo, hi, d)
                kfl = krec["flags"].cpu().numpy()
                assert (((kfl & vp.PART_MISMATCH) != 0) == (kref[:, 6] != 0)).all(), "mismatch flag"
                bad = ((kfl & (vp.PART_NANINF | vp.PART_NANINF_B)) != 0)
                assert (bad == (kref[:, 5] != 0)).all(), "NaN flags"
                ok = ~bad & (kref[:, 6] == 0) & np.isfinite(kref[:, 0]) & np.isfinite(kref[:, 2])
                assert (krec["m"].double().cpu().numpy()[ok] == kref[ok, 0]).all()
                assert (krec["m_b"].double().cpu().numpy()[ok] == kref[ok, 2]).all()
                assert np.allclose(krec["S"].cpu().numpy()[ok], kref[ok, 1], rtol=rtol, atol=0)
                assert np.allclose(krec["S_b"].cpu().numpy()[ok], kref[ok, 3], rtol=rtol, atol=0)
                Wk = krec["W"].cpu().numpy()[ok]
                assert (np.abs(Wk - kref[ok, 4]) <= rtol * (np.abs(kref[ok, 4]) + 10 * kref[ok, 1])).all()


def test_merge_is_batch_invariant():
    N, V, cuts = 64, 20011, (0, 9000, 20011)
    a, b, t, g = _inputs(N, V, torch.bfloat16, seed=9, cuts=cuts)
    a, b = a.to(DEV), b.to(DEV)
    parts = torch.stack([vp.vp_kl_partial(a[:, lo:hi], b[:, lo:hi]) for lo, hi in zip(cuts[:-1], cuts[1:])])
    kl, sa, sb = vp.vp_kl_merge(parts)
    sub = parts[:, 17:40].contiguous()
    kl2, sa2, sb2 = vp.vp_kl_merge(sub)
    torch.cuda.synchronize()
    assert torch.equal(kl[17:40].view(torch.int32), kl2.view(torch.int32))
    assert torch.equal(sa[17:40].view(torch.int32), sa2.view(torch.int32))
    parts = torch.stack([vp.vp_entropy_partial(a[:, lo:hi]) for lo, hi in zip(cuts[:-1], cuts[1:])])
    H, _ = vp.vp_entropy_merge(parts)
    H2, _ = vp.vp_entropy_merge(parts[:, 3:4].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(H[3:4].view(torch.int32), H2.view(torch.int32))


def test_merge_argument_errors():
    parts = vp.partials(4, DEV, K=2)
    with pytest.raises(vp.VPError):
        vp.vp_entropy_merge(parts[:, :, :4].contiguous())
    with pytest.raises(vp.VPError):
        vp.vp_kl_merge(parts, direction=7)
    H, st = vp.vp_entropy_merge(vp.partials(0, DEV, K=3))
    assert H.numel() == 0
