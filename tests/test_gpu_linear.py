"""GPU parity of the fused linear logp (tcgen05 path) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import vocab_wide_logprobs_gb300 as vp
from vocab_wide_logprobs_gb300 import workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_fwd(w, rows=None, vocab_start=0, tag=""):
    h, W, t = w["hidden"].to(DEV), w["weight"].to(DEV), (w["targets"] + vocab_start).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp, st = vp.vp_linear_logp_fwd(h, W, t, vocab_start, err_word=err)
    torch.cuda.synchronize()
    sel = np.arange(h.shape[0]) if rows is None else np.asarray(rows)
    ref_lp, ref_m, ref_ls, ref_err = oracle.linear_logp_fwd(parity.to64(w["hidden"][sel]), parity.to64(w["weight"]),
                                                            (w["targets"] + vocab_start)[sel].numpy(), vocab_start)
    idx = torch.as_tensor(sel, device=DEV)
    parity.check_out(lp[idx], ref_lp, f"{tag}logp")
    d = vp.decode_rowstats(st[idx])
    parity.check_out(d["m"], ref_m, f"{tag}max logit")        # fp32 accumulations vs fp64 logits
    parity.check_out(d["logS"], ref_ls, f"{tag}logS")
    assert int(err.item()) == ref_err
    return lp


@pytest.mark.parametrize("N,V,D", [(256, 1024, 256), (200, 777, 128), (130, 300, 64), (64, 4096, 1024)])
def test_linear_logp_fwd_small(N, V, D):
    w = workloads.linear(seed=N + V + D, N=N, V=V, D=D)
    w["weight"] = (w["weight"].float() * 25).to(torch.bfloat16)   # logits with a spread of several units
    _check_fwd(w, tag=f"{N}x{V}x{D} ")


def test_linear_logp_targets_and_vocab_start():
    w = workloads.linear(seed=5, N=160, V=600, D=128)
    w["targets"][3] = -1          # ignored
    w["targets"][4] = 600         # past the shard
    _check_fwd(w, vocab_start=1000, tag="vocab_start ")


def test_linear_logp_batch_invariance():
    w = workloads.linear(seed=6, N=384, V=2000, D=256)
    h, W, t = w["hidden"].to(DEV), w["weight"].to(DEV), w["targets"].to(DEV)
    full, _ = vp.vp_linear_logp_fwd(h, W, t)
    part, _ = vp.vp_linear_logp_fwd(h[128:256].contiguous(), W, t[128:256].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(full[128:256].view(torch.int32), part.view(torch.int32))


@pytest.mark.slow
def test_linear_logp_full_size_sampled():
    w = workloads.linear()
    rows = [0, 1, 127, 128, 4095, 8191]
    lp = _check_fwd(w, rows=rows, tag="config 5 ")
    assert torch.isfinite(lp).all() and (lp <= 0).all()


# ---------------------------------------------------------------------------
# Backward: dhidden and dW, held to the GEMM-gradient bound of parity.check_gemm_grad.
# ---------------------------------------------------------------------------
_check_gemm_grad = parity.check_gemm_grad


def _bwd_case(N, V, D, seed, vocab_start=0, scale=25.0):
    w = workloads.linear(seed=seed, N=N, V=V, D=D)
    w["weight"] = (w["weight"].float() * scale).to(torch.bfloat16)
    w["targets"] = w["targets"] + vocab_start
    return w


def _run_bwd(w, vocab_start=0, **kw):
    h, W, t, g = (w[k].to(DEV) for k in ("hidden", "weight", "targets", "grad"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp, st = vp.vp_linear_logp_fwd(h, W, t, vocab_start, err_word=err)
    dh, dW = vp.vp_linear_logp_bwd(h, W, t, st, g, vocab_start, err_word=err, **kw)
    torch.cuda.synchronize()
    return dh, dW, int(err.item())


@pytest.mark.parametrize("N,V,D", [(256, 1024, 256), (200, 777, 128), (130, 300, 64), (64, 9000, 128),
                                   (72, 70000, 64)])   # the last: three vocabulary chunks, a ragged last one
def test_linear_logp_bwd_small(N, V, D):
    w = _bwd_case(N, V, D, seed=N + 7 * V + D)
    dh, dW, _ = _run_bwd(w)
    h64, W64 = parity.to64(w["hidden"]), parity.to64(w["weight"])
    t, g = w["targets"].numpy(), w["grad"].double().numpy()
    ref_dh, ref_dW = oracle.linear_logp_bwd(h64, W64, t, g)
    dz = np.abs(oracle.logprobs_bwd(oracle.linear_logits(h64, W64), t, g))
    _check_gemm_grad(dh, ref_dh, parity.gemm_norms(dz, W64), f"{N}x{V}x{D} dhidden")
    _check_gemm_grad(dW, ref_dW, parity.gemm_norms(dz.T, h64), f"{N}x{V}x{D} dW")


def test_linear_logp_bwd_single_outputs_and_special_targets():
    w = _bwd_case(136, 1500, 128, seed=3, vocab_start=500)
    w["targets"][5] = -1            # ignored: contributes nothing
    full_dh, full_dW, _ = _run_bwd(w, vocab_start=500)
    dh_only, none_w, _ = _run_bwd(w, vocab_start=500, want_dW=False)
    none_h, dW_only, _ = _run_bwd(w, vocab_start=500, want_dhidden=False)
    assert none_w is None and none_h is None
    assert torch.equal(dh_only, full_dh) and torch.equal(dW_only, full_dW)
    assert (full_dh[5] == 0).all()
    w["targets"][7] = 500 + 1500    # past the shard: NaN row of dhidden, NaN dW, error bit
    dh, dW, err = _run_bwd(w, vocab_start=500)
    assert err == 1 and torch.isnan(dh[7]).all() and torch.isfinite(dh[8]).all() and torch.isnan(dW).all()


@pytest.mark.slow
def test_linear_logp_bwd_full_size_sampled():
    w = workloads.linear()
    h, W, t, g = (w[k].to(DEV) for k in ("hidden", "weight", "targets", "grad"))
    lp, st = vp.vp_linear_logp_fwd(h, W, t)
    dh, dW = vp.vp_linear_logp_bwd(h, W, t, st, g)
    torch.cuda.synchronize()
    rows = [0, 777, 8191]
    h64, W64 = parity.to64(w["hidden"][rows]), parity.to64(w["weight"])
    tt, gg = w["targets"][rows].numpy(), w["grad"][rows].double().numpy()
    ref_dh, _ = oracle.linear_logp_bwd(h64, W64, tt, gg, want_dW=False)
    dz = np.abs(oracle.logprobs_bwd(oracle.linear_logits(h64, W64), tt, gg))
    _check_gemm_grad(dh[rows], ref_dh, parity.gemm_norms(dz, W64), "config 5 dhidden")
    # dW on every row: each column of dW sums to 0 over the vocabulary (every dz row sums to 0)
    col = dW.double().sum(0).abs()
    scale = dW.double().abs().sum(0)
    assert torch.isfinite(dW).all() and (col <= 2.0 ** -7 * scale + 1e-6).all()


@pytest.mark.slow
def test_linear_logp_bwd_full_size_dW_rows():
    """Whole rows of dW (all D columns) at the full linear workload: dW_j = sum_n dz[n, j] h_n needs
    every row's normaliser, which the oracle takes block by block in fp64 (linear_row_stats)."""
    w = workloads.linear()
    h, W, t, g = (w[k].to(DEV) for k in ("hidden", "weight", "targets", "grad"))
    lp, st = vp.vp_linear_logp_fwd(h, W, t)
    dh, dW = vp.vp_linear_logp_bwd(h, W, t, st, g)
    torch.cuda.synchronize()
    h64, W64 = parity.to64(w["hidden"]), parity.to64(w["weight"])
    tt, gg = w["targets"].numpy(), w["grad"].double().numpy()
    V = W64.shape[0]
    # chunk edges (32768 columns) and the targets of a few rows
    ids = np.unique(np.concatenate([[0, 1, 32767, 32768, 65535, 65536, V - 1], tt[[0, 5, 4096]]]))
    ref, dz = oracle.linear_logp_dW_rows(h64, W64, tt, gg, ids)
    _check_gemm_grad(dW[torch.as_tensor(ids, device=DEV)], ref, parity.gemm_norms(dz.T, h64), "config 5 dW rows")


@pytest.mark.parametrize("N", [9000, 17000])   # vocabulary chunks of 16384 and 8192 columns
def test_linear_logp_bwd_many_rows_sampled(N):
    V, D = 20011, 128
    w = _bwd_case(N, V, D, seed=N)
    dh, dW, err = _run_bwd(w)
    assert err == 0
    rows = [0, 1, 4095, 8191, N // 2, N - 1]
    h64, W64 = parity.to64(w["hidden"][rows]), parity.to64(w["weight"])
    t, g = w["targets"][rows].numpy(), w["grad"][rows].double().numpy()
    ref_dh, _ = oracle.linear_logp_bwd(h64, W64, t, g, want_dW=False)
    dz = np.abs(oracle.logprobs_bwd(oracle.linear_logits(h64, W64), t, g))
    _check_gemm_grad(dh[rows], ref_dh, parity.gemm_norms(dz, W64), f"{N} rows dhidden")
    # every dz row sums to 0, so each column of dW sums to 0 over the vocabulary
    col = dW.double().sum(0).abs()
    scale = dW.double().abs().sum(0)
    assert torch.isfinite(dW).all() and (col <= 2.0 ** -7 * scale + 1e-6).all()
