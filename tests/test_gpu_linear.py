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
