"""The no-allocation linear-logp entry point, called through the C ABI.

vp_linear_logp_fwd_noalloc keeps its scratch in a fixed array inside the
library, for callers that cannot allocate device memory themselves (a plugin
whose host framework owns every device allocation, a service that fixes its
memory footprint at start-up). It runs the same kernels as vp_linear_logp_fwd,
which takes a caller workspace, so its results must equal that entry point's
bit for bit, on consecutive calls (the array keeps the previous call's
contents), and match the fp64 oracle. This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import vocab_wide_logprobs_gb300 as vp
from vocab_wide_logprobs_gb300 import _lib, workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"
VP_ERR_SCRATCH = 9
SCRATCH_BYTES = 24 << 20


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(h, W, t, vocab_start=0):
    N, D = h.shape
    V = W.shape[0]
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    stats = vp.rowstats(N, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    status = _lib.lib().vp_linear_logp_fwd_noalloc(_p(h), _p(W), N, V, D, vocab_start, _p(t), _p(logp), _p(stats),
                                                   _p(err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return status, logp, stats, err


def _case(N, V, D, seed):
    w = workloads.linear(seed=seed, N=N, V=V, D=D)
    w["weight"] = (w["weight"].float() * 25).to(torch.bfloat16)   # logits with a spread of several units
    return w


def _bits(x):
    return x.view(torch.int32)


def _same_as_workspace_entry_point(w, tag, oracle_rows):
    h, W, t = w["hidden"].to(DEV), w["weight"].to(DEV), w["targets"].to(DEV)
    t[1] = -1                                         # an ignored target
    status, logp, stats, err = _noalloc(h, W, t)
    assert status == 0, _lib.status_string(status)
    err_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref_logp, ref_stats = vp.vp_linear_logp_fwd(h, W, t, err_word=err_ref)
    torch.cuda.synchronize()
    assert torch.equal(_bits(logp), _bits(ref_logp)), f"{tag}: logp differs from the workspace entry point"
    assert torch.equal(_bits(stats), _bits(ref_stats)), f"{tag}: records differ from the workspace entry point"
    assert int(err.item()) == int(err_ref.item()) == 0
    rows = np.asarray(oracle_rows)
    tt = t.cpu().numpy()[rows]
    o_lp, o_m, o_ls, o_err = oracle.linear_logp_fwd(parity.to64(w["hidden"][rows]), parity.to64(w["weight"]), tt)
    idx = torch.as_tensor(rows, device=DEV)
    parity.check_out(logp[idx], o_lp, f"{tag} logp vs oracle")
    parity.check_out(vp.decode_rowstats(stats[idx])["logS"], o_ls, f"{tag} logS vs oracle")
    assert o_err == 0


@pytest.mark.parametrize("shape", [(384, 3000, 256), (200, 777, 128)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(shape):
    N, V, D = shape
    for call, seed in enumerate((21, 22)):           # two calls in a row, different inputs
        _same_as_workspace_entry_point(_case(N, V, D, seed + N), f"call {call}", np.arange(N))


def _largest_rows(V, D):
    """The most rows whose scratch fits the fixed array (the workspace entry point's size rule)."""
    lo, hi = 1, 1 << 20
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if vp.vp_linear_logp_workspace_size(mid, V, D) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_noalloc_at_the_scratch_limit():
    V, D = 75968, 64
    N = _largest_rows(V, D)
    assert vp.vp_linear_logp_workspace_size(N + 1, V, D) > SCRATCH_BYTES
    # the last rows' target logits sit at the end of the array
    _same_as_workspace_entry_point(_case(N, V, D, 5), f"{N} rows (limit)", [0, 1, N // 2, N - 2, N - 1])
    w = _case(N + 1, V, D, 6)
    status, logp, _, _ = _noalloc(w["hidden"].to(DEV), w["weight"].to(DEV), w["targets"].to(DEV))
    torch.cuda.synchronize()
    assert status == VP_ERR_SCRATCH
    assert torch.isnan(logp).all()                    # refused before any work was queued


def test_noalloc_rejects_problems_beyond_its_scratch():
    h = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(256, 64, dtype=torch.bfloat16, device=DEV)
    t = torch.zeros(128, dtype=torch.int64, device=DEV)
    out = torch.zeros(128, dtype=torch.float32, device=DEV)
    stats = vp.rowstats(128, DEV)
    # 2^20 rows x 297 vocabulary tiles needs ~2.4 GB of scratch: refused before any work is queued
    status = _lib.lib().vp_linear_logp_fwd_noalloc(_p(h), _p(W), 1 << 20, 75968, 64, 0, _p(t), _p(out), _p(stats),
                                                   None, None)
    assert status == VP_ERR_SCRATCH
    assert "scratch" in _lib.status_string(status)
