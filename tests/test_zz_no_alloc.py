"""The no-allocation linear-logp entry point, called through the C ABI.

vp_linear_logp_fwd_noalloc keeps its scratch in a fixed array inside the
library, for callers that cannot allocate device memory themselves (a plugin
whose host framework owns every device allocation, a service that fixes its
memory footprint at start-up). Its results must equal those of
vp_linear_logp_fwd, which takes a caller workspace, on consecutive calls (the
array keeps the previous call's contents). This file is collected last so that
a run stopping at the first failure has already run every other test; it also
passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import vocab_wide_logprobs_gb300 as vp
from vocab_wide_logprobs_gb300 import _lib, workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"
VP_ERR_SCRATCH = 9


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


@pytest.mark.parametrize("shape", [(384, 3000, 256), (200, 777, 128)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(shape):
    N, V, D = shape
    for call, seed in enumerate((21, 22)):           # two calls in a row, different inputs
        w = workloads.linear(seed=seed + N, N=N, V=V, D=D)
        w["weight"] = (w["weight"].float() * 25).to(torch.bfloat16)
        h, W, t = w["hidden"].to(DEV), w["weight"].to(DEV), w["targets"].to(DEV)
        t[1] = -1                                     # an ignored target
        status, logp, stats, err = _noalloc(h, W, t)
        assert status == 0, _lib.status_string(status)
        err_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
        ref_logp, ref_stats = vp.vp_linear_logp_fwd(h, W, t, err_word=err_ref)
        torch.cuda.synchronize()
        parity.check_out(logp, parity.to64(ref_logp), f"call {call} logp")
        parity.check_out(vp.decode_rowstats(stats)["logS"], parity.to64(vp.decode_rowstats(ref_stats)["logS"]),
                         f"call {call} logS")
        assert int(err.item()) == int(err_ref.item()) == 0


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
