"""The binding refuses tensors that do not fit the pointer they would be passed as.

The C ABI takes plain pointers and trusts the caller for their sizes; the Python
binding checks every caller-provided tensor against the N, V (and K, D) it
derives from the logits before anything reaches the library: element count,
dtype, device and contiguity. Every case here is refused on the host, before
the library is called, so these tests run anywhere (CPU tensors suffice).
"""
import pytest
import torch

import vocab_wide_logprobs_gb300 as vp

N, V = 6, 40


def _x(dtype=torch.bfloat16):
    return torch.zeros(N, V, dtype=dtype)


def _status(fn):
    with pytest.raises(vp.VPError) as e:
        fn()
    return e.value.status


def test_gradient_outputs_are_checked():
    x, t, g, st = _x(), torch.zeros(N, dtype=torch.int64), torch.zeros(N), vp.rowstats(N, "cpu")
    assert _status(lambda: vp.vp_logprobs_bwd(x, t, st, g, dx=torch.empty(N - 1, V, dtype=x.dtype))) == 2
    assert _status(lambda: vp.vp_logprobs_bwd(x, t, st, g, dx=torch.empty(N, V, dtype=torch.float32))) == 3
    assert _status(lambda: vp.vp_entropy_bwd(x, st, g, dx=torch.empty(V, N, dtype=x.dtype).t())) == 4
    a, b = _x(), _x()
    assert _status(lambda: vp.vp_kl_bwd(a, b, vp.KL_REVERSE, st, st, g, db=torch.empty(N, V + 1, dtype=a.dtype))) == 2
    assert _status(lambda: vp.vp_jsd_bwd(a, b, 0.5, st, st, g, da=torch.empty(N * V, dtype=torch.float32))) == 3


def test_per_row_arguments_are_checked():
    x, st = _x(), vp.rowstats(N, "cpu")
    t32 = torch.zeros(N, dtype=torch.int32)
    assert _status(lambda: vp.vp_logprobs_fwd(x, t32)) == 3                               # targets must be int64
    assert _status(lambda: vp.vp_logprobs_fwd(x, torch.zeros(N + 1, dtype=torch.int64))) == 2
    assert _status(lambda: vp.vp_entropy_fwd(x, stats=vp.rowstats(N - 1, "cpu"))) == 2
    assert _status(lambda: vp.vp_entropy_fwd(x, H=torch.empty(N, dtype=torch.float64))) == 3
    assert _status(lambda: vp.vp_entropy_bwd(x, st, torch.zeros(2 * N)[::2])) == 4        # a strided upstream gradient
    err64 = torch.zeros(1, dtype=torch.int64)
    assert _status(lambda: vp.vp_logprobs_fwd(x, torch.zeros(N, dtype=torch.int64), err_word=err64)) == 3


def test_topk_arguments_are_checked():
    x, K = _x(), 3
    ids = torch.zeros(N, K, dtype=torch.int64)
    st = vp.rowstats(N, "cpu")
    assert _status(lambda: vp.vp_logprobs_topk_fwd(x, ids, logp=torch.empty(N))) == 2
    assert _status(lambda: vp.vp_logprobs_topk_bwd(x, ids, st, torch.zeros(N))) == 2     # grad is [N, K]


def test_sharded_records_and_merges_are_checked():
    x = _x()
    assert _status(lambda: vp.vp_entropy_partial(x, parts=vp.partials(N + 1, "cpu"))) == 2
    assert _status(lambda: vp.vp_entropy_partial(x, parts=torch.empty(N, 5, dtype=torch.float32))) == 3
    parts = vp.partials(N, "cpu", K=2)
    assert _status(lambda: vp.vp_entropy_merge(parts, stats=vp.rowstats(2 * N, "cpu"))) == 2
    assert _status(lambda: vp.vp_kl_merge(parts, kl=torch.empty(N, dtype=torch.bfloat16))) == 3


def test_linear_arguments_are_checked():
    D, Vw = 64, 32
    h, W = torch.zeros(N, D, dtype=torch.bfloat16), torch.zeros(Vw, D, dtype=torch.bfloat16)
    t, g, st = torch.zeros(N, dtype=torch.int64), torch.zeros(N), vp.rowstats(N, "cpu")
    assert _status(lambda: vp.vp_linear_logp_bwd(h, W, t, st, g, dW=torch.empty(Vw, D + 1, dtype=torch.bfloat16))) == 2
    assert _status(lambda: vp.vp_linear_logp_bwd(h, W.float(), t, st, g)) == 3
    assert _status(lambda: vp.vp_linear_entropy_bwd(h, W, st, g, dhidden=torch.empty(N, D))) == 3
    outs = [torch.empty(N, D, dtype=torch.bfloat16), torch.empty(Vw, D, dtype=torch.bfloat16), None,
            torch.empty(Vw, 2 * D, dtype=torch.bfloat16)]
    assert _status(lambda: vp.vp_linear_kl_bwd(h, W, h, W, vp.KL_REVERSE, st, st, g, outs=outs)) == 2
    assert _status(lambda: vp.vp_linear_jsd_bwd(h, W, h, W, 0.5, st, st, g, outs=outs[:3])) == 7
    assert _status(lambda: vp.vp_linear_logp_fwd_noalloc(h, W, t, logp=torch.empty(N + 2))) == 2
