"""ctypes binding of libvp: one Python function per C entry point, same names.

Argument marshalling only: a function turns torch CUDA tensors into device
pointers, sizes and the two row strides of ``include/vp.h``, allocates any
output the caller did not pass (torch owns device memory), calls the C
function on the current torch stream and raises ``VPError`` on a non-zero
status. Every step of the computation runs in libvp's CUDA kernels; there is
no CPU or PyTorch fallback, and a missing library or device raises.

Row layouts accepted for logits (last stride must be 1):
  * ``[N, V]``: any row stride (R = N, s_i = stride(0));
  * ``[B, T, V]``: any two outer strides, e.g. ``logits[:, :-1]`` of a
    contiguous ``[B, T + 1, V]`` tensor (N = B T, R = T, s_o = stride(0),
    s_i = stride(1)).
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

F32, BF16 = 0, 1
KL_REVERSE, KL_FORWARD = 0, 1
GRAD_EXACT, GRAD_FAST = 0, 1   # precision of the fused linear backwards (VP_GRAD_EXACT / VP_GRAD_FAST)
ERRBIT_TARGET = 1
ROW_NANINF, ROW_EMPTY, ROW_MISMATCH, ROW_SHARDED, ROW_BADTARGET = 1, 2, 4, 8, 16
ROWSTAT_FLOATS = 8  # sizeof(vp_rowstat) / 4
PART_NANINF, PART_NANINF_B, PART_MISMATCH, PART_HAS_TARGET, PART_IGNORED = 1, 2, 4, 8, 16
PARTIAL_DOUBLES = 5  # sizeof(vp_partial) / 8


def rowstats(N: int, device) -> torch.Tensor:
    """Storage for N vp_rowstat records: a float32 [N, 8] tensor (32 bytes per row)."""
    return torch.empty((N, ROWSTAT_FLOATS), dtype=torch.float32, device=device)


def decode_rowstats(stats: torch.Tensor) -> dict:
    """Fields of vp_rowstat records as tensors: m, logS (hi + lo in fp64), c (hi + lo in fp64), flags."""
    s = stats.detach()
    return {"m": s[:, 0], "logS": s[:, 1].double() + s[:, 2].double(), "c": s[:, 3].double() + s[:, 4].double(),
            "flags": s[:, 5].view(torch.int32)}


class VPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.status_string(status)} (status {status})")


def partials(N: int, device, K: int = None) -> torch.Tensor:
    """Storage for vp_partial records: float64 [N, 5] (40 bytes per row), or [K, N, 5] for K shards."""
    shape = (N, PARTIAL_DOUBLES) if K is None else (K, N, PARTIAL_DOUBLES)
    return torch.empty(shape, dtype=torch.float64, device=device)


def decode_partials(parts: torch.Tensor) -> dict:
    """Fields of vp_partial records ([..., 5] float64) as tensors: m, m_b, S, S_b, W, z_t, flags."""
    p = parts.detach()
    f = p.view(torch.float32)
    return {"m": f[..., 0], "m_b": f[..., 1], "S": p[..., 1], "S_b": p[..., 2], "W": p[..., 3], "z_t": f[..., 8],
            "flags": p.view(torch.int32)[..., 9]}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise VPError(3, f"dtype {t.dtype}")


def rows_of(x: torch.Tensor):
    """(N, V, R, s_o, s_i) of a [N, V] or [B, T, V] logits view with unit last stride."""
    if x.dim() == 2:
        N, V = x.shape
        if V > 1 and x.stride(1) != 1:
            raise VPError(4, "logits need a unit stride along V")
        return N, V, max(N, 1), 0, x.stride(0)
    if x.dim() == 3:
        B, T, V = x.shape
        if V > 1 and x.stride(2) != 1:
            raise VPError(4, "logits need a unit stride along V")
        return B * T, V, max(T, 1), x.stride(0), x.stride(1)
    raise VPError(2, f"logits must be 2-D or 3-D, got {x.dim()}-D")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _precision(p):
    return GRAD_EXACT if p is None else int(p)


def _check(status: int, where: str):
    if status != 0:
        raise VPError(status, where)


def _f32(n, like):
    return torch.empty(n, dtype=torch.float32, device=like.device)


def _arg(t, n: int, dtype, like, what: str):
    """A caller's tensor behind one of the C ABI's pointers. The library reads or writes exactly n elements
    of dtype there, so another size, dtype or device, or a strided view, is refused here, before a kernel
    could run past its end. None passes (an output to allocate, or an optional pointer)."""
    if t is None:
        return None
    bad = (2 if t.numel() != n else 3 if t.dtype != dtype else 4 if (t.device != like.device or not t.is_contiguous())
           else 0)
    if bad:
        raise VPError(bad, f"{what}: needs {n} contiguous {dtype} elements on {like.device}, got "
                           f"{tuple(t.shape)} {t.dtype} on {t.device}{'' if t.is_contiguous() else ', strided'}")
    return t


def _row_args(like, N, targets=None, stats=(), grad=None, err_word=None, outs=(), K=1):
    """The per-row arguments of a logits call: targets int64 [N] ([N, K] for top-k), vp_rowstat records,
    the upstream gradient fp32 [N] ([N, K]), the error word int32 [1] and fp32 [N] ([N, K]) outputs."""
    _arg(targets, N * K, torch.int64, like, "targets")
    for i, st in enumerate(stats):
        _arg(st, N * ROWSTAT_FLOATS, torch.float32, like, f"stats{'' if len(stats) == 1 else ' ' + 'ab'[i]}")
    _arg(grad, N * K, torch.float32, like, "grad")
    _arg(err_word, 1, torch.int32, like, "err_word")
    for o in outs:
        _arg(o, N * K, torch.float32, like, "per-row output")


def _parts_arg(parts, n_records: int, like):
    _arg(parts, n_records * PARTIAL_DOUBLES, torch.float64, like, "parts")


def _same_layout(a: torch.Tensor, b: torch.Tensor):
    if a.shape != b.shape or a.stride() != b.stride() or a.dtype != b.dtype:
        raise VPError(4, "A and B must share shape, strides and dtype")


def vp_logprobs_fwd(x, targets, vocab_start: int = 0, err_word=None, logp=None, stats=None):
    """Returns (logp fp32 [N], stats vp_rowstat [N] as float32 [N, 8])."""
    N, V, R, s_o, s_i = rows_of(x)
    _row_args(x, N, targets=targets, stats=(stats,), err_word=err_word, outs=(logp,))
    logp = _f32(N, x) if logp is None else logp
    stats = rowstats(N, x.device) if stats is None else stats
    _check(_lib.lib().vp_logprobs_fwd(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, vocab_start, _ptr(targets),
                                      _ptr(logp), _ptr(stats), _ptr(err_word), _stream()), "vp_logprobs_fwd")
    return logp, stats


def vp_logprobs_bwd(x, targets, stats, grad, vocab_start: int = 0, err_word=None, dx=None):
    """Returns dx, contiguous [N, V] in the dtype of x."""
    N, V, R, s_o, s_i = rows_of(x)
    _row_args(x, N, targets=targets, stats=(stats,), grad=grad, err_word=err_word)
    _arg(dx, N * V, x.dtype, x, "dx")
    dx = torch.empty((N, V), dtype=x.dtype, device=x.device) if dx is None else dx
    _check(_lib.lib().vp_logprobs_bwd(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, vocab_start, _ptr(targets),
                                      _ptr(stats), _ptr(grad), _ptr(dx), _ptr(err_word), _stream()),
           "vp_logprobs_bwd")
    return dx


def _topk_ids(targets):
    if targets.dim() != 2 or targets.dtype != torch.int64 or not targets.is_contiguous():
        raise VPError(2, "top-k ids must be a contiguous int64 [N, K] tensor")
    return targets.shape[1]


def vp_logprobs_topk_fwd(x, targets, vocab_start: int = 0, err_word=None, logp=None, stats=None):
    """logp of K ids per row; targets int64 [N, K]. Returns (logp fp32 [N, K], stats)."""
    N, V, R, s_o, s_i = rows_of(x)
    K = _topk_ids(targets)
    _row_args(x, N, targets=targets, err_word=err_word, outs=(logp,), K=K)
    _row_args(x, N, stats=(stats,))
    logp = torch.empty((N, K), dtype=torch.float32, device=x.device) if logp is None else logp
    stats = rowstats(N, x.device) if stats is None else stats
    _check(_lib.lib().vp_logprobs_topk_fwd(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, vocab_start, _ptr(targets), K,
                                           _ptr(logp), _ptr(stats), _ptr(err_word), _stream()), "vp_logprobs_topk_fwd")
    return logp, stats


def vp_logprobs_topk_bwd(x, targets, stats, grad, vocab_start: int = 0, err_word=None, dx=None):
    """Gradient of sum_k grad[r, k] logp[r, k] (grad fp32 [N, K]); returns dx [N, V] in the dtype of x."""
    N, V, R, s_o, s_i = rows_of(x)
    K = _topk_ids(targets)
    _row_args(x, N, targets=targets, grad=grad, err_word=err_word, K=K)
    _row_args(x, N, stats=(stats,))
    _arg(dx, N * V, x.dtype, x, "dx")
    dx = torch.empty((N, V), dtype=x.dtype, device=x.device) if dx is None else dx
    _check(_lib.lib().vp_logprobs_topk_bwd(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, vocab_start, _ptr(targets), K,
                                           _ptr(stats), _ptr(grad), _ptr(dx), _ptr(err_word), _stream()),
           "vp_logprobs_topk_bwd")
    return dx


def vp_entropy_fwd(x, H=None, stats=None):
    """Returns (H fp32 [N], stats)."""
    N, V, R, s_o, s_i = rows_of(x)
    _row_args(x, N, stats=(stats,), outs=(H,))
    H = _f32(N, x) if H is None else H
    stats = rowstats(N, x.device) if stats is None else stats
    _check(_lib.lib().vp_entropy_fwd(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, _ptr(H), _ptr(stats), _stream()),
           "vp_entropy_fwd")
    return H, stats


def vp_entropy_bwd(x, stats, grad, dx=None):
    N, V, R, s_o, s_i = rows_of(x)
    _row_args(x, N, stats=(stats,), grad=grad)
    _arg(dx, N * V, x.dtype, x, "dx")
    dx = torch.empty((N, V), dtype=x.dtype, device=x.device) if dx is None else dx
    _check(_lib.lib().vp_entropy_bwd(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, _ptr(stats), _ptr(grad),
                                     _ptr(dx), _stream()), "vp_entropy_bwd")
    return dx


def vp_kl_fwd(a, b, direction: int = KL_REVERSE, kl=None, stats_a=None, stats_b=None):
    """Returns (kl, stats_a, stats_b); reverse = KL(A||B), forward = KL(B||A)."""
    _same_layout(a, b)
    N, V, R, s_o, s_i = rows_of(a)
    _row_args(a, N, stats=(stats_a, stats_b), outs=(kl,))
    kl = _f32(N, a) if kl is None else kl
    stats_a = rowstats(N, a.device) if stats_a is None else stats_a
    stats_b = rowstats(N, a.device) if stats_b is None else stats_b
    _check(_lib.lib().vp_kl_fwd(_ptr(a), _ptr(b), _dtype_code(a), N, V, R, s_o, s_i, int(direction), _ptr(kl),
                                _ptr(stats_a), _ptr(stats_b), _stream()), "vp_kl_fwd")
    return kl, stats_a, stats_b


def vp_kl_bwd(a, b, direction, stats_a, stats_b, grad, want_da=True, want_db=True, da=None, db=None):
    """Returns (da, db); an unwanted gradient is None and is not computed."""
    _same_layout(a, b)
    N, V, R, s_o, s_i = rows_of(a)
    _row_args(a, N, stats=(stats_a, stats_b), grad=grad)
    _arg(da if want_da else None, N * V, a.dtype, a, "da")
    _arg(db if want_db else None, N * V, a.dtype, a, "db")
    if want_da and da is None:
        da = torch.empty((N, V), dtype=a.dtype, device=a.device)
    if want_db and db is None:
        db = torch.empty((N, V), dtype=a.dtype, device=a.device)
    da = da if want_da else None
    db = db if want_db else None
    _check(_lib.lib().vp_kl_bwd(_ptr(a), _ptr(b), _dtype_code(a), N, V, R, s_o, s_i, int(direction),
                                _ptr(stats_a), _ptr(stats_b), _ptr(grad), _ptr(da), _ptr(db), _stream()),
           "vp_kl_bwd")
    return da, db


def vp_jsd_fwd(a, b, beta: float = 0.5, jsd=None, stats_a=None, stats_b=None):
    """Generalized JSD per row (a: student, b: teacher); beta = 0 / 1 are KL(b||a) / KL(a||b).

    Returns (jsd fp32 [N], stats of a, stats of b)."""
    _same_layout(a, b)
    N, V, R, s_o, s_i = rows_of(a)
    _row_args(a, N, stats=(stats_a, stats_b), outs=(jsd,))
    jsd = _f32(N, a) if jsd is None else jsd
    stats_a = rowstats(N, a.device) if stats_a is None else stats_a
    stats_b = rowstats(N, a.device) if stats_b is None else stats_b
    _check(_lib.lib().vp_jsd_fwd(_ptr(a), _ptr(b), _dtype_code(a), N, V, R, s_o, s_i, float(beta), _ptr(jsd),
                                 _ptr(stats_a), _ptr(stats_b), _stream()), "vp_jsd_fwd")
    return jsd, stats_a, stats_b


def vp_jsd_bwd(a, b, beta, stats_a, stats_b, grad, want_da=True, want_db=True, da=None, db=None):
    """Returns (da, db); an unwanted gradient (a frozen input) is None and is not computed."""
    _same_layout(a, b)
    N, V, R, s_o, s_i = rows_of(a)
    _row_args(a, N, stats=(stats_a, stats_b), grad=grad)
    _arg(da if want_da else None, N * V, a.dtype, a, "da")
    _arg(db if want_db else None, N * V, a.dtype, a, "db")
    if want_da and da is None:
        da = torch.empty((N, V), dtype=a.dtype, device=a.device)
    if want_db and db is None:
        db = torch.empty((N, V), dtype=a.dtype, device=a.device)
    da = da if want_da else None
    db = db if want_db else None
    _check(_lib.lib().vp_jsd_bwd(_ptr(a), _ptr(b), _dtype_code(a), N, V, R, s_o, s_i, float(beta), _ptr(stats_a),
                                 _ptr(stats_b), _ptr(grad), _ptr(da), _ptr(db), _stream()), "vp_jsd_bwd")
    return da, db


def vp_linear_logp_workspace_size(N: int, V: int, D: int) -> int:
    return int(_lib.lib().vp_linear_logp_workspace_size(N, V, D))


def vp_linear_logp_fwd(hidden, weight, targets, vocab_start: int = 0, err_word=None, logp=None, stats=None,
                       workspace=None):
    """logp of targets under softmax(hidden @ weight^T) without materialising the logits.

    hidden: bf16 [N, D], weight: bf16 [V, D] (contiguous). Returns (logp fp32 [N], stats)."""
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise VPError(3, "vp_linear_logp_fwd takes bf16 hidden and weight")
    if not (hidden.is_contiguous() and weight.is_contiguous()) or hidden.dim() != 2 or weight.dim() != 2:
        raise VPError(4, "hidden and weight must be contiguous 2-D tensors")
    N, D = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != D:
        raise VPError(2, "hidden and weight disagree on D")
    _row_args(hidden, N, targets=targets, stats=(stats,), err_word=err_word, outs=(logp,))
    logp = _f32(N, hidden) if logp is None else logp
    stats = rowstats(N, hidden.device) if stats is None else stats
    need = vp_linear_logp_workspace_size(N, V, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=hidden.device)
    _check(_lib.lib().vp_linear_logp_fwd(_ptr(hidden), _ptr(weight), N, V, D, vocab_start, _ptr(targets),
                                         _ptr(logp), _ptr(stats), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _ptr(err_word),
                                         _stream()), "vp_linear_logp_fwd")
    return logp, stats


def vp_linear_logp_bwd_workspace_size(N: int, V: int, D: int) -> int:
    return int(_lib.lib().vp_linear_logp_bwd_workspace_size(N, V, D))


def vp_linear_logp_bwd(hidden, weight, targets, stats, grad, vocab_start: int = 0, want_dhidden=True, want_dW=True,
                       err_word=None, dhidden=None, dW=None, workspace=None, precision: int = None):
    """Returns (dhidden bf16 [N, D] or None, dW bf16 [V, D] or None). precision: GRAD_EXACT (default:
    dz as a bf16 pair hi + lo in the gradient GEMMs) or GRAD_FAST (dz rounded to bf16)."""
    N, V, D = _linear_model(hidden, weight, "vp_linear_logp_bwd")
    _row_args(hidden, N, targets=targets, stats=(stats,), grad=grad, err_word=err_word)
    _arg(dhidden if want_dhidden else None, N * D, torch.bfloat16, hidden, "dhidden")
    _arg(dW if want_dW else None, V * D, torch.bfloat16, hidden, "dW")
    if want_dhidden and dhidden is None:
        dhidden = torch.empty((N, D), dtype=torch.bfloat16, device=hidden.device)
    if want_dW and dW is None:
        dW = torch.empty((V, D), dtype=torch.bfloat16, device=hidden.device)
    dhidden = dhidden if want_dhidden else None
    dW = dW if want_dW else None
    if workspace is None:
        need = vp_linear_logp_bwd_workspace_size(N, V, D)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=hidden.device)
    _check(_lib.lib().vp_linear_logp_bwd(_ptr(hidden), _ptr(weight), N, V, D, vocab_start, _ptr(targets),
                                         _ptr(stats), _ptr(grad), _ptr(dhidden), _ptr(dW), _precision(precision),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _ptr(err_word), _stream()),
           "vp_linear_logp_bwd")
    return dhidden, dW


def vp_linear_logp_fwd_noalloc(hidden, weight, targets, vocab_start: int = 0, err_word=None, logp=None,
                               stats=None):
    """vp_linear_logp_fwd with the library's fixed internal scratch instead of a workspace."""
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise VPError(3, "vp_linear_logp_fwd_noalloc takes bf16 hidden and weight")
    if not (hidden.is_contiguous() and weight.is_contiguous()) or hidden.dim() != 2 or weight.dim() != 2:
        raise VPError(4, "hidden and weight must be contiguous 2-D tensors")
    N, V, D = _linear_model(hidden, weight, "vp_linear_logp_fwd_noalloc")
    _row_args(hidden, N, targets=targets, stats=(stats,), err_word=err_word, outs=(logp,))
    logp = _f32(N, hidden) if logp is None else logp
    stats = rowstats(N, hidden.device) if stats is None else stats
    _check(_lib.lib().vp_linear_logp_fwd_noalloc(_ptr(hidden), _ptr(weight), N, V, D, vocab_start, _ptr(targets),
                                                 _ptr(logp), _ptr(stats), _ptr(err_word), _stream()),
           "vp_linear_logp_fwd_noalloc")
    return logp, stats


# ---------------------------------------------------------------------------
# Fused linear entropy and KL (logits never materialised)
# ---------------------------------------------------------------------------
def _linear_model(hidden, weight, what):
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise VPError(3, f"{what} takes bf16 hidden and weight")
    if not (hidden.is_contiguous() and weight.is_contiguous()) or hidden.dim() != 2 or weight.dim() != 2:
        raise VPError(4, "hidden and weight must be contiguous 2-D tensors")
    if weight.shape[1] != hidden.shape[1]:
        raise VPError(2, "hidden and weight disagree on D")
    return hidden.shape[0], weight.shape[0], hidden.shape[1]


def _workspace(nbytes, like):
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=like.device)


def vp_linear_entropy_workspace_size(N: int, V: int, D: int) -> int:
    return int(_lib.lib().vp_linear_entropy_workspace_size(N, V, D))


def vp_linear_entropy_bwd_workspace_size(N: int, V: int, D: int) -> int:
    return int(_lib.lib().vp_linear_entropy_bwd_workspace_size(N, V, D))


def vp_linear_kl_workspace_size(N: int, V: int) -> int:
    return int(_lib.lib().vp_linear_kl_workspace_size(N, V))


def vp_linear_kl_bwd_workspace_size(N: int, V: int, Da: int, Db: int) -> int:
    return int(_lib.lib().vp_linear_kl_bwd_workspace_size(N, V, Da, Db))


def vp_linear_jsd_workspace_size(N: int, V: int) -> int:
    return int(_lib.lib().vp_linear_jsd_workspace_size(N, V))


def vp_linear_jsd_bwd_workspace_size(N: int, V: int, Da: int, Db: int) -> int:
    return int(_lib.lib().vp_linear_jsd_bwd_workspace_size(N, V, Da, Db))


def _same_bytes(dst, src):
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise VPError(4, "host-buffer transfers take contiguous tensors")
    n = dst.numel() * dst.element_size()
    if n != src.numel() * src.element_size():
        raise VPError(2, "source and destination sizes differ")
    return n


def vp_upload(dst, src):
    """Copy a (page-locked) host tensor into a device tensor of the same size, on the current stream."""
    _check(_lib.lib().vp_upload(_ptr(dst), _ptr(src), _same_bytes(dst, src), _stream()), "vp_upload")
    return dst


def vp_download(dst, src):
    """Copy a device tensor into a (page-locked) host tensor of the same size, on the current stream."""
    _check(_lib.lib().vp_download(_ptr(dst), _ptr(src), _same_bytes(dst, src), _stream()), "vp_download")
    return dst


def vp_status_string(status: int) -> str:
    return _lib.status_string(status)


def vp_version() -> int:
    return int(_lib.lib().vp_version())


def vp_linear_entropy_fwd(hidden, weight, H=None, stats=None, workspace=None):
    """Entropy of softmax(hidden @ weight^T) per row; returns (H fp32 [N], stats)."""
    N, V, D = _linear_model(hidden, weight, "vp_linear_entropy_fwd")
    _row_args(hidden, N, stats=(stats,), outs=(H,))
    H = _f32(N, hidden) if H is None else H
    stats = rowstats(N, hidden.device) if stats is None else stats
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_entropy_workspace_size(N, V, D), hidden)
    _check(_lib.lib().vp_linear_entropy_fwd(_ptr(hidden), _ptr(weight), N, V, D, _ptr(H), _ptr(stats),
                                            _ptr(workspace), workspace.numel(), _stream()), "vp_linear_entropy_fwd")
    return H, stats


def vp_linear_entropy_bwd(hidden, weight, stats, grad, want_dhidden=True, want_dW=True, dhidden=None, dW=None,
                          workspace=None, precision: int = None):
    """Gradients of sum_r grad[r] H[r]: (dhidden bf16 [N, D] or None, dW bf16 [V, D] or None)."""
    N, V, D = _linear_model(hidden, weight, "vp_linear_entropy_bwd")
    _row_args(hidden, N, stats=(stats,), grad=grad)
    _arg(dhidden if want_dhidden else None, N * D, torch.bfloat16, hidden, "dhidden")
    _arg(dW if want_dW else None, V * D, torch.bfloat16, hidden, "dW")
    dhidden = (torch.empty((N, D), dtype=torch.bfloat16, device=hidden.device) if dhidden is None else dhidden) \
        if want_dhidden else None
    dW = (torch.empty((V, D), dtype=torch.bfloat16, device=hidden.device) if dW is None else dW) if want_dW else None
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_entropy_bwd_workspace_size(N, V, D), hidden)
    _check(_lib.lib().vp_linear_entropy_bwd(_ptr(hidden), _ptr(weight), N, V, D, _ptr(stats), _ptr(grad),
                                            _ptr(dhidden), _ptr(dW), _precision(precision), _ptr(workspace),
                                            workspace.numel(), _stream()),
           "vp_linear_entropy_bwd")
    return dhidden, dW


def _two_models(ha, wa, hb, wb, what):
    N, V, Da = _linear_model(ha, wa, what)
    Nb, Vb, Db = _linear_model(hb, wb, what)
    if (Nb, Vb) != (N, V):
        raise VPError(2, "the two models disagree on N or V")
    return N, V, Da, Db


def vp_linear_kl_fwd(ha, wa, hb, wb, direction: int = KL_REVERSE, kl=None, stats_a=None, stats_b=None,
                     workspace=None):
    """KL between softmax(ha @ wa^T) and softmax(hb @ wb^T); reverse = KL(A||B).
    Returns (kl fp32 [N], stats_a, stats_b)."""
    N, V, Da, Db = _two_models(ha, wa, hb, wb, "vp_linear_kl_fwd")
    _row_args(ha, N, stats=(stats_a, stats_b), outs=(kl,))
    kl = _f32(N, ha) if kl is None else kl
    stats_a = rowstats(N, ha.device) if stats_a is None else stats_a
    stats_b = rowstats(N, ha.device) if stats_b is None else stats_b
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_kl_workspace_size(N, V), ha)
    _check(_lib.lib().vp_linear_kl_fwd(_ptr(ha), _ptr(wa), _ptr(hb), _ptr(wb), N, V, Da, Db, int(direction), _ptr(kl),
                                       _ptr(stats_a), _ptr(stats_b), _ptr(workspace), workspace.numel(), _stream()),
           "vp_linear_kl_fwd")
    return kl, stats_a, stats_b


def vp_linear_kl_bwd(ha, wa, hb, wb, direction, stats_a, stats_b, grad, want=(True, True, True, True), outs=None,
                     workspace=None, precision: int = None):
    """Gradients of sum_r grad[r] KL[r]: (dha, dwa, dhb, dwb), bf16, None where not wanted."""
    N, V, Da, Db = _two_models(ha, wa, hb, wb, "vp_linear_kl_bwd")
    shapes = ((N, Da), (V, Da), (N, Db), (V, Db))
    _row_args(ha, N, stats=(stats_a, stats_b), grad=grad)
    if outs is not None:
        if len(outs) != 4:
            raise VPError(7, "outs: four gradients (dha, dwa, dhb, dwb), None where not wanted")
        for o, sh, w, nm in zip(outs, shapes, want, ("dha", "dwa", "dhb", "dwb")):
            _arg(o if w else None, sh[0] * sh[1], torch.bfloat16, ha, nm)
        outs = [o if w else None for o, w in zip(outs, want)]
    if outs is None:
        outs = [torch.empty(s, dtype=torch.bfloat16, device=ha.device) if w else None for s, w in zip(shapes, want)]
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_kl_bwd_workspace_size(N, V, Da, Db), ha)
    _check(_lib.lib().vp_linear_kl_bwd(_ptr(ha), _ptr(wa), _ptr(hb), _ptr(wb), N, V, Da, Db, int(direction),
                                       _ptr(stats_a), _ptr(stats_b), _ptr(grad), *[_ptr(o) for o in outs],
                                       _precision(precision), _ptr(workspace), workspace.numel(), _stream()),
           "vp_linear_kl_bwd")
    return tuple(outs)


def vp_linear_jsd_fwd(ha, wa, hb, wb, beta: float = 0.5, jsd=None, stats_a=None, stats_b=None, workspace=None):
    """Generalized JSD of softmax(ha @ wa^T) (student) and softmax(hb @ wb^T) (teacher).
    Returns (jsd fp32 [N], stats_a, stats_b)."""
    N, V, Da, Db = _two_models(ha, wa, hb, wb, "vp_linear_jsd_fwd")
    _row_args(ha, N, stats=(stats_a, stats_b), outs=(jsd,))
    jsd = _f32(N, ha) if jsd is None else jsd
    stats_a = rowstats(N, ha.device) if stats_a is None else stats_a
    stats_b = rowstats(N, ha.device) if stats_b is None else stats_b
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_jsd_workspace_size(N, V), ha)
    _check(_lib.lib().vp_linear_jsd_fwd(_ptr(ha), _ptr(wa), _ptr(hb), _ptr(wb), N, V, Da, Db, float(beta),
                                        _ptr(jsd), _ptr(stats_a), _ptr(stats_b), _ptr(workspace), workspace.numel(),
                                        _stream()), "vp_linear_jsd_fwd")
    return jsd, stats_a, stats_b


def vp_linear_jsd_bwd(ha, wa, hb, wb, beta, stats_a, stats_b, grad, want=(True, True, True, True), outs=None,
                      workspace=None, precision: int = None):
    """Gradients of sum_r grad[r] JSD[r]: (dha, dwa, dhb, dwb), bf16, None where not wanted."""
    N, V, Da, Db = _two_models(ha, wa, hb, wb, "vp_linear_jsd_bwd")
    shapes = ((N, Da), (V, Da), (N, Db), (V, Db))
    _row_args(ha, N, stats=(stats_a, stats_b), grad=grad)
    if outs is not None:
        if len(outs) != 4:
            raise VPError(7, "outs: four gradients (dha, dwa, dhb, dwb), None where not wanted")
        for o, sh, w, nm in zip(outs, shapes, want, ("dha", "dwa", "dhb", "dwb")):
            _arg(o if w else None, sh[0] * sh[1], torch.bfloat16, ha, nm)
        outs = [o if w else None for o, w in zip(outs, want)]
    if outs is None:
        outs = [torch.empty(s, dtype=torch.bfloat16, device=ha.device) if w else None for s, w in zip(shapes, want)]
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_jsd_bwd_workspace_size(N, V, Da, Db), ha)
    _check(_lib.lib().vp_linear_jsd_bwd(_ptr(ha), _ptr(wa), _ptr(hb), _ptr(wb), N, V, Da, Db, float(beta),
                                        _ptr(stats_a), _ptr(stats_b), _ptr(grad), *[_ptr(o) for o in outs],
                                        _precision(precision), _ptr(workspace), workspace.numel(), _stream()),
           "vp_linear_jsd_bwd")
    return tuple(outs)


# ---------------------------------------------------------------------------
# Vocabulary-sharded forms: per-shard records, gathered by the caller, merged
# ---------------------------------------------------------------------------
def vp_logprobs_partial(x, targets, vocab_start: int = 0, parts=None):
    """Per-row records of logprobs over the shard x (columns vocab_start .. vocab_start + V)."""
    N, V, R, s_o, s_i = rows_of(x)
    _row_args(x, N, targets=targets)
    _parts_arg(parts, N, x)
    parts = partials(N, x.device) if parts is None else parts
    _check(_lib.lib().vp_logprobs_partial(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, vocab_start, _ptr(targets),
                                          _ptr(parts), _stream()), "vp_logprobs_partial")
    return parts


def vp_entropy_partial(x, parts=None):
    """Per-row records of entropy over the shard x."""
    N, V, R, s_o, s_i = rows_of(x)
    _parts_arg(parts, N, x)
    parts = partials(N, x.device) if parts is None else parts
    _check(_lib.lib().vp_entropy_partial(_ptr(x), _dtype_code(x), N, V, R, s_o, s_i, _ptr(parts), _stream()),
           "vp_entropy_partial")
    return parts


def vp_kl_partial(a, b, direction: int = KL_REVERSE, parts=None):
    """Per-row records of KL over the shard held by a and b."""
    _same_layout(a, b)
    N, V, R, s_o, s_i = rows_of(a)
    _parts_arg(parts, N, a)
    parts = partials(N, a.device) if parts is None else parts
    _check(_lib.lib().vp_kl_partial(_ptr(a), _ptr(b), _dtype_code(a), N, V, R, s_o, s_i, int(direction),
                                    _ptr(parts), _stream()), "vp_kl_partial")
    return parts


def _gathered(parts):
    if parts.dim() != 3 or parts.shape[2] != PARTIAL_DOUBLES or parts.dtype != torch.float64 \
            or not parts.is_contiguous():
        raise VPError(2, "gathered records must be a contiguous float64 [K, N, 5] tensor")
    return parts.shape[0], parts.shape[1]


def vp_logprobs_merge(parts, err_word=None, logp=None, stats=None):
    """Merges [K, N] shard records (shard-major) into (logp fp32 [N], stats) for the whole rows."""
    K, N = _gathered(parts)
    _row_args(parts, N, stats=(stats,), err_word=err_word, outs=(logp,))
    logp = _f32(N, parts) if logp is None else logp
    stats = rowstats(N, parts.device) if stats is None else stats
    _check(_lib.lib().vp_logprobs_merge(_ptr(parts), K, N, _ptr(logp), _ptr(stats), _ptr(err_word), _stream()),
           "vp_logprobs_merge")
    return logp, stats


def vp_entropy_merge(parts, H=None, stats=None):
    """Merges [K, N] shard records into (H fp32 [N], stats)."""
    K, N = _gathered(parts)
    _row_args(parts, N, stats=(stats,), outs=(H,))
    H = _f32(N, parts) if H is None else H
    stats = rowstats(N, parts.device) if stats is None else stats
    _check(_lib.lib().vp_entropy_merge(_ptr(parts), K, N, _ptr(H), _ptr(stats), _stream()), "vp_entropy_merge")
    return H, stats


def vp_kl_merge(parts, direction: int = KL_REVERSE, kl=None, stats_a=None, stats_b=None):
    """Merges [K, N] shard records into (kl fp32 [N], stats of A, stats of B)."""
    K, N = _gathered(parts)
    _row_args(parts, N, stats=(stats_a, stats_b), outs=(kl,))
    kl = _f32(N, parts) if kl is None else kl
    stats_a = rowstats(N, parts.device) if stats_a is None else stats_a
    stats_b = rowstats(N, parts.device) if stats_b is None else stats_b
    _check(_lib.lib().vp_kl_merge(_ptr(parts), K, N, int(direction), _ptr(kl), _ptr(stats_a), _ptr(stats_b),
                                  _stream()), "vp_kl_merge")
    return kl, stats_a, stats_b


def vp_fault_status(clear: bool = False) -> int:
    """The device fault word (non-zero if a kernel's bounded wait gave up); synchronises."""
    v = ctypes.c_uint32(0)
    _check(_lib.lib().vp_fault_status(ctypes.byref(v), int(clear)), "vp_fault_status")
    return int(v.value)


def vp_set_row_split(ctas: int) -> None:
    """CTAs sharing one row's vocabulary in the forward scans (1, the default, or 2; process-wide)."""
    _check(_lib.lib().vp_set_row_split(int(ctas)), "vp_set_row_split")


def vp_get_row_split() -> int:
    return int(_lib.lib().vp_get_row_split())


def vp_linear_logp_partial(hidden, weight, targets, vocab_start: int = 0, parts=None, workspace=None):
    """Per-row logprobs records over the vocabulary shard held by weight (rows vocab_start .. + V of the head)."""
    N, V, D = _linear_model(hidden, weight, "vp_linear_logp_partial")
    _row_args(hidden, N, targets=targets)
    _parts_arg(parts, N, hidden)
    parts = partials(N, hidden.device) if parts is None else parts
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_logp_workspace_size(N, V, D), hidden)
    _check(_lib.lib().vp_linear_logp_partial(_ptr(hidden), _ptr(weight), N, V, D, vocab_start, _ptr(targets),
                                             _ptr(parts), _ptr(workspace), workspace.numel(), _stream()),
           "vp_linear_logp_partial")
    return parts


def vp_linear_entropy_partial(hidden, weight, parts=None, workspace=None):
    """Per-row entropy records over the vocabulary shard held by weight."""
    N, V, D = _linear_model(hidden, weight, "vp_linear_entropy_partial")
    _parts_arg(parts, N, hidden)
    parts = partials(N, hidden.device) if parts is None else parts
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_entropy_workspace_size(N, V, D), hidden)
    _check(_lib.lib().vp_linear_entropy_partial(_ptr(hidden), _ptr(weight), N, V, D, _ptr(parts), _ptr(workspace),
                                                workspace.numel(), _stream()), "vp_linear_entropy_partial")
    return parts


def vp_linear_kl_partial(ha, wa, hb, wb, direction: int = KL_REVERSE, parts=None, workspace=None):
    """Per-row KL records of two models over the vocabulary shard held by wa and wb."""
    N, V, Da, Db = _two_models(ha, wa, hb, wb, "vp_linear_kl_partial")
    _parts_arg(parts, N, ha)
    parts = partials(N, ha.device) if parts is None else parts
    if workspace is None:
        workspace = _workspace(_lib.lib().vp_linear_kl_workspace_size(N, V), ha)
    _check(_lib.lib().vp_linear_kl_partial(_ptr(ha), _ptr(wa), _ptr(hb), _ptr(wb), N, V, Da, Db, int(direction),
                                           _ptr(parts), _ptr(workspace), workspace.numel(), _stream()),
           "vp_linear_kl_partial")
    return parts
