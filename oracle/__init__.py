"""fp64 CPU oracle for vocab-wide logprobs, entropy, KL and fused linear logp.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` leg may import this package.
The product path (``vocab_wide_logprobs_gb300``) never imports it, and the two
share no code: this module loads ``vp_oracle.c`` (plain C, fp64, OpenMP over
rows) through ctypes and passes it numpy float64 arrays.

Every function takes exact fp64 copies of the inputs (bf16 / fp32 values upcast
without rounding) as C-contiguous ``[N, V]`` arrays and returns fp64 results.
The definitions each C function writes out, and the readings R1-R5 it takes
where the pages are silent, are listed at the top of ``vp_oracle.c``.

Parity unpinned: nothing. Every function here is pinned by ``tests/test_oracle_*``
(Decimal brute force, closed forms, finite differences, invariants, shard
merges, hand-built special rows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libvp_oracle.so")
_lock = threading.Lock()
_lib = None

REVERSE = 0  # KL(A || B)
FORWARD = 1  # KL(B || A)
ERR_TARGET = 1


def build(force: bool = False) -> str:
    """Compile vp_oracle.c with gcc into oracle/libvp_oracle.so (OpenMP if available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-Wall", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_SIGS = {
    "vpo_num_threads": ([], ctypes.c_int),
    "vpo_set_num_threads": (["i"], None),
    "vpo_logprobs_fwd": (["P", "I", "I", "I", "P", "P", "P", "P", "P"], None),
    "vpo_logprobs_bwd": (["P", "I", "I", "I", "P", "P", "P"], None),
    "vpo_logprobs_topk_fwd": (["P", "I", "I", "I", "I", "P", "P", "P"], None),
    "vpo_logprobs_topk_bwd": (["P", "I", "I", "I", "I", "P", "P", "P"], None),
    "vpo_entropy_fwd": (["P", "I", "I", "P", "P", "P"], None),
    "vpo_entropy_bwd": (["P", "I", "I", "P", "P"], None),
    "vpo_kl_fwd": (["P", "P", "I", "I", "i", "P", "P", "P", "P", "P"], None),
    "vpo_kl_bwd": (["P", "P", "I", "I", "i", "P", "P", "P"], None),
    "vpo_entropy_sharded": (["P", "I", "I", "P", "i", "P"], None),
    "vpo_kl_sharded": (["P", "P", "I", "I", "i", "P", "i", "P"], None),
    "vpo_shard_stats": (["P", "I", "I", "I", "I", "P"], None),
    "vpo_shard_kl_stats": (["P", "P", "I", "I", "i", "I", "I", "P"], None),
    "vpo_jsd_fwd": (["P", "P", "I", "I", "d", "P"], None),
    "vpo_jsd_bwd": (["P", "P", "I", "I", "d", "P", "P", "P"], None),
    "vpo_merge_entropy_records": (["P", "I", "I", "P"], None),
    "vpo_merge_kl_records": (["P", "I", "I", "P"], None),
    "vpo_linear_logits": (["P", "P", "I", "I", "I", "P"], None),
    "vpo_linear_logp_fwd": (["P", "P", "I", "I", "I", "I", "P", "P", "P", "P", "P", "P"], None),
    "vpo_linear_logp_bwd": (["P", "P", "I", "I", "I", "I", "P", "P", "P", "P", "P"], None),
    "vpo_linear_entropy_fwd": (["P", "P", "I", "I", "I", "P", "P", "P", "P"], None),
    "vpo_linear_entropy_bwd": (["P", "P", "I", "I", "I", "P", "P", "P", "P"], None),
    "vpo_linear_kl_fwd": (["P", "P", "P", "P", "I", "I", "I", "I", "i", "P", "P", "P", "P", "P", "P"], None),
    "vpo_linear_kl_bwd": (["P", "P", "P", "P", "I", "I", "I", "I", "i", "P", "P", "P", "P", "P", "P"], None),
    "vpo_linear_jsd_fwd": (["P", "P", "P", "P", "I", "I", "I", "I", "d", "P", "P"], None),
    "vpo_linear_jsd_bwd": (["P", "P", "P", "P", "I", "I", "I", "I", "d", "P", "P", "P", "P", "P", "P"], None),
}
_CT = {"P": ctypes.c_void_p, "I": ctypes.c_int64, "i": ctypes.c_int, "d": ctypes.c_double}


def load_library(path: str):
    """ctypes handle on a compiled oracle library with every signature declared."""
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = [_CT[a] for a in args]
        fn.restype = res
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def num_threads(lib=None) -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all host cores)."""
    return (lib or _load()).vpo_num_threads()


def set_num_threads(n: int, lib=None) -> None:
    """OpenMP threads for the following oracle calls (timing only; results do not depend on it)."""
    (lib or _load()).vpo_set_num_threads(int(n))


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _p(a):
    return None if a is None else a.ctypes.data


def _shape(x):
    if x.ndim != 2:
        raise ValueError("oracle inputs are [N, V] arrays")
    return x.shape


def logprobs_fwd(x, targets, vocab_start=0, lib=None):
    """Returns (logp, m, logS, err) for rows of x; targets are global ids."""
    x = _f64(x)
    N, V = _shape(x)
    t = _i64(targets)
    logp, m, logS = (np.empty(N) for _ in range(3))
    err = np.zeros(1, dtype=np.int32)
    (lib or _load()).vpo_logprobs_fwd(_p(x), N, V, vocab_start, _p(t), _p(logp), _p(m), _p(logS), _p(err))
    return logp, m, logS, int(err[0])


def logprobs_bwd(x, targets, g, vocab_start=0, lib=None):
    x = _f64(x)
    N, V = _shape(x)
    t, g = _i64(targets), _f64(g)
    dx = np.empty((N, V))
    (lib or _load()).vpo_logprobs_bwd(_p(x), N, V, vocab_start, _p(t), _p(g), _p(dx))
    return dx


def logprobs_topk_fwd(x, targets, vocab_start=0, lib=None):
    """logp [N, K] of K target ids per row (targets [N, K]); returns (logp, err)."""
    x, t = _f64(x), _i64(targets)
    N, V = _shape(x)
    K = t.shape[1]
    logp = np.empty((N, K))
    err = np.zeros(1, dtype=np.int32)
    (lib or _load()).vpo_logprobs_topk_fwd(_p(x), N, V, K, vocab_start, _p(t), _p(logp), _p(err))
    return logp, int(err[0])


def logprobs_topk_bwd(x, targets, g, vocab_start=0, lib=None):
    """Gradient of sum_k g[r, k] logp[r, k]; targets and g are [N, K]."""
    x, t, g = _f64(x), _i64(targets), _f64(g)
    N, V = _shape(x)
    K = t.shape[1]
    dx = np.empty((N, V))
    (lib or _load()).vpo_logprobs_topk_bwd(_p(x), N, V, K, vocab_start, _p(t), _p(g), _p(dx))
    return dx


def entropy_fwd(x, lib=None):
    """Returns (H, m, logS)."""
    x = _f64(x)
    N, V = _shape(x)
    H, m, logS = (np.empty(N) for _ in range(3))
    (lib or _load()).vpo_entropy_fwd(_p(x), N, V, _p(H), _p(m), _p(logS))
    return H, m, logS


def entropy_bwd(x, g, lib=None):
    x = _f64(x)
    N, V = _shape(x)
    g = _f64(g)
    dx = np.empty((N, V))
    (lib or _load()).vpo_entropy_bwd(_p(x), N, V, _p(g), _p(dx))
    return dx


def kl_fwd(a, b, direction=REVERSE, lib=None):
    """Returns (kl, ma, logSa, mb, logSb); reverse = KL(A||B), forward = KL(B||A)."""
    a, b = _f64(a), _f64(b)
    N, V = _shape(a)
    if b.shape != a.shape:
        raise ValueError("a and b differ in shape")
    kl, ma, lsa, mb, lsb = (np.empty(N) for _ in range(5))
    (lib or _load()).vpo_kl_fwd(_p(a), _p(b), N, V, int(direction), _p(kl), _p(ma), _p(lsa), _p(mb), _p(lsb))
    return kl, ma, lsa, mb, lsb


def kl_bwd(a, b, g, direction=REVERSE, lib=None):
    """Returns (dA, dB) of g * KL in the given direction."""
    a, b = _f64(a), _f64(b)
    N, V = _shape(a)
    g = _f64(g)
    da, db = np.empty((N, V)), np.empty((N, V))
    (lib or _load()).vpo_kl_bwd(_p(a), _p(b), N, V, int(direction), _p(g), _p(da), _p(db))
    return da, db


def jsd_fwd(a, b, beta, lib=None):
    """Generalized JSD per row: beta KL(q || mix) + (1 - beta) KL(p || mix), mix = beta q + (1 - beta) p
    (p = softmax(a), q = softmax(b)); beta = 0 is KL(b || a), beta = 1 is KL(a || b)."""
    a, b = _f64(a), _f64(b)
    N, V = _shape(a)
    out = np.empty(N)
    (lib or _load()).vpo_jsd_fwd(_p(a), _p(b), N, V, float(beta), _p(out))
    return out


def jsd_bwd(a, b, beta, g, lib=None):
    """(dA, dB) of sum_r g[r] JSD_r."""
    a, b, g = _f64(a), _f64(b), _f64(g)
    N, V = _shape(a)
    da, db = np.empty((N, V)), np.empty((N, V))
    (lib or _load()).vpo_jsd_bwd(_p(a), _p(b), N, V, float(beta), _p(g), _p(da), _p(db))
    return da, db


def entropy_sharded(x, cuts, lib=None):
    """Entropy from per-shard (m, S, W) merged by re-centring on the row max."""
    x = _f64(x)
    N, V = _shape(x)
    c = _i64(cuts)
    if c[0] != 0 or c[-1] != V or len(c) - 1 > 64:
        raise ValueError("cuts must run from 0 to V with at most 64 shards")
    H = np.empty(N)
    (lib or _load()).vpo_entropy_sharded(_p(x), N, V, _p(c), len(c) - 1, _p(H))
    return H


def kl_sharded(a, b, cuts, direction=REVERSE, lib=None):
    a, b = _f64(a), _f64(b)
    N, V = _shape(a)
    c = _i64(cuts)
    if c[0] != 0 or c[-1] != V or len(c) - 1 > 64:
        raise ValueError("cuts must run from 0 to V with at most 64 shards")
    kl = np.empty(N)
    (lib or _load()).vpo_kl_sharded(_p(a), _p(b), N, V, int(direction), _p(c), len(c) - 1, _p(kl))
    return kl


def shard_stats(x, lo, hi, lib=None):
    """Per-row records of the vocabulary shard [lo, hi): columns m, S, W, bad (see vpo_shard_stats)."""
    x = _f64(x)
    N, V = _shape(x)
    if not 0 <= lo <= hi <= V:
        raise ValueError("shard outside the row")
    out = np.empty((N, 4))
    (lib or _load()).vpo_shard_stats(_p(x), N, V, int(lo), int(hi), _p(out))
    return out


def shard_kl_stats(a, b, lo, hi, direction=REVERSE, lib=None):
    """Per-row KL(P||Q) records of the shard [lo, hi): m_P, S_P, m_Q, S_Q, W, bad, mismatch."""
    a, b = _f64(a), _f64(b)
    N, V = _shape(a)
    if not 0 <= lo <= hi <= V:
        raise ValueError("shard outside the row")
    out = np.empty((N, 7))
    (lib or _load()).vpo_shard_kl_stats(_p(a), _p(b), N, V, int(direction), int(lo), int(hi), _p(out))
    return out


def merge_entropy_records(recs, lib=None):
    """Entropy per row from gathered shard records [K, N, 4] (as shard_stats returns them)."""
    recs = _f64(recs)
    if recs.ndim != 3 or recs.shape[2] != 4 or not 1 <= recs.shape[0] <= 64:
        raise ValueError("records must be [K <= 64, N, 4]")
    K, N = recs.shape[:2]
    H = np.empty(N)
    (lib or _load()).vpo_merge_entropy_records(_p(recs), K, N, _p(H))
    return H


def merge_kl_records(recs, lib=None):
    """KL per row from gathered shard records [K, N, 7] (as shard_kl_stats returns them)."""
    recs = _f64(recs)
    if recs.ndim != 3 or recs.shape[2] != 7 or not 1 <= recs.shape[0] <= 64:
        raise ValueError("records must be [K <= 64, N, 7]")
    K, N = recs.shape[:2]
    kl = np.empty(N)
    (lib or _load()).vpo_merge_kl_records(_p(recs), K, N, _p(kl))
    return kl


def linear_logits(h, W, lib=None):
    """fp64 logits h . W^T (materialised; for small cases only)."""
    h, W = _f64(h), _f64(W)
    N, D = h.shape
    V = W.shape[0]
    out = np.empty((N, V))
    (lib or _load()).vpo_linear_logits(_p(h), _p(W), N, V, D, _p(out))
    return out


def linear_row_stats(h, W, rows_per_block=512):
    """Exact row max m and log S = log sum_j exp(z_j - m) of the logits z = h . W^T for every row,
    in fp64: one fp64 matrix product per block of rows (numpy), then the max and the sum of
    exponentials of each row written out. For the full-size linear workload, where every row's
    normaliser is needed and the per-row loop of linear_logp_fwd would take minutes; the two agree
    (tests/test_oracle_pins.py)."""
    h, W = _f64(h), _f64(W)
    if h.ndim != 2 or W.ndim != 2 or W.shape[1] != h.shape[1]:
        raise ValueError("hidden [N, D] and weight [V, D] disagree")
    N = h.shape[0]
    m, logS = np.empty(N), np.empty(N)
    for r0 in range(0, N, rows_per_block):
        z = h[r0:r0 + rows_per_block] @ W.T
        mb = z.max(axis=1)
        m[r0:r0 + len(mb)] = mb
        logS[r0:r0 + len(mb)] = np.log(np.exp(z - mb[:, None]).sum(axis=1))
    return m, logS


def linear_logp_dW_rows(h, W, targets, g, ids, vocab_start=0):
    """Rows `ids` (shard columns) of dW for sum_r g_r logp_r, in fp64: every row's normaliser
    (linear_row_stats), then dz[:, ids] = g (onehot - p) and dW[ids] = dz[:, ids]^T . h.
    Returns (dW rows [len(ids), D], dz[:, ids] [N, len(ids)]). Rows with a negative target
    contribute nothing; targets outside the shard are not expected here."""
    h, W = _f64(h), _f64(W)
    t, g = _i64(targets), _f64(g)
    ids = np.asarray(ids, np.int64)
    m, logS = linear_row_stats(h, W)
    z = h @ W[ids].T
    p = np.exp((z - m[:, None]) - logS[:, None])
    onehot = ((t - vocab_start)[:, None] == ids[None, :]).astype(np.float64)
    dz = np.where((t >= 0)[:, None], g[:, None] * (onehot - p), 0.0)
    return dz.T @ h, dz


def linear_logp_fwd(h, W, targets, vocab_start=0, lib=None):
    """Returns (logp, m, logS, err) of logits h . W^T, one fp64 logits row at a time."""
    h, W = _f64(h), _f64(W)
    N, D = h.shape
    V = W.shape[0]
    if W.shape[1] != D:
        raise ValueError("hidden and weight disagree on D")
    t = _i64(targets)
    logp, m, logS = (np.empty(N) for _ in range(3))
    scratch = np.empty((max(1, num_threads(lib)), V))
    err = np.zeros(1, dtype=np.int32)
    (lib or _load()).vpo_linear_logp_fwd(_p(h), _p(W), N, V, D, vocab_start, _p(t), _p(logp), _p(m),
                                _p(logS), _p(scratch), _p(err))
    return logp, m, logS, int(err[0])


def linear_logp_bwd(h, W, targets, g, vocab_start=0, want_dh=True, want_dW=True, lib=None):
    """Returns (dhidden, dW) of sum_r g_r logp_r; either is None when not wanted."""
    h, W = _f64(h), _f64(W)
    N, D = h.shape
    V = W.shape[0]
    t, g = _i64(targets), _f64(g)
    dh = np.empty((N, D)) if want_dh else None
    dW = np.empty((V, D)) if want_dW else None
    dz = np.empty((N, V))
    (lib or _load()).vpo_linear_logp_bwd(_p(h), _p(W), N, V, D, vocab_start, _p(t), _p(g), _p(dh),
                                _p(dW), _p(dz))
    return dh, dW


def _linear_shapes(h, W):
    h, W = _f64(h), _f64(W)
    if h.ndim != 2 or W.ndim != 2 or W.shape[1] != h.shape[1]:
        raise ValueError("hidden [N, D] and weight [V, D] disagree")
    return h, W, h.shape[0], W.shape[0], h.shape[1]


def linear_entropy_fwd(h, W, lib=None):
    """Returns (H, m, logS) of the logits h . W^T (materialised in fp64; small cases only)."""
    h, W, N, V, D = _linear_shapes(h, W)
    H, m, logS = (np.empty(N) for _ in range(3))
    logits = np.empty((N, V))
    (lib or _load()).vpo_linear_entropy_fwd(_p(h), _p(W), N, V, D, _p(H), _p(m), _p(logS), _p(logits))
    return H, m, logS


def linear_entropy_bwd(h, W, g, want_dh=True, want_dW=True, lib=None):
    """Returns (dhidden, dW) of sum_r g_r H_r; either is None when not wanted."""
    h, W, N, V, D = _linear_shapes(h, W)
    g = _f64(g)
    dh = np.empty((N, D)) if want_dh else None
    dW = np.empty((V, D)) if want_dW else None
    scratch = np.empty((2, N, V))
    (lib or _load()).vpo_linear_entropy_bwd(_p(h), _p(W), N, V, D, _p(g), _p(dh), _p(dW), _p(scratch))
    return dh, dW


def linear_kl_fwd(ha, Wa, hb, Wb, direction=REVERSE, lib=None):
    """KL between model A (ha . Wa^T) and model B (hb . Wb^T); reverse = KL(A||B).
    Returns (kl, ma, logSa, mb, logSb)."""
    ha, Wa, N, V, Da = _linear_shapes(ha, Wa)
    hb, Wb, Nb, Vb, Db = _linear_shapes(hb, Wb)
    if (Nb, Vb) != (N, V):
        raise ValueError("the two models disagree on N or V")
    kl, ma, lsa, mb, lsb = (np.empty(N) for _ in range(5))
    scratch = np.empty((2, N, V))
    (lib or _load()).vpo_linear_kl_fwd(_p(ha), _p(Wa), _p(hb), _p(Wb), N, V, Da, Db, int(direction), _p(kl),
                                       _p(ma), _p(lsa), _p(mb), _p(lsb), _p(scratch))
    return kl, ma, lsa, mb, lsb


def linear_kl_bwd(ha, Wa, hb, Wb, g, direction=REVERSE, want=(True, True, True, True), lib=None):
    """Returns (dha, dWa, dhb, dWb) of sum_r g_r KL_r; entries not wanted are None."""
    ha, Wa, N, V, Da = _linear_shapes(ha, Wa)
    hb, Wb, _, _, Db = _linear_shapes(hb, Wb)
    g = _f64(g)
    outs = [np.empty(s) if w else None for s, w in zip(((N, Da), (V, Da), (N, Db), (V, Db)), want)]
    scratch = np.empty((4, N, V))
    (lib or _load()).vpo_linear_kl_bwd(_p(ha), _p(Wa), _p(hb), _p(Wb), N, V, Da, Db, int(direction), _p(g),
                                       *[_p(o) for o in outs], _p(scratch))
    return tuple(outs)


def linear_jsd_fwd(ha, Wa, hb, Wb, beta, lib=None):
    """Generalized JSD (jsd_fwd) between model A (ha . Wa^T, the student) and model B (hb . Wb^T)."""
    ha, Wa, N, V, Da = _linear_shapes(ha, Wa)
    hb, Wb, Nb, Vb, Db = _linear_shapes(hb, Wb)
    if (Nb, Vb) != (N, V):
        raise ValueError("the two models disagree on N or V")
    out = np.empty(N)
    scratch = np.empty((2, N, V))
    (lib or _load()).vpo_linear_jsd_fwd(_p(ha), _p(Wa), _p(hb), _p(Wb), N, V, Da, Db, float(beta), _p(out),
                                        _p(scratch))
    return out


def linear_jsd_bwd(ha, Wa, hb, Wb, beta, g, want=(True, True, True, True), lib=None):
    """Returns (dha, dWa, dhb, dWb) of sum_r g_r JSD_r; entries not wanted are None."""
    ha, Wa, N, V, Da = _linear_shapes(ha, Wa)
    hb, Wb, _, _, Db = _linear_shapes(hb, Wb)
    g = _f64(g)
    outs = [np.empty(s) if w else None for s, w in zip(((N, Da), (V, Da), (N, Db), (V, Db)), want)]
    scratch = np.empty((4, N, V))
    (lib or _load()).vpo_linear_jsd_bwd(_p(ha), _p(Wa), _p(hb), _p(Wb), N, V, Da, Db, float(beta), _p(g),
                                        *[_p(o) for o in outs], _p(scratch))
    return tuple(outs)
