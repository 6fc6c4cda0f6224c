"""The C-ABI library: it loads, exports every entry point include/vp.h declares,
and rejects bad arguments on the host before any device work (CPU-only checks)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from vocab_wide_logprobs_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vp.h")

OK, ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_LAYOUT, ERR_ALIGN, ERR_LAUNCH, ERR_ARG, ERR_DEVICE = range(9)


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"VP_API\s+[\w\s\*]*?\b(vp_\w+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("vp_logprobs_fwd", "vp_logprobs_bwd", "vp_entropy_fwd", "vp_entropy_bwd", "vp_kl_fwd",
              "vp_kl_bwd", "vp_status_string", "vp_version"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = _lib.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (vp_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
    assert lib.vp_version() >= 1
    assert _lib.status_string(ERR_ALIGN) == "misaligned pointer"


def test_library_is_built_for_sm_103a():
    # the fatbinary carries only sm_103a code (checked from the build flags, not by reading the binary)
    from vocab_wide_logprobs_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


# ---------------------------------------------------------------------------
# host-side argument checks: these return before any device is touched
# ---------------------------------------------------------------------------
FAKE = ctypes.c_void_p(0x100000)      # never dereferenced: every call below fails its host checks
FAKE_ODD = ctypes.c_void_p(0x100001)


def ent_fwd(x=FAKE, dtype=1, N=4, V=16, R=4, s_o=0, s_i=16, H=FAKE, stats=FAKE):
    return _lib.lib().vp_entropy_fwd(x, dtype, N, V, R, s_o, s_i, H, stats, None)


def test_status_codes_for_bad_arguments():
    assert ent_fwd(dtype=7) == ERR_DTYPE
    assert ent_fwd(N=-1) == ERR_SHAPE
    assert ent_fwd(V=0) == ERR_SHAPE
    assert ent_fwd(V=2**31) == ERR_SHAPE
    assert ent_fwd(R=0) == ERR_SHAPE
    assert ent_fwd(s_i=-16) == ERR_LAYOUT
    assert ent_fwd(s_o=-1) == ERR_LAYOUT
    assert ent_fwd(x=None) == ERR_NULL
    assert ent_fwd(H=None) == ERR_NULL
    assert ent_fwd(x=FAKE_ODD) == ERR_ALIGN
    assert ent_fwd(stats=FAKE_ODD) == ERR_ALIGN
    assert ent_fwd(stats=ctypes.c_void_p(0x100008)) == ERR_ALIGN  # records need 16-byte alignment
    assert ent_fwd(N=0, x=None, H=None, stats=None) == OK  # N = 0 queues nothing
    L = _lib.lib()
    args = (FAKE, FAKE, 1, 4, 16, 4, 0, 16)
    assert L.vp_kl_fwd(*args, 2, FAKE, FAKE, FAKE, None) == ERR_ARG
    assert L.vp_kl_bwd(*args, 0, FAKE, FAKE, FAKE, None, None, None) == ERR_ARG
    assert L.vp_kl_bwd(FAKE, FAKE, 1, 0, 16, 4, 0, 16, 0, FAKE, FAKE, FAKE, None, None, None) == OK
    assert L.vp_logprobs_fwd(FAKE, 1, 4, 16, 4, 0, 16, 0, FAKE_ODD, FAKE, FAKE, None, None) == ERR_ALIGN
    assert L.vp_logprobs_bwd(FAKE, 1, 4, 16, 4, 0, 16, 0, FAKE, FAKE, FAKE, None, None, None) == ERR_NULL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device status; needs a machine without a GPU")
def test_no_device_status_without_gpu():
    assert ent_fwd() == ERR_DEVICE


def test_binding_rejects_bad_layouts_before_calling():
    from vocab_wide_logprobs_gb300 import VPError, rows_of
    x = torch.zeros(4, 6, 16)
    assert rows_of(x) == (24, 16, 6, 96, 16)
    assert rows_of(x[:, :-1]) == (20, 16, 5, 96, 16)
    assert rows_of(x[0]) == (6, 16, 6, 0, 16)
    with pytest.raises(VPError):
        rows_of(x.transpose(1, 2))
    with pytest.raises(VPError):
        rows_of(torch.zeros(3))


def test_sharded_entry_points_check_arguments_on_the_host():
    lib = _lib.lib()
    # merges: K >= 1, parts non-NULL and 8-byte aligned, a valid direction
    assert lib.vp_entropy_merge(FAKE, 0, 4, FAKE, FAKE, None) == ERR_SHAPE
    assert lib.vp_entropy_merge(None, 2, 4, FAKE, FAKE, None) == ERR_NULL
    assert lib.vp_entropy_merge(FAKE_ODD, 2, 4, FAKE, FAKE, None) == ERR_ALIGN
    assert lib.vp_entropy_merge(None, 2, 0, None, None, None) == OK          # N = 0 queues nothing
    assert lib.vp_logprobs_merge(FAKE, 2, 4, None, FAKE, None, None) == ERR_NULL
    assert lib.vp_kl_merge(FAKE, 2, 4, 5, FAKE, FAKE, FAKE, None) == ERR_ARG
    assert lib.vp_kl_merge(FAKE, 2, 4, 0, FAKE, FAKE_ODD, FAKE, None) == ERR_ALIGN
    # partials: the same row checks as the forward calls
    assert lib.vp_entropy_partial(FAKE, 9, 4, 16, 4, 0, 16, FAKE, None) == ERR_DTYPE
    assert lib.vp_entropy_partial(FAKE, 1, 4, 0, 4, 0, 16, FAKE, None) == ERR_SHAPE
    assert lib.vp_logprobs_partial(FAKE, 1, 4, 16, 4, 0, 16, 0, None, FAKE, None) == ERR_NULL
    assert lib.vp_logprobs_partial(FAKE, 1, 4, 16, 4, 0, 16, 0, FAKE, FAKE_ODD, None) == ERR_ALIGN
    assert lib.vp_kl_partial(FAKE, FAKE, 1, 4, 16, 4, 0, 16, 3, FAKE, None) == ERR_ARG
    assert lib.vp_kl_partial(FAKE, FAKE, 1, 4, 16, 4, -1, 16, 0, FAKE, None) == ERR_LAYOUT


def test_jsd_entry_points_check_beta_first():
    lib = _lib.lib()
    for beta in (-0.1, 1.5, float("nan")):
        assert lib.vp_jsd_fwd(FAKE, FAKE, 1, 4, 16, 4, 0, 16, beta, FAKE, FAKE, FAKE, None) == ERR_ARG
        assert lib.vp_jsd_bwd(FAKE, FAKE, 1, 4, 16, 4, 0, 16, beta, FAKE, FAKE, FAKE, FAKE, FAKE, None) == ERR_ARG
    assert lib.vp_jsd_fwd(FAKE, FAKE, 7, 4, 16, 4, 0, 16, 0.5, FAKE, FAKE, FAKE, None) == ERR_DTYPE
    assert lib.vp_jsd_bwd(FAKE, FAKE, 1, 4, 16, 4, 0, 16, 0.5, FAKE, FAKE, FAKE, None, None, None) == ERR_ARG
    assert lib.vp_jsd_fwd(FAKE, FAKE, 1, 4, 16, 4, 0, 16, 0.5, FAKE_ODD, FAKE, FAKE, None) == ERR_ALIGN


def test_topk_entry_points_check_arguments_on_the_host():
    lib = _lib.lib()
    row = (FAKE, 1, 4, 16, 4, 0, 16, 0)                  # x, dtype, N, V, R, s_o, s_i, vocab_start
    assert lib.vp_logprobs_topk_fwd(*row, FAKE, 0, FAKE, FAKE, None, None) == ERR_SHAPE        # K = 0
    assert lib.vp_logprobs_topk_fwd(*row, None, 3, FAKE, FAKE, None, None) == ERR_NULL
    assert lib.vp_logprobs_topk_fwd(*row, FAKE_ODD, 3, FAKE, FAKE, None, None) == ERR_ALIGN
    assert lib.vp_logprobs_topk_fwd(FAKE, 5, 4, 16, 4, 0, 16, 0, FAKE, 3, FAKE, FAKE, None, None) == ERR_DTYPE
    assert lib.vp_logprobs_topk_bwd(*row, FAKE, 3, FAKE, None, FAKE, None, None) == ERR_NULL
    assert lib.vp_logprobs_topk_bwd(*row, FAKE, 3, ctypes.c_void_p(0x100008), FAKE, FAKE, None, None) == ERR_ALIGN
    assert lib.vp_logprobs_topk_fwd(None, 1, 0, 16, 1, 0, 16, 0, None, 3, None, None, None, None) == OK   # N = 0


def test_linear_entropy_kl_entry_points_check_arguments_on_the_host():
    lib = _lib.lib()
    size_t = ctypes.c_size_t
    ws = size_t(1 << 30)
    # hidden sizes must be positive multiples of 64
    assert lib.vp_linear_entropy_fwd(FAKE, FAKE, 4, 16, 96, FAKE, FAKE, FAKE, ws, None) == ERR_SHAPE
    assert lib.vp_linear_entropy_workspace_size(4, 16, 96) == 0
    assert lib.vp_linear_entropy_fwd(FAKE, None, 4, 16, 64, FAKE, FAKE, FAKE, ws, None) == ERR_NULL
    assert lib.vp_linear_entropy_fwd(FAKE_ODD, FAKE, 4, 16, 64, FAKE, FAKE, FAKE, ws, None) == ERR_ALIGN
    assert lib.vp_linear_entropy_fwd(FAKE, FAKE, 4, 16, 64, FAKE, FAKE, FAKE, size_t(16), None) == ERR_ARG
    assert lib.vp_linear_entropy_bwd(FAKE, FAKE, 4, 16, 64, FAKE, FAKE, None, None, 0, FAKE, ws, None) == ERR_ARG
    # precision: VP_GRAD_EXACT (0) or VP_GRAD_FAST (1) only
    assert lib.vp_linear_entropy_bwd(FAKE, FAKE, 4, 16, 64, FAKE, FAKE, FAKE, None, 2, FAKE, ws, None) == ERR_ARG
    assert lib.vp_linear_entropy_fwd(None, None, 0, 16, 64, None, None, None, size_t(0), None) == OK   # N = 0
    two = (FAKE, FAKE, FAKE, FAKE, 4, 16)
    assert lib.vp_linear_kl_fwd(*two, 64, 100, 0, FAKE, FAKE, FAKE, FAKE, ws, None) == ERR_SHAPE     # Db
    assert lib.vp_linear_kl_fwd(*two, 64, 128, 2, FAKE, FAKE, FAKE, FAKE, ws, None) == ERR_ARG       # direction
    assert lib.vp_linear_kl_fwd(*two, 64, 128, 0, FAKE, FAKE, FAKE, FAKE, size_t(64), None) == ERR_ARG
    assert lib.vp_linear_kl_fwd(*two, 64, 128, 0, FAKE, FAKE_ODD, FAKE, FAKE, ws, None) == ERR_ALIGN
    assert lib.vp_linear_kl_bwd(*two, 64, 128, 1, FAKE, FAKE, FAKE, None, None, None, None, 0, FAKE, ws,
                                None) == ERR_ARG                                                  # no output
    assert lib.vp_linear_kl_bwd(*two, 64, 128, 1, FAKE, FAKE, None, FAKE, None, None, None, 0, FAKE, ws,
                                None) == ERR_NULL
    assert lib.vp_linear_kl_bwd(*two, 64, 128, 1, FAKE, FAKE, FAKE, FAKE, None, None, None, -1, FAKE, ws,
                                None) == ERR_ARG                                                  # precision
    assert lib.vp_linear_kl_bwd_workspace_size(4, 16, 64, 128) > 0
    assert lib.vp_linear_kl_workspace_size(4, 0) == 0


def test_linear_jsd_entry_points_check_beta_first():
    lib = _lib.lib()
    ws = ctypes.c_size_t(1 << 30)
    two = (FAKE, FAKE, FAKE, FAKE, 4, 16, 64, 128)
    for beta in (-0.1, 1.5, float("nan")):
        assert lib.vp_linear_jsd_fwd(*two, beta, FAKE, FAKE, FAKE, FAKE, ws, None) == ERR_ARG
        assert lib.vp_linear_jsd_bwd(*two, beta, FAKE, FAKE, FAKE, FAKE, None, None, None, 0, FAKE, ws,
                                     None) == ERR_ARG
    assert lib.vp_linear_jsd_fwd(FAKE, FAKE, FAKE, FAKE, 4, 16, 64, 96, 0.5, FAKE, FAKE, FAKE, FAKE, ws,
                                 None) == ERR_SHAPE
    assert lib.vp_linear_jsd_bwd(*two, 0.5, FAKE, FAKE, FAKE, None, None, None, None, 0, FAKE, ws, None) == ERR_ARG
    assert lib.vp_linear_jsd_bwd(*two, 0.5, FAKE, FAKE, FAKE, FAKE, None, None, None, 5, FAKE, ws, None) == ERR_ARG
    assert lib.vp_linear_jsd_fwd(*two, 0.5, FAKE_ODD, FAKE, FAKE, FAKE, ws, None) == ERR_ALIGN
    assert lib.vp_linear_jsd_workspace_size(4, 16) == lib.vp_linear_kl_workspace_size(4, 16)


def test_linear_partial_entry_points_check_arguments_on_the_host():
    lib = _lib.lib()
    ws = ctypes.c_size_t(1 << 30)
    assert lib.vp_linear_logp_partial(FAKE, FAKE, 4, 16, 96, 0, FAKE, FAKE, FAKE, ws, None) == ERR_SHAPE   # D
    assert lib.vp_linear_logp_partial(FAKE, FAKE, 4, 16, 64, 0, FAKE, None, FAKE, ws, None) == ERR_NULL   # parts
    assert lib.vp_linear_logp_partial(FAKE, FAKE, 4, 16, 64, 0, FAKE_ODD, FAKE, FAKE, ws, None) == ERR_ALIGN
    assert lib.vp_linear_logp_partial(FAKE, FAKE, 4, 16, 64, 0, FAKE, FAKE, FAKE, ctypes.c_size_t(8),
                                      None) == ERR_ARG                                             # workspace
    assert lib.vp_linear_logp_partial(None, None, 0, 16, 64, 0, None, None, None, ctypes.c_size_t(0), None) == OK
    assert lib.vp_linear_entropy_partial(FAKE, FAKE, 4, 0, 64, FAKE, FAKE, ws, None) == ERR_SHAPE        # V
    assert lib.vp_linear_entropy_partial(FAKE, FAKE, 4, 16, 64, FAKE_ODD, FAKE, ws, None) == ERR_ALIGN
    two = (FAKE, FAKE, FAKE, FAKE, 4, 16, 64, 128)
    assert lib.vp_linear_kl_partial(*two, 2, FAKE, FAKE, ws, None) == ERR_ARG                           # direction
    assert lib.vp_linear_kl_partial(*two, 0, None, FAKE, ws, None) == ERR_NULL
    assert lib.vp_linear_kl_partial(FAKE, FAKE, FAKE, FAKE, 4, 16, 64, 32, 1, FAKE, FAKE, ws, None) == ERR_SHAPE


def test_binding_wraps_every_entry_point():
    import vocab_wide_logprobs_gb300 as vp
    missing = [n for n in declared_functions() if not hasattr(vp, n)]
    assert not missing, missing
    assert vp.vp_version() >= 1 and vp.vp_status_string(ERR_ARG) == "invalid argument"
    assert vp.vp_linear_kl_workspace_size(4, 16) == vp.vp_linear_jsd_workspace_size(4, 16) > 0


def test_host_transfers_check_arguments_on_the_host():
    lib = _lib.lib()
    assert lib.vp_upload(None, FAKE, ctypes.c_size_t(16), None) == ERR_NULL
    assert lib.vp_download(FAKE, None, ctypes.c_size_t(16), None) == ERR_NULL
    assert lib.vp_upload(None, None, ctypes.c_size_t(0), None) == OK        # nothing to copy


def test_row_split_setting_checks_its_value():
    # host-side setting: 1 or 2 CTAs per row in the forward scans, anything else refused and ignored
    L = _lib.lib()
    old = L.vp_get_row_split()
    assert old in (1, 2)
    try:
        for bad in (0, 3, -1, 64):
            assert L.vp_set_row_split(bad) == ERR_ARG
            assert L.vp_get_row_split() == old
        assert L.vp_set_row_split(2) == OK and L.vp_get_row_split() == 2
        assert L.vp_set_row_split(1) == OK and L.vp_get_row_split() == 1
    finally:
        L.vp_set_row_split(old)
