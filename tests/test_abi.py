"""The C-ABI library loads and exports every symbol ``include/poetx.h`` declares,
and its host-side argument checks reject bad calls before anything is launched.
No compute call is made here: these run without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT
from orthogonal_equivalence_neumann_b300 import _lib, build as libbuild

HEADER = os.path.join(ROOT, "include", "poetx.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(poetx_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for must in ("poetx_cayley_neumann", "poetx_forward", "poetx_backward", "poetx_invert_perm",
                 "poetx_check_perm", "poetx_merge_w0", "poetx_workspace_bytes"):
        assert must in syms


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (poetx_\w+)", out))
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, missing
    assert sorted(_lib.EXPORTS) == declared_symbols()
    for s in declared_symbols():
        assert getattr(lib, s) is not None


def test_status_strings_and_version(lib):
    for code, name in _lib.STATUS.items():
        assert lib.poetx_status_string(code).decode() == name
    assert lib.poetx_version() >= 100


def test_workspace_bytes_host_logic(lib):
    f = lib.poetx_workspace_bytes
    assert f(64, 256, 256, 32, 32, _lib.F32) > 0
    assert f(64, 256, 256, 33, 32, _lib.F32) == 0      # b not a power of two
    assert f(64, 250, 256, 32, 32, _lib.F32) == 0      # d % b != 0
    assert f(-1, 256, 256, 32, 32, _lib.F32) == 0
    assert f(64, 256, 256, 32, 32, 7) == 0             # bad dtype
    # monotone in T and at least the u buffer of the forward
    a, b = f(64, 2048, 2048, 256, 256, _lib.BF16), f(128, 2048, 2048, 256, 256, _lib.BF16)
    assert b > a >= 64 * 2048 * 2


def test_host_validation_rejects_before_launch(lib):
    null = None
    # bad block size, bad n, bad dtype, negative nb: rejected on the host
    assert lib.poetx_cayley_neumann(null, 4, 24, 3, null, _lib.F32, null) == 3
    assert lib.poetx_cayley_neumann(null, 4, 32, 0, null, _lib.F32, null) == 1
    assert lib.poetx_cayley_neumann(null, 4, 32, 3, null, 9, null) == 1
    assert lib.poetx_cayley_neumann(null, -1, 32, 3, null, _lib.F32, null) == 2
    assert lib.poetx_cayley_neumann(null, 4, 32, 3, null, _lib.F32, null) == 1   # null pointers
    # misaligned pointer
    assert lib.poetx_cayley_neumann(ctypes.c_void_p(8), 4, 32, 3, ctypes.c_void_p(16),
                                    _lib.F32, null) == 1
    pair = lib.poetx_cayley_neumann_pair
    assert pair(null, 4, 24, null, 4, 32, 3, null, null, _lib.BF16, null) == 3   # b_P unsupported
    assert pair(null, 4, 32, null, -1, 32, 3, null, null, _lib.BF16, null) == 2  # nb_R < 0
    assert pair(null, 4, 32, null, 4, 32, 0, null, null, _lib.BF16, null) == 1   # n < 1
    assert pair(null, 4, 32, null, 0, 32, 3, null, null, _lib.BF16, null) == 1   # null theta_P
    assert pair(null, 0, 32, null, 0, 32, 3, null, null, _lib.BF16, null) == 0   # nothing to do
    assert lib.poetx_cayley_neumann_backward(null, null, 4, 32, 0, null, null) == 1
    assert lib.poetx_invert_perm(null, null, -3, null) == 2
    assert lib.poetx_merge_w0(null, null, 0, 4, _lib.F32, null, null, null) == 2
    fwd = lib.poetx_forward
    args = [null] * 8 + [16, 256, 256, 32, 32, _lib.F32, null, null, null, 0, null]
    assert fwd(*args) == 1                                    # null weights
    args2 = list(args)
    args2[11] = 24                                            # b_in unsupported
    assert fwd(*args2) == 3
    args3 = list(args)
    args3[9] = 250                                            # d_in % b_in != 0
    assert fwd(*args3) == 2
    bwd = lib.poetx_backward
    bargs = [null] * 5 + [0] + [null] * 7 + [16, 256, 256, 32, 32, _lib.F32, null, null, null,
                                            null, 0, null]
    assert bwd(*bargs) == 1                                   # n < 1


def test_fold_and_xq_host_logic(lib):
    """Workspace sizes and argument checks of the inner-loop fold and POET-XQ
    entry points (host only: every call here returns before any launch)."""
    null = None
    fb = lib.poetx_fold_workspace_bytes
    # one [d_out, d_in] matrix at least; invalid sizes give 0
    assert fb(384, 256, 32, 64, _lib.BF16) >= 384 * 256 * 2
    assert fb(384, 256, 32, 64, _lib.F32) >= 384 * 256 * 4
    assert fb(384, 250, 32, 64, _lib.F32) == 0          # d_in % b_in != 0
    assert fb(384, 256, 24, 64, _lib.F32) == 0          # b not a power of two
    assert fb(384, 256, 32, 64, 5) == 0                 # bad dtype
    fold = lib.poetx_fold_w0
    ok_ptr = ctypes.c_void_p(4096)
    args = [ok_ptr] * 5
    assert fold(*args, 384, 256, 32, 64, _lib.F32, ok_ptr, ok_ptr, 0, null) == 2   # workspace too small
    assert fold(*args, 384, 256, 32, 64, 7, ok_ptr, ok_ptr, 1 << 30, null) == 1    # bad dtype
    assert fold(null, *args[1:], 384, 256, 32, 64, _lib.F32, ok_ptr, ok_ptr, 1 << 30, null) == 1
    assert fold(*args, 384, 256, 48, 64, _lib.F32, ok_ptr, ok_ptr, 1 << 30, null) == 3  # b_in = 48
    # POET-XQ: the workspace adds the dequantised weight to the layer's
    wq, w = lib.poetx_workspace_bytes_xq, lib.poetx_workspace_bytes
    for dt, es in ((_lib.F32, 4), (_lib.BF16, 2)):
        extra = -(-2048 * 2048 * es // 256) * 256
        assert wq(1024, 2048, 2048, 256, 256, dt) == w(1024, 2048, 2048, 256, 256, dt) + extra
    assert wq(64, 250, 256, 2, 32, _lib.F32) == 0       # d_in % 4 != 0 is not supported
    q = lib.poetx_quantize_w0
    assert q(ok_ptr, 16, 10, _lib.F32, ok_ptr, ok_ptr, null) == 2       # d_in % 4 != 0
    assert q(ok_ptr, 16, 16, 9, ok_ptr, ok_ptr, null) == 1              # bad dtype
    assert q(ok_ptr, 16, 16, _lib.F32, null, ok_ptr, null) == 1         # null codes
    assert q(ctypes.c_void_p(4100), 16, 16, _lib.F32, ok_ptr, ok_ptr, null) == 1   # misaligned
    dq = lib.poetx_dequantize_w0
    assert dq(ok_ptr, null, 16, 16, _lib.BF16, ok_ptr, null) == 1       # null scales
    assert dq(ok_ptr, ok_ptr, 0, 16, _lib.BF16, ok_ptr, null) == 2      # no rows
    fx = lib.poetx_forward_xq
    assert fx(*([ok_ptr] * 9), 64, 256, 256, 32, 32, _lib.F32, ok_ptr, null, ok_ptr, 0, null) == 2


def test_diag_expire_wait_rejects_bad_arguments(lib):
    # host checks only: nothing is launched for arguments out of range
    assert lib.poetx_diag_expire_wait(2, 10, None) == 1
    assert lib.poetx_diag_expire_wait(-1, 10, None) == 1
    assert lib.poetx_diag_expire_wait(0, 0, None) == 1
    assert lib.poetx_diag_expire_wait(1, (1 << 20) + 1, None) == 1
