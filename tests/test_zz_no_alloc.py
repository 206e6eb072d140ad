"""poetx_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a host framework that owns all device memory through its own
pool, or a loop in which allocation is forbidden after start-up) get the
forward's scratch from a static device array inside the library instead of a
caller-provided workspace.  This test calls the entry point through the C ABI
twice in a row (the array keeps the previous call's contents) and checks its
outputs against poetx_forward with a caller workspace.  This file is collected
last, so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from orthogonal_equivalence_neumann_b300 import TransformedLinear, _lib, inputs

pytestmark = pytest.mark.gpu


def _rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("case,tol", [
    (inputs.LinearCase("noalloc_bf16", 512, 768, 128, 256, 3, 300, 0.005, "bf16", 9001), 2e-2),
    (inputs.LinearCase("noalloc_f32", 256, 256, 32, 32, 4, 64, 0.01, "f32", 9002), 1e-5),
])
def test_noalloc_forward_matches_workspace_forward_twice(case, tol):
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T)
    lay.cayley_neumann()
    x = inp["x"].cuda()
    y_ref = lay.forward(x)
    z_ref = lay.z[:case.T].clone()
    for call in range(2):
        y = torch.full_like(y_ref, float("nan"))
        z = torch.full_like(z_ref, float("nan"))
        _lib.poetx_forward_noalloc(x, lay.W0m, lay.Q_P, lay.Q_R, lay.perm_in, lay.inv_in,
                                   lay.perm_out, lay.inv_out, case.b_in, case.b_out, y, z)
        _lib.poetx_stream_status()
        torch.cuda.synchronize()
        assert torch.isfinite(y.float()).all() and torch.isfinite(z.float()).all()
        assert _rel(y, y_ref) <= tol, ("call", call, _rel(y, y_ref))
        assert _rel(z, z_ref) <= tol, ("call", call, _rel(z, z_ref))
    # without a saved z the forward keeps z in the static array too
    y = torch.full_like(y_ref, float("nan"))
    _lib.poetx_forward_noalloc(x, lay.W0m, lay.Q_P, lay.Q_R, lay.perm_in, lay.inv_in,
                               lay.perm_out, lay.inv_out, case.b_in, case.b_out, y, None)
    _lib.poetx_stream_status()
    assert _rel(y, y_ref) <= tol


def test_noalloc_rejects_sizes_beyond_the_static_array():
    lib = _lib.load()
    T, d = 4096, 2048
    need = lib.poetx_workspace_bytes(T, d, d, 256, 256, _lib.BF16)
    assert need > 32 << 20
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    code = lib.poetx_forward_noalloc(p, p, p, p, p, p, p, p, T, d, d, 256, 256, _lib.BF16, p, p,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 2   # POETX_ERR_SHAPE, before anything is launched
