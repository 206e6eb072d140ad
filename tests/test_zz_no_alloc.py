"""poetx_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a host framework that owns all device memory through its own
pool, or a loop in which allocation is forbidden after start-up) get the
forward's scratch from a static device array inside the library instead of a
caller-provided workspace.  This test calls the entry point through the C ABI
twice in a row (the array keeps the previous call's contents) and checks its
outputs against poetx_forward with a caller workspace: the same kernels run on
the same inputs, so the results must be identical bit for bit (a read of stale
scratch would show here).  It also checks that the calls take no device
memory: neither the driver's free-memory figure nor PyTorch's allocator moves
across them.  This file is collected last, so that a run stopping at the first
failure has run every other test.
"""
import ctypes

import pytest
import torch

from orthogonal_equivalence_neumann_b300 import TransformedLinear, _lib, inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    inputs.LinearCase("noalloc_bf16", 512, 768, 128, 256, 3, 300, 0.005, "bf16", 9001),
    inputs.LinearCase("noalloc_f32", 256, 256, 32, 32, 4, 64, 0.01, "f32", 9002),
])
def test_noalloc_forward_matches_workspace_forward_twice(case):
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T)
    lay.cayley_neumann()
    x = inp["x"].cuda()
    y_ref = lay.forward(x)
    z_ref = lay.z[:case.T].clone()
    args = (x, lay.W0m, lay.Q_P, lay.Q_R, lay.perm_in, lay.inv_in, lay.perm_out, lay.inv_out,
            case.b_in, case.b_out)
    # every output buffer exists before the memory figures are taken
    outs = [(torch.full_like(y_ref, float("nan")), torch.full_like(z_ref, float("nan")))
            for _ in range(2)]
    y_noz = torch.full_like(y_ref, float("nan"))
    # a first call sets the library up on this device (the array's address)
    _lib.poetx_forward_noalloc(*args, torch.empty_like(y_ref), None)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    alloc_before = torch.cuda.memory_allocated()
    for y, z in outs:
        _lib.poetx_forward_noalloc(*args, y, z)
        _lib.poetx_stream_status()
    # without a saved z the forward keeps z in the static array too
    _lib.poetx_forward_noalloc(*args, y_noz, None)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert torch.cuda.memory_allocated() == alloc_before
    for call, (y, z) in enumerate(outs):
        assert torch.equal(y, y_ref), ("call", call, "y")
        assert torch.equal(z, z_ref), ("call", call, "z")
    assert torch.equal(y_noz, y_ref)


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
