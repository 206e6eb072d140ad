"""The failure path of the bounded device waits, exercised without a fault.

Every tensor-core kernel waits on mbarriers through bounded polls; when one
gives up, the kernel records POETX_ERR_TIMEOUT in the library's device error
word and winds down instead of hanging, and poetx_stream_status() reports it.
poetx_diag_expire_wait launches one thread whose wait cannot complete (an
mbarrier in its own shared memory that nothing arrives on; no TMA, MMA or
remote arrive in flight) with a short poll limit.  The test checks the status
the host reads, that the status is cleared by reading it, and that the next
ordinary call computes correctly on the same context.
"""
import ctypes

import pytest
import torch

import oracle
from orthogonal_equivalence_neumann_b300 import _lib, inputs

pytestmark = pytest.mark.gpu

TIMEOUT = 6


def _status():
    return _lib.load().poetx_stream_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("cluster_scope", [0, 1])
def test_expired_wait_is_reported_and_the_context_stays_usable(cluster_scope):
    assert _status() == 0
    _lib.poetx_diag_expire_wait(cluster_scope, 256)
    assert _status() == TIMEOUT
    assert _status() == 0          # reading the status cleared the error word
    # an ordinary call afterwards runs and is right (tiny fp32 blocks, 1e-5)
    th = inputs.make_theta(8, 32, 0.01, 4242)
    Q = torch.empty(8, 32, 32, dtype=torch.float32, device="cuda")
    _lib.poetx_cayley_neumann(th.cuda(), 32, 4, Q)
    assert _status() == 0
    ref = oracle.cnp(th.double().numpy(), 32, 4)
    assert oracle.rel_fro(Q.double().cpu().numpy(), ref) <= 1e-5
