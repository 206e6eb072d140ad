"""CPU oracle for the POET-X transformed linear layer (double precision).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library (``orthogonal_equivalence_neumann_b300``)
and neither imports the other; the GPU path never falls back to it.

The arithmetic lives in ``poetx_oracle.c`` (plain loops, IEEE double); this
module only marshals numpy arrays.  Source of the method: the page "POET-X:
Memory-efficient LLM Training by Scaling Orthogonal Transformation"
(gist.science technical summary), section 2.A-2.E.  Every function below names
the part it follows; the conventions the pages leave open are stated at the top
of ``poetx_oracle.c``.

Pins (see ``tests/test_oracle_pins.py``): every function here is checked
against closed forms, library routines, hand-derived golden values or finite
differences.  Agreement with the authors' own (unpublished) code is not
checkable: the pages print no numeric example.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_dp = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_ip = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")


def _load(path):
    """Load an oracle build at ``path`` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    c_int, c_long = ctypes.c_int, ctypes.c_long
    sig = {
        "orc_skew_count": (c_long, [c_int]),
        "orc_unpack_skew": (None, [_dp, c_int, _dp]),
        "orc_pack_upper": (None, [_dp, c_int, _dp]),
        "orc_cnp": (None, [_dp, c_int, c_int, c_int, _dp]),
        "orc_cayley": (c_int, [_dp, c_int, c_int, _dp]),
        "orc_cnp_backward": (None, [_dp, c_int, c_int, c_int, _dp, _dp]),
        "orc_invert_perm": (c_int, [_ip, c_int, _ip]),
        "orc_perm_matrix": (None, [_ip, c_int, _dp]),
        "orc_blockdiag": (None, [_dp, c_int, c_int, _dp]),
        "orc_merge_w0": (None, [_dp, c_int, c_int, _ip, _ip, _dp]),
        "orc_forward": (None, [c_int, c_int, c_int, _dp, _dp, _dp, c_int, _dp, c_int,
                               _ip, _ip, _dp, ctypes.c_void_p]),
        "orc_forward_dense": (None, [c_int, c_int, c_int, _dp, _dp, _dp, _dp, _dp]),
        "orc_backward": (None, [c_int, c_int, c_int, _dp, _dp, _dp, _dp, c_int, _dp,
                                c_int, _ip, _ip, _dp, _dp, _dp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = _load(_build.build())
    return _LIB


def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def skew_count(b):
    """Packed parameters per block, b(b-1)/2 ([POET-X §2.D])."""
    return int(_lib().orc_skew_count(int(b)))


def unpack_skew(theta, b):
    """theta [nb, b(b-1)/2] -> K [nb, b, b], strict upper triangle row by row."""
    theta = _d(theta).reshape(-1, skew_count(b))
    K = np.empty((theta.shape[0], b, b))
    for j in range(theta.shape[0]):
        out = np.empty((b, b))
        _lib().orc_unpack_skew(_d(theta[j]), b, out)
        K[j] = out
    return K


def pack_upper(M):
    """M [nb, b, b] -> its strict upper triangles [nb, b(b-1)/2] in packing order."""
    M = _d(M)
    nb, b, _ = M.shape
    out = np.empty((nb, skew_count(b)))
    for j in range(nb):
        t = np.empty(skew_count(b))
        _lib().orc_pack_upper(_d(M[j]), b, t)
        out[j] = t
    return out


def cnp(theta, b, n):
    """[POET-X §2.D] Cayley-Neumann blocks Q = (I + K)(I + K + ... + K^n).

    theta [nb, b(b-1)/2] -> Q [nb, b, b]."""
    theta = _d(theta).reshape(-1, skew_count(b))
    nb = theta.shape[0]
    Q = np.empty((nb, b, b))
    _lib().orc_cnp(theta, nb, b, int(n), Q)
    return Q


def cayley(theta, b):
    """Exact Cayley map (I + K)(I - K)^{-1} per block (Gauss-Jordan in double)."""
    theta = _d(theta).reshape(-1, skew_count(b))
    nb = theta.shape[0]
    C = np.empty((nb, b, b))
    if _lib().orc_cayley(theta, nb, b, C) != 0:
        raise ArithmeticError("singular I - K")
    return C


def cnp_backward(theta, b, n, dQ):
    """Chain rule of ``cnp``: dL/dQ [nb,b,b] -> dL/dtheta [nb, b(b-1)/2]."""
    theta = _d(theta).reshape(-1, skew_count(b))
    nb = theta.shape[0]
    dQ = _d(dQ).reshape(nb, b, b)
    out = np.empty((nb, skew_count(b)))
    _lib().orc_cnp_backward(theta, nb, b, int(n), dQ, out)
    return out


def invert_perm(perm):
    """[POET-X §2.B] inverse index map, inv[perm[i]] = i; ValueError if not a permutation."""
    perm = _i(perm)
    inv = np.empty_like(perm)
    if _lib().orc_invert_perm(perm, perm.size, inv) != 0:
        raise ValueError("not a permutation")
    return inv


def perm_matrix(perm):
    """Dense permutation matrix with Pi[i, perm[i]] = 1, so Pi @ v = v[perm]."""
    perm = _i(perm)
    Pi = np.empty((perm.size, perm.size))
    _lib().orc_perm_matrix(perm, perm.size, Pi)
    return Pi


def blockdiag(Qs):
    """[POET-X §2.C] dense blockdiag(Q_0, ..., Q_{nb-1})."""
    Qs = _d(Qs)
    nb, b, _ = Qs.shape
    B = np.empty((nb * b, nb * b))
    _lib().orc_blockdiag(Qs, nb, b, B)
    return B


def merge_w0(W0, perm_out, perm_in):
    """[POET-X §2.B] W0m = Pi_R W0 Pi_P^T, i.e. W0m[i, k] = W0[perm_out[i], perm_in[k]]."""
    W0 = _d(W0)
    d_out, d_in = W0.shape
    out = np.empty_like(W0)
    _lib().orc_merge_w0(W0, d_out, d_in, _i(perm_out), _i(perm_in), out)
    return out


def fold_w0(W0, QP, QR, perm_in, perm_out):
    """[POET-X §2.B] the effective weight R W0 P, written out densely.

    P = Pi_P^T blockdiag(QP) Pi_P and R = Pi_R^T blockdiag(QR) Pi_R, each built
    from the dense permutation matrix and the dense block-diagonal above; two
    numpy matmuls in double.  This is what the weight becomes when an inner
    loop ends and the learned rotations are folded into it."""
    W0 = _d(W0)
    Pi_P, Pi_R = perm_matrix(perm_in), perm_matrix(perm_out)
    P = Pi_P.T @ blockdiag(QP) @ Pi_P
    R = Pi_R.T @ blockdiag(QR) @ Pi_R
    return R @ W0 @ P


def quantize_rows_int8(W):
    """[POET-X §2.E] POET-XQ: the frozen weight as INT8 codes, one symmetric
    scale per row (the page gives no granularity; this is the reading).

    s_i = max_k |W[i, k]| / 127 and q[i, k] = rint(W[i, k] / s_i), ties to even,
    clipped to [-127, 127]; a row of zeros has s_i = 0 and codes 0.  The codes
    are integers decided by floating point, so this takes the decisions in the
    precision the kernel takes them in: IEEE fp32 divisions.  Returns (q int8,
    s float32)."""
    W = np.asarray(W, dtype=np.float32)
    s = (np.abs(W).max(axis=1) / np.float32(127)).astype(np.float32)
    q = np.zeros(W.shape, dtype=np.int8)
    nz = s > 0
    q[nz] = np.clip(np.rint(W[nz] / s[nz, None]), -127, 127).astype(np.int8)
    return q, s


def dequantize_rows(q, s):
    """Inverse map of ``quantize_rows_int8``: W'[i, k] = q[i, k] * s_i, in double."""
    return np.asarray(q, dtype=np.float64) * np.asarray(s, dtype=np.float64)[:, None]


def forward(x, W0, QP, QR, perm_in, perm_out, return_z=False):
    """[POET-X §2.A-§2.C] y = Pi_R^T B_R Pi_R W0 Pi_P^T B_P Pi_P x, token by token.

    Uses the unmerged W0 and all four permutation applications.  x [T, d_in],
    W0 [d_out, d_in], QP [d_in/b_in, b_in, b_in], QR [d_out/b_out, b_out, b_out].
    With ``return_z`` also returns z = Pi_R W0 Pi_P^T B_P Pi_P x [T, d_out]."""
    x, W0, QP, QR = _d(x), _d(W0), _d(QP), _d(QR)
    T, d_in = x.shape
    d_out = W0.shape[0]
    y = np.empty((T, d_out))
    z = np.empty((T, d_out)) if return_z else None
    _lib().orc_forward(T, d_in, d_out, x, W0, QP, QP.shape[1], QR, QR.shape[1],
                       _i(perm_in), _i(perm_out), y,
                       z.ctypes.data_as(ctypes.c_void_p) if return_z else None)
    return (y, z) if return_z else y


def forward_dense(x, W0, P, R):
    """y_t = R W0 P x_t with dense P [d_in, d_in] and R [d_out, d_out]."""
    x, W0 = _d(x), _d(W0)
    T, d_in = x.shape
    d_out = W0.shape[0]
    y = np.empty((T, d_out))
    _lib().orc_forward_dense(T, d_in, d_out, x, W0, _d(P), _d(R), y)
    return y


def backward(x, dy, W0, QP, QR, perm_in, perm_out):
    """Backward of ``forward`` for an upstream gradient dy [T, d_out].

    Returns dX [T, d_in], dQP [d_in/b_in, b_in, b_in], dQR [d_out/b_out, ...]."""
    x, dy, W0, QP, QR = _d(x), _d(dy), _d(W0), _d(QP), _d(QR)
    T, d_in = x.shape
    d_out = W0.shape[0]
    dX = np.empty((T, d_in))
    dQP = np.empty_like(QP)
    dQR = np.empty_like(QR)
    _lib().orc_backward(T, d_in, d_out, x, dy, W0, QP, QP.shape[1], QR, QR.shape[1],
                        _i(perm_in), _i(perm_out), dX, dQP, dQR)
    return dX, dQP, dQR


def layer(x, W0, theta_P, theta_R, n, perm_in, perm_out, b_in, b_out, dy=None):
    """Whole transformed linear: CNP of both sides, forward, and (with dy) backward.

    Returns a dict with Q_P, Q_R, y and, with dy, dX, dQ_P, dQ_R, dtheta_P, dtheta_R."""
    QP = cnp(theta_P, b_in, n)
    QR = cnp(theta_R, b_out, n)
    out = {"Q_P": QP, "Q_R": QR, "y": forward(x, W0, QP, QR, perm_in, perm_out)}
    if dy is not None:
        dX, dQP, dQR = backward(x, dy, W0, QP, QR, perm_in, perm_out)
        out.update(dX=dX, dQ_P=dQP, dQ_R=dQR,
                   dtheta_P=cnp_backward(theta_P, b_in, n, dQP),
                   dtheta_R=cnp_backward(theta_R, b_out, n, dQR))
    return out


def orth_error(Q):
    """Per block ||Q^T Q - I||_F (numpy matmul in double)."""
    Q = _d(Q)
    eye = np.eye(Q.shape[-1])
    return np.sqrt(((np.swapaxes(Q, -1, -2) @ Q - eye) ** 2).sum(axis=(-1, -2)))


def rel_fro(got, ref):
    """Relative Frobenius error ||got - ref||_F / ||ref||_F (the parity metric).

    An all-zero reference gives the absolute error ||got||_F instead."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    return num / den if den > 0 else num


def rel_fro_rows(got, ref):
    """The same metric for every slice along the first axis (a token row of an
    activation, one block of Q, the packed parameters of one block):
    ||got[i] - ref[i]||_F / ||ref[i]||_F, or the absolute ||got[i]||_F where
    ref[i] is all zeros.  Returns a vector of length shape[0]."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    g = got.reshape(got.shape[0], -1)
    r = ref.reshape(ref.shape[0], -1)
    den = np.sqrt((r * r).sum(axis=1))
    num = np.sqrt(((g - r) ** 2).sum(axis=1))
    out = num.copy()
    nz = den > 0
    out[nz] = num[nz] / den[nz]
    return out
