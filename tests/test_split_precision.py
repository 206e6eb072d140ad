"""Precision of the split products behind fp32 Q on the tensor cores (CPU).

The library forms fp32 Q of b >= 32 on the tensor cores: every operand of the
Horner chain X_1 = K, X_{i+1} = X_i K + 2K, Q = I + X_{n+1} is held as two
16-bit parts, x = hi + lo (hi the rounded value, lo the rounded remainder),
and each product is taken as X_hi K_hi + X_hi K_lo + X_lo K_hi with fp32
accumulation.  This module emulates that arithmetic in numpy (the parts
rounded exactly as the kernels round them, the products summed in double and
rounded to fp32, which is what an fp32 accumulator can at best give) and
compares it with the oracle's exact Q.  It pins the choice of fp16 parts:
with bf16 parts (8 significant bits each, 16 for the pair) rows of Q drift
towards the fp32 bar of 1e-5 at the largest parameter scale the tests use;
with fp16 parts (11 each, 22 for the pair) they stay far below it.
"""
import numpy as np
import pytest
import torch

import oracle
from orthogonal_equivalence_neumann_b300 import inputs

BAR = 1e-5


def _round(x, dtype):
    return torch.from_numpy(np.asarray(x, np.float32)).to(dtype).to(torch.float64).numpy()


def _split(x, dtype):
    hi = _round(x, dtype)
    lo = _round(np.asarray(x, np.float32) - hi, dtype)
    return hi, lo


def _f32(x):
    return np.asarray(x, np.float32).astype(np.float64)


def split_chain_q(K, n, dtype):
    """Q from the three-term split chain, parts of type `dtype`."""
    Kh, Kl = _split(K, dtype)
    X = K
    for _ in range(n):
        Xh, Xl = _split(X, dtype)
        X = _f32(Xh @ Kh + Xh @ Kl + Xl @ Kh + 2.0 * (Kh + Kl))
    return _f32(np.eye(K.shape[0]) + X)


def worst_row(got, ref):
    return float((np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)).max())


@pytest.mark.parametrize("b", [128, 256])
def test_fp16_parts_keep_q_well_inside_the_fp32_bar(b):
    th = inputs.make_theta(2, b, 0.05, 1700 + b).double().numpy()
    K = oracle.unpack_skew(th, b)
    Q = oracle.cnp(th, b, 3)
    for j in range(2):
        err = worst_row(split_chain_q(K[j], 3, torch.float16), Q[j])
        assert err < BAR / 10, err


def test_bf16_parts_come_close_to_the_fp32_bar():
    # the reason the kernels split into fp16 parts: with bf16 parts the worst
    # row of a 256-block at sigma = 0.05 lies within a factor of three of 1e-5
    b = 256
    th = inputs.make_theta(2, b, 0.05, 1956).double().numpy()
    K = oracle.unpack_skew(th, b)
    Q = oracle.cnp(th, b, 3)
    err = max(worst_row(split_chain_q(K[j], 3, torch.bfloat16), Q[j]) for j in range(2))
    assert err > BAR / 3, err


def test_the_emulation_is_exact_without_splitting():
    # the harness itself: parts of float64 (no rounding) reproduce the oracle
    b = 64
    th = inputs.make_theta(1, b, 0.05, 1957).double().numpy()
    K = oracle.unpack_skew(th, b)[0]
    X = K
    for _ in range(3):
        X = X @ K + 2.0 * K
    assert np.abs(np.eye(b) + X - oracle.cnp(th, b, 3)[0]).max() < 1e-12
