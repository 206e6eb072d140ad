"""The oracle pins have teeth: plausible mistakes planted in a COPY of the
oracle source (on the CPU, in a temporary directory) each fail at least one
pin of ``test_oracle_pins.py``.  The oracle itself is never modified."""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import build as obuild
import test_oracle_pins as pins

# (name, exact text in poetx_oracle.c, replacement)
MUTANTS = [
    ("unpack: lower triangle not negated",
     "K[(size_t)k * b + i] = -theta[p];", "K[(size_t)k * b + i] = theta[p];"),
    ("cnp: Neumann sum stops one power early",
     "for (int i = 1; i <= n; ++i) {       /* Pw = K^i, S += Pw */",
     "for (int i = 1; i < n; ++i) {       /* Pw = K^i, S += Pw */"),
    ("cnp: (I + K) factor dropped",
     "for (size_t e = 0; e < bb; ++e) IpK[e] += K[e];\n  mat_mul(b, IpK, S, Q);",
     "mat_mul(b, IpK, S, Q);"),
    ("cnp backward: all coefficients 1",
     "const double cm = (m <= n) ? 2.0 : 1.0;", "const double cm = 1.0;"),
    ("cnp backward: powers not transposed",
     "mat_mul(b, pwT + (size_t)a * bb, G, T1);", "mat_mul(b, pw + (size_t)a * bb, G, T1);"),
    ("cnp backward: packed gradient misses the lower entry",
     "dtheta[p++] = dK[(size_t)i * b + k] - dK[(size_t)k * b + i];",
     "dtheta[p++] = dK[(size_t)i * b + k];"),
    ("forward: P-side scatter replaced by a second gather",
     "for (int i = 0; i < d_in; ++i) v3[perm_in[i]] = v2[i];        /* Pi_P^T . */",
     "for (int i = 0; i < d_in; ++i) v3[i] = v2[perm_in[i]];        /* Pi_P^T . */"),
    ("forward: R block applied transposed",
     "block_apply(QR, nbo, b_out, v5, v6);                          /* B_R . */",
     "block_apply_t(QR, nbo, b_out, v5, v6);                        /* B_R . */"),
    ("backward: B_R not transposed",
     "block_apply_t(QR, nbo, b_out, g6, g5);                        /* B_R^T . */",
     "block_apply(QR, nbo, b_out, g6, g5);                          /* B_R^T . */"),
    ("backward: dQ operands swapped",
     "dq_token_sum(T, d_in, b_in, nbi, G2, V1, dQP);",
     "dq_token_sum(T, d_in, b_in, nbi, V1, G2, dQP);"),
    ("merge: input permutation applied to rows",
     "W0m[(size_t)i * d_in + k] = W0[(size_t)perm_out[i] * d_in + perm_in[k]];",
     "W0m[(size_t)i * d_in + k] = W0[(size_t)i * d_in + perm_in[k]];"),
    ("cayley: pivot row swap forgets the right-hand side",
     "        Inv[(size_t)piv * b + k] = t;\n", "\n"),
    ("perm matrix transposed",
     "Pi[(size_t)i * d + perm[i]] = 1.0;", "Pi[(size_t)perm[i] * d + i] = 1.0;"),
]

PIN_CALLS = [
    ("unpack golden", lambda: pins.test_unpack_matches_golden_layout()),
    ("unpack skew", lambda: pins.test_unpack_is_skew_and_round_trips(5)),
    ("b2 closed form", lambda: pins.test_cnp_b2_complex_closed_form(3)),
    ("b3 golden", lambda: pins.test_cnp_b3_golden_hand_derived()),
    ("Q = C (I - K^{n+1})", lambda: pins.test_cnp_equals_cayley_times_truncation_residual(16, 2, 0.05)),
    ("orth defect", lambda: pins.test_cnp_orthogonality_defect_closed_form(3)),
    ("cayley lapack", lambda: pins.test_cayley_matches_lapack_and_is_orthogonal()),
    ("cnp bwd FD", lambda: pins.test_cnp_backward_matches_finite_differences(4, 3)),
    ("perm golden", lambda: pins.test_perm_golden()),
    ("merge", lambda: pins.test_merge_w0_matches_dense_permutation_products()),
    ("fwd materialised", lambda: pins.test_forward_input_centric_equals_materialised((8, 12, 4, 6, 3))),
    ("fwd merged", lambda: pins.test_forward_merged_weight_takes_two_permutations()),
    ("dX transpose", lambda: pins.test_backward_dx_is_transpose_product((8, 12, 4, 6, 3))),
    ("dQ FD", lambda: pins.test_backward_dq_blocks_match_finite_differences()),
]


@pytest.fixture(scope="module")
def tmpdir_mod():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught_by_a_pin(name, old, new, tmpdir_mod):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, "mutation anchor not found: " + name
    path = os.path.join(tmpdir_mod, "mut_%d.c" % abs(hash(name)))
    lib = path[:-2] + ".so"
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", *obuild.CFLAGS[:-1], path, "-o", lib, obuild.CFLAGS[-1]], check=True)
    saved = oracle._LIB
    oracle._LIB = oracle._load(lib)
    caught = []
    try:
        for pin_name, call in PIN_CALLS:
            try:
                with np.errstate(all="ignore"):
                    call()
            except (AssertionError, ValueError, ArithmeticError):
                caught.append(pin_name)
    finally:
        oracle._LIB = saved
    assert caught, "no pin caught the planted mistake: " + name


# ---- the oracle's numpy-level functions (the fold, the INT8 quantiser): the
# mutated function is a copy of the oracle's own source with one change,
# compiled into a namespace of its own and swapped in for the pins' calls.
PY_MUTANTS = [
    ("fold: P-side permutation transposed", "fold_w0",
     "P = Pi_P.T @ blockdiag(QP) @ Pi_P", "P = Pi_P @ blockdiag(QP) @ Pi_P.T"),
    ("fold: R blocks transposed", "fold_w0",
     "R = Pi_R.T @ blockdiag(QR) @ Pi_R", "R = Pi_R.T @ blockdiag(QR).T @ Pi_R"),
    ("fold: R applied as its transpose", "fold_w0", "return R @ W0 @ P", "return R.T @ W0 @ P"),
    ("quantiser: truncation instead of rounding", "quantize_rows_int8",
     "np.rint(W[nz] / s[nz, None])", "np.trunc(W[nz] / s[nz, None])"),
    ("quantiser: ties away from zero", "quantize_rows_int8",
     "np.rint(W[nz] / s[nz, None])", "np.sign(W[nz]) * np.floor(np.abs(W[nz] / s[nz, None]) + 0.5)"),
    ("quantiser: scale over 128", "quantize_rows_int8", "np.float32(127)", "np.float32(128)"),
    ("parity metric: divided by the result's norm", "rel_fro",
     "den = np.linalg.norm(ref.ravel())", "den = np.linalg.norm(got.ravel())"),
    ("parity metric: squared ratio", "rel_fro",
     "return num / den if den > 0 else num", "return (num / den) ** 2 if den > 0 else num"),
    ("parity metric: largest entry instead of the norm", "rel_fro",
     "num = np.linalg.norm((got - ref).ravel())", "num = np.abs(got - ref).max()"),
    ("per-row metric: rows against the whole tensor's norm", "rel_fro_rows",
     "den = np.sqrt((r * r).sum(axis=1))", "den = np.full(r.shape[0], np.sqrt((r * r).sum()))"),
    ("per-row metric: largest entry of a row", "rel_fro_rows",
     "num = np.sqrt(((g - r) ** 2).sum(axis=1))", "num = np.sqrt(((g - r) ** 2).max(axis=1))"),
    ("orthogonality defect: Q Q without the transpose", "orth_error",
     "np.swapaxes(Q, -1, -2) @ Q", "Q @ Q"),
    ("orthogonality defect: identity not subtracted", "orth_error", " - eye) ** 2", ") ** 2"),
    ("orthogonality defect: no square root", "orth_error", "return np.sqrt(", "return ("),
    ("orthogonality defect: summed over all blocks", "orth_error",
     ".sum(axis=(-1, -2))", ".sum()"),
]

PY_PIN_CALLS = [
    ("fold = effective weight", lambda: pins.test_fold_w0_is_the_effective_weight((8, 12, 4, 6, 3))),
    ("fold keeps the function", lambda: pins.test_fold_then_fresh_permutations_and_zero_theta_keep_the_function()),
    ("quantiser golden", lambda: pins.test_quantize_rows_int8_golden()),
    ("quantiser bounds", lambda: pins.test_quantize_rows_int8_bounds_and_round_trip_error()),
    ("parity metric hand values", lambda: pins.test_rel_fro_hand_values()),
    ("per-row metric hand values", lambda: pins.test_rel_fro_rows_hand_values()),
    ("orthogonality defect hand values", lambda: pins.test_orth_error_hand_values()),
    ("orthogonality defect closed form",
     lambda: pins.test_orth_error_closed_form_of_the_neumann_truncation(3)),
]


@pytest.mark.parametrize("name,fn,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_python_mutant_is_caught_by_a_pin(name, fn, old, new, monkeypatch):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn)))
    assert src.count(old) == 1, "mutation anchor not found: " + name
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant %s>" % name, "exec"), ns)
    monkeypatch.setattr(oracle, fn, ns[fn])
    caught = []
    for pin_name, call in PY_PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                call()
        except (AssertionError, ValueError, ArithmeticError):
            caught.append(pin_name)
    assert caught, "no pin caught the planted mistake: " + name
