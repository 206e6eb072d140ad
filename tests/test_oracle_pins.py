"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks one oracle function against a hand-derived golden value, a
closed form, a library routine (numpy / scipy), a brute-force construction or
finite differences, chosen so that a dropped term, a wrong sign, a wrong power,
a transposed operand or a wrong index in the oracle fails at least one of them.

Source of the method: "POET-X: Memory-efficient LLM Training by Scaling
Orthogonal Transformation" (gist.science summary), section 2.A-2.E; the
spectrum-preservation property of two-sided orthogonal transforms is also
stated on the page "Pion: 保持谱稳定的大语言模型训练优化器" (section 数学原理).
"""
import numpy as np
import pytest
import scipy.linalg

import oracle
from conftest import as_f64, read_golden

RNG = np.random.default_rng(20260305)


def rand_theta(nb, b, sigma, rng=RNG):
    return rng.standard_normal((nb, b * (b - 1) // 2)) * sigma


def np_perm_matrix(perm):
    # brute force: row i of the identity's rows reordered, M[i, perm[i]] = 1
    return np.eye(len(perm))[np.asarray(perm)]


# ---------------------------------------------------------------- packing (§2.D)

def test_skew_count_halves_parameters():
    for b in range(2, 40):
        assert oracle.skew_count(b) == b * (b - 1) // 2


def test_unpack_matches_golden_layout():
    g = read_golden("skew_pack_b4.txt")
    K = oracle.unpack_skew(as_f64(g["theta"])[None], 4)[0]
    np.testing.assert_array_equal(K, as_f64(g["K"]))


@pytest.mark.parametrize("b", [2, 3, 5, 16, 33])
def test_unpack_is_skew_and_round_trips(b):
    th = rand_theta(3, b, 1.0)
    K = oracle.unpack_skew(th, b)
    np.testing.assert_array_equal(K, -np.swapaxes(K, 1, 2))
    np.testing.assert_array_equal(oracle.pack_upper(K), th)
    # every parameter appears exactly once above the diagonal (numpy triu order)
    iu = np.triu_indices(b, 1)
    np.testing.assert_array_equal(K[:, iu[0], iu[1]], th)


# ---------------------------------------------------------------- CNP (§2.D)

@pytest.mark.parametrize("b,n", [(2, 1), (4, 3), (32, 6), (7, 2)])
def test_cnp_zero_params_give_identity(b, n):
    Q = oracle.cnp(np.zeros((2, b * (b - 1) // 2)), b, n)
    np.testing.assert_array_equal(Q, np.broadcast_to(np.eye(b), Q.shape))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_cnp_b2_complex_closed_form(n):
    # For b = 2, K = t J with J^2 = -I, so a I + c J behaves as a + c i.
    # Q = (1 + it) sum_{k=0}^n (it)^k  ->  [[Re, Im], [-Im, Re]].
    for t in (0.3, -0.05, 1e-3):
        z = (1 + 1j * t) * sum((1j * t) ** k for k in range(n + 1))
        want = np.array([[z.real, z.imag], [-z.imag, z.real]])
        got = oracle.cnp(np.array([[t]]), 2, n)[0]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_cnp_b3_golden_hand_derived():
    g = read_golden("cnp_b3.txt")
    th = as_f64(g["theta"])[None]
    np.testing.assert_allclose(oracle.cnp(th, 3, 1)[0], as_f64(g["Q_n1"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.cnp(th, 3, 2)[0], as_f64(g["Q_n2"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.cayley(th, 3)[0], as_f64(g["C"]), rtol=0, atol=1e-15)


@pytest.mark.parametrize("b,n,sigma", [(8, 1, 0.1), (16, 2, 0.05), (32, 3, 0.01),
                                       (32, 4, 0.03), (64, 6, 0.01), (17, 5, 0.08)])
def test_cnp_equals_cayley_times_truncation_residual(b, n, sigma):
    # (I - K) sum_{i<=n} K^i = I - K^{n+1}, and all factors commute, so
    # Q = C (I - K^{n+1}) with C = (I - K)^{-1}(I + K) the exact Cayley map.
    # C from LAPACK (numpy.linalg.solve), powers from numpy.matrix_power.
    th = rand_theta(3, b, sigma)
    Q = oracle.cnp(th, b, n)
    K = oracle.unpack_skew(th, b)
    I = np.eye(b)
    for j in range(3):
        C = np.linalg.solve(I - K[j], I + K[j])
        Kn1 = np.linalg.matrix_power(K[j], n + 1)
        np.testing.assert_allclose(Q[j], C @ (I - Kn1), rtol=0, atol=1e-13)
        # so ||Q - C||_F = ||K^{n+1}||_F exactly (C is orthogonal)
        np.testing.assert_allclose(np.linalg.norm(Q[j] - C), np.linalg.norm(Kn1), rtol=1e-9)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_cnp_orthogonality_defect_closed_form(n):
    # Q^T Q - I = -K^{2n+2} (n even),  -2K^{n+1} + K^{2n+2} (n odd).
    b = 12
    th = rand_theta(2, b, 0.2)
    Q = oracle.cnp(th, b, n)
    K = oracle.unpack_skew(th, b)
    for j in range(2):
        Kn1 = np.linalg.matrix_power(K[j], n + 1)
        K2n2 = np.linalg.matrix_power(K[j], 2 * n + 2)
        want = -K2n2 if n % 2 == 0 else -2 * Kn1 + K2n2
        np.testing.assert_allclose(Q[j].T @ Q[j] - np.eye(b), want, rtol=0, atol=1e-14)


def test_cayley_matches_lapack_and_is_orthogonal():
    for b in (2, 5, 32, 64):
        th = rand_theta(2, b, 0.3)
        C = oracle.cayley(th, b)
        K = oracle.unpack_skew(th, b)
        for j in range(2):
            ref = np.linalg.solve(np.eye(b) - K[j], np.eye(b) + K[j])
            np.testing.assert_allclose(C[j], ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(C[j].T @ C[j], np.eye(b), rtol=0, atol=1e-12)


def test_neumann_error_shrinks_with_n():
    b = 32
    th = rand_theta(4, b, 0.01)
    C = oracle.cayley(th, b)
    errs = [np.linalg.norm(oracle.cnp(th, b, n) - C) for n in range(1, 7)]
    assert all(e2 < e1 for e1, e2 in zip(errs, errs[1:])), errs
    orth = [oracle.orth_error(oracle.cnp(th, b, n)).max() for n in range(1, 7)]
    assert orth[-1] < 1e-9 < orth[0]


@pytest.mark.parametrize("b,n", [(3, 1), (4, 3), (6, 4), (5, 6)])
def test_cnp_backward_matches_finite_differences(b, n):
    th = rand_theta(2, b, 0.2)
    G = RNG.standard_normal((2, b, b))
    for sym in (False, True):
        Gs = G + np.swapaxes(G, 1, 2) if sym else G   # a symmetric dQ too
        dth = oracle.cnp_backward(th, b, n, Gs)
        h = 1e-6
        fd = np.zeros_like(th)
        for j in range(2):
            for p in range(th.shape[1]):
                tp, tm = th.copy(), th.copy()
                tp[j, p] += h
                tm[j, p] -= h
                fd[j, p] = (np.sum(Gs[j] * oracle.cnp(tp[j:j + 1], b, n)[0]) -
                            np.sum(Gs[j] * oracle.cnp(tm[j:j + 1], b, n)[0])) / (2 * h)
        np.testing.assert_allclose(dth, fd, rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------- permutations (§2.B)

def test_perm_golden():
    g = read_golden("perm_d3.txt")
    perm = np.array([int(v) for v in g["perm"]], dtype=np.int32)
    v = as_f64(g["v"])
    np.testing.assert_array_equal(oracle.invert_perm(perm), [int(v) for v in g["inv"]])
    Pi = oracle.perm_matrix(perm)
    np.testing.assert_array_equal(Pi @ v, as_f64(g["Pi_v"]))
    np.testing.assert_array_equal(Pi.T @ v, as_f64(g["PiT_v"]))


def test_perm_then_inverse_is_identity_and_matches_dense():
    for d in (1, 7, 256, 2048):
        perm = RNG.permutation(d).astype(np.int32)
        inv = oracle.invert_perm(perm)
        np.testing.assert_array_equal(perm[inv], np.arange(d))
        np.testing.assert_array_equal(inv[perm], np.arange(d))
        if d <= 256:
            np.testing.assert_array_equal(oracle.perm_matrix(perm), np_perm_matrix(perm))


def test_invert_perm_rejects_non_permutations():
    for bad in ([0, 0, 1], [0, 3, 1], [-1, 0, 1]):
        with pytest.raises(ValueError):
            oracle.invert_perm(np.array(bad, dtype=np.int32))


def test_blockdiag_matches_scipy():
    Qs = RNG.standard_normal((3, 4, 4))
    np.testing.assert_array_equal(oracle.blockdiag(Qs), scipy.linalg.block_diag(*Qs))


def test_merge_w0_matches_dense_permutation_products():
    d_out, d_in = 12, 8
    W0 = RNG.standard_normal((d_out, d_in))
    po, pi = RNG.permutation(d_out), RNG.permutation(d_in)
    want = np_perm_matrix(po) @ W0 @ np_perm_matrix(pi).T
    np.testing.assert_allclose(oracle.merge_w0(W0, po, pi), want, rtol=0, atol=0)


# ---------------------------------------------------------------- the layer (§2.A-§2.C)

def _layer_case(d_in, d_out, b_in, b_out, T, sigma=0.1, n=3, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d_in))
    W0 = rng.standard_normal((d_out, d_in)) / np.sqrt(d_in)
    thP = rand_theta(d_in // b_in, b_in, sigma, rng)
    thR = rand_theta(d_out // b_out, b_out, sigma, rng)
    pi = rng.permutation(d_in).astype(np.int32)
    po = rng.permutation(d_out).astype(np.int32)
    dy = rng.standard_normal((T, d_out))
    return x, W0, thP, thR, pi, po, dy, n


def _np_dense_PR(QP, QR, pi, po):
    P = np_perm_matrix(pi).T @ scipy.linalg.block_diag(*QP) @ np_perm_matrix(pi)
    R = np_perm_matrix(po).T @ scipy.linalg.block_diag(*QR) @ np_perm_matrix(po)
    return P, R


@pytest.mark.parametrize("shape", [(16, 16, 4, 4, 5), (8, 12, 4, 6, 3), (32, 16, 8, 4, 7)])
def test_forward_input_centric_equals_materialised(shape):
    d_in, d_out, b_in, b_out, T = shape
    x, W0, thP, thR, pi, po, dy, n = _layer_case(d_in, d_out, b_in, b_out, T)
    QP, QR = oracle.cnp(thP, b_in, n), oracle.cnp(thR, b_out, n)
    y = oracle.forward(x, W0, QP, QR, pi, po)
    P, R = _np_dense_PR(QP, QR, pi, po)
    W = R @ W0 @ P                                  # materialised R W0 P
    np.testing.assert_allclose(y, x @ W.T, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.forward_dense(x, W0, P, R), y, rtol=0, atol=1e-12)


def test_forward_merged_weight_takes_two_permutations():
    # y = Pi_R^T B_R (Pi_R W0 Pi_P^T) B_P Pi_P x: merged W0, one gather, one scatter.
    d_in, d_out, b_in, b_out, T = 16, 24, 4, 8, 6
    x, W0, thP, thR, pi, po, dy, n = _layer_case(d_in, d_out, b_in, b_out, T)
    QP, QR = oracle.cnp(thP, b_in, n), oracle.cnp(thR, b_out, n)
    W0m = oracle.merge_w0(W0, po, pi)
    u = x[:, pi] @ scipy.linalg.block_diag(*QP).T          # gather, then B_P
    z = u @ W0m.T
    v = z @ scipy.linalg.block_diag(*QR).T
    y = np.empty_like(v)
    y[:, po] = v                                           # scatter
    y_ref, z_ref = oracle.forward(x, W0, QP, QR, pi, po, return_z=True)
    np.testing.assert_allclose(y, y_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(z, z_ref, rtol=0, atol=1e-12)


def test_spectrum_preserved_with_exact_cayley_blocks():
    d_in, d_out = 64, 48
    x, W0, thP, thR, pi, po, dy, n = _layer_case(d_in, d_out, 16, 8, 1, sigma=0.5)
    CP, CR = oracle.cayley(thP, 16), oracle.cayley(thR, 8)
    P, R = _np_dense_PR(CP, CR, pi, po)
    s0 = np.linalg.svd(W0, compute_uv=False)
    s1 = np.linalg.svd(R @ W0 @ P, compute_uv=False)
    np.testing.assert_allclose(s1, s0, rtol=1e-12, atol=1e-12)
    # the truncated series is only approximately orthogonal: spectrum moves
    QP, QR = oracle.cnp(thP, 16, 1), oracle.cnp(thR, 8, 1)
    P1, R1 = _np_dense_PR(QP, QR, pi, po)
    assert np.abs(np.linalg.svd(R1 @ W0 @ P1, compute_uv=False) - s0).max() > 1e-3


# ---------------------------------------------------------------- end of an inner loop (§2.B)

@pytest.mark.parametrize("shape", [(16, 16, 4, 4, 5), (8, 12, 4, 6, 3), (32, 16, 8, 4, 7)])
def test_fold_w0_is_the_effective_weight(shape):
    d_in, d_out, b_in, b_out, T = shape
    x, W0, thP, thR, pi, po, dy, n = _layer_case(d_in, d_out, b_in, b_out, T)
    QP, QR = oracle.cnp(thP, b_in, n), oracle.cnp(thR, b_out, n)
    W = oracle.fold_w0(W0, QP, QR, pi, po)
    # the C oracle's token-by-token forward, with the unmerged W0
    np.testing.assert_allclose(x @ W.T, oracle.forward(x, W0, QP, QR, pi, po), rtol=0, atol=1e-12)
    # brute-force dense construction (numpy permutation rows, scipy block_diag)
    P, R = _np_dense_PR(QP, QR, pi, po)
    np.testing.assert_allclose(W, R @ W0 @ P, rtol=0, atol=1e-13)


def test_fold_w0_with_identity_blocks_is_w0():
    x, W0, thP, thR, pi, po, dy, n = _layer_case(24, 16, 8, 4, 1)
    IP = np.broadcast_to(np.eye(8), (3, 8, 8))
    IR = np.broadcast_to(np.eye(4), (4, 4, 4))
    np.testing.assert_array_equal(oracle.fold_w0(W0, IP, IR, pi, po), W0)


def test_fold_then_fresh_permutations_and_zero_theta_keep_the_function():
    # an inner loop ends: W0 <- R W0 P, theta <- 0 (Q = I), new permutations
    d_in, d_out, b_in, b_out, T = 32, 16, 8, 4, 6
    x, W0, thP, thR, pi, po, dy, n = _layer_case(d_in, d_out, b_in, b_out, T)
    QP, QR = oracle.cnp(thP, b_in, n), oracle.cnp(thR, b_out, n)
    y0 = oracle.forward(x, W0, QP, QR, pi, po)
    W1 = oracle.fold_w0(W0, QP, QR, pi, po)
    rng = np.random.default_rng(7)
    pi1 = rng.permutation(d_in).astype(np.int32)
    po1 = rng.permutation(d_out).astype(np.int32)
    QP1 = oracle.cnp(np.zeros_like(thP), b_in, n)
    QR1 = oracle.cnp(np.zeros_like(thR), b_out, n)
    np.testing.assert_allclose(oracle.forward(x, W1, QP1, QR1, pi1, po1), y0, rtol=0, atol=1e-12)
    # and the fold keeps the spectrum when the blocks are exactly orthogonal
    CP, CR = oracle.cayley(thP, b_in), oracle.cayley(thR, b_out)
    np.testing.assert_allclose(np.linalg.svd(oracle.fold_w0(W0, CP, CR, pi, po), compute_uv=False),
                               np.linalg.svd(W0, compute_uv=False), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", [(16, 16, 4, 4, 5), (8, 12, 4, 6, 3)])
def test_backward_dx_is_transpose_product(shape):
    d_in, d_out, b_in, b_out, T = shape
    x, W0, thP, thR, pi, po, dy, n = _layer_case(d_in, d_out, b_in, b_out, T)
    QP, QR = oracle.cnp(thP, b_in, n), oracle.cnp(thR, b_out, n)
    dX, dQP, dQR = oracle.backward(x, dy, W0, QP, QR, pi, po)
    P, R = _np_dense_PR(QP, QR, pi, po)
    np.testing.assert_allclose(dX, dy @ (R @ W0 @ P), rtol=0, atol=1e-12)


def test_backward_dq_blocks_match_finite_differences():
    d_in, d_out, b_in, b_out, T = 8, 12, 4, 6, 3
    x, W0, thP, thR, pi, po, dy, n = _layer_case(d_in, d_out, b_in, b_out, T)
    QP, QR = oracle.cnp(thP, b_in, n), oracle.cnp(thR, b_out, n)
    _, dQP, dQR = oracle.backward(x, dy, W0, QP, QR, pi, po)

    def loss(QP_, QR_):
        return np.sum(dy * oracle.forward(x, W0, QP_, QR_, pi, po))

    h = 1e-6
    for which, Qs, dQ in (("P", QP, dQP), ("R", QR, dQR)):
        fd = np.zeros_like(Qs)
        for idx in np.ndindex(*Qs.shape):
            Qp, Qm = Qs.copy(), Qs.copy()
            Qp[idx] += h
            Qm[idx] -= h
            if which == "P":
                fd[idx] = (loss(Qp, QR) - loss(Qm, QR)) / (2 * h)
            else:
                fd[idx] = (loss(QP, Qp) - loss(QP, Qm)) / (2 * h)
        np.testing.assert_allclose(dQ, fd, rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("shape", [(8, 12, 4, 4, 3, 3), (16, 8, 8, 4, 4, 2), (8, 8, 2, 4, 2, 5)])
def test_layer_dtheta_matches_finite_differences(shape):
    d_in, d_out, b_in, b_out, T, n = shape
    x, W0, thP, thR, pi, po, dy, _ = _layer_case(d_in, d_out, b_in, b_out, T, sigma=0.2)
    out = oracle.layer(x, W0, thP, thR, n, pi, po, b_in, b_out, dy=dy)

    def loss(tP, tR):
        return np.sum(dy * oracle.layer(x, W0, tP, tR, n, pi, po, b_in, b_out)["y"])

    h = 1e-6
    for which, th, got in (("P", thP, out["dtheta_P"]), ("R", thR, out["dtheta_R"])):
        fd = np.zeros_like(th)
        for idx in np.ndindex(*th.shape):
            tp, tm = th.copy(), th.copy()
            tp[idx] += h
            tm[idx] -= h
            if which == "P":
                fd[idx] = (loss(tp, thR) - loss(tm, thR)) / (2 * h)
            else:
                fd[idx] = (loss(thP, tp) - loss(thP, tm)) / (2 * h)
        np.testing.assert_allclose(got, fd, rtol=1e-6, atol=1e-8)


def test_oracle_results_do_not_depend_on_thread_count():
    import os
    import subprocess
    import sys
    code = ("import numpy as np, oracle;"
            "r=np.random.default_rng(1);x=r.standard_normal((9,16));W=r.standard_normal((16,16));"
            "tp=r.standard_normal((4,6))*.1;tr=r.standard_normal((4,6))*.1;"
            "pi=r.permutation(16).astype(np.int32);po=r.permutation(16).astype(np.int32);"
            "dy=r.standard_normal((9,16));o=oracle.layer(x,W,tp,tr,3,pi,po,4,4,dy=dy);"
            "import sys;sys.stdout.buffer.write(np.concatenate([o['y'].ravel(),o['dX'].ravel(),"
            "o['dtheta_P'].ravel(),o['dtheta_R'].ravel()]).tobytes())")
    outs = []
    for nt in ("1", "3"):
        env = dict(os.environ, OMP_NUM_THREADS=nt)
        outs.append(subprocess.run([sys.executable, "-c", code], env=env, check=True,
                                   capture_output=True,
                                   cwd=os.path.dirname(os.path.dirname(__file__))).stdout)
    assert outs[0] == outs[1] and len(outs[0]) > 0


# ---------------------------------------------------------------- POET-XQ (§2.E)

def test_quantize_rows_int8_golden():
    g = read_golden("xq_rows.txt")
    q, s = oracle.quantize_rows_int8(as_f64(g["W"]))
    np.testing.assert_array_equal(s, as_f64(g["scale"]).astype(np.float32))
    np.testing.assert_array_equal(q, as_f64(g["codes"]).astype(np.int8))


def test_quantize_rows_int8_bounds_and_round_trip_error():
    rng = np.random.default_rng(11)
    W = (rng.standard_normal((37, 64)) * rng.uniform(0.01, 3.0, (37, 1))).astype(np.float32)
    q, s = oracle.quantize_rows_int8(W)
    assert q.dtype == np.int8 and s.dtype == np.float32
    # every row uses the full code range at its maximum, and nothing beyond it
    np.testing.assert_array_equal(np.abs(q.astype(np.int32)).max(axis=1), 127)
    # nearest code: |W - q s| <= s / 2 (plus the fp32 rounding of the division)
    err = np.abs(W.astype(np.float64) - oracle.dequantize_rows(q, s))
    assert np.all(err <= s.astype(np.float64)[:, None] * (0.5 + 1e-6))


def test_quantize_commutes_with_the_merge():
    # quantising the merged weight = merging the quantised weight (codes and scales)
    rng = np.random.default_rng(12)
    W = rng.standard_normal((24, 16)).astype(np.float32)
    po = rng.permutation(24).astype(np.int32)
    pi = rng.permutation(16).astype(np.int32)
    qm, sm = oracle.quantize_rows_int8(oracle.merge_w0(W, po, pi))
    q, s = oracle.quantize_rows_int8(W)
    np.testing.assert_array_equal(qm, q[po][:, pi])
    np.testing.assert_array_equal(sm, s[po])


# ---------------------------------------------------------------- parity metrics
# Every GPU parity verdict is taken with these functions, so they are pinned to
# values worked out by hand (not by retyping their formulas).

def test_rel_fro_hand_values():
    # ||(0, 2, 2)|| / ||(1, 0, 0)|| = sqrt(8)
    assert oracle.rel_fro([1.0, 2.0, 2.0], [1.0, 0.0, 0.0]) == pytest.approx(np.sqrt(8.0), rel=1e-15)
    # ||(0, 5)|| / ||(3, 4)|| = 1; dividing by ||got|| = sqrt(90) would give 0.527
    assert oracle.rel_fro([3.0, 9.0], [3.0, 4.0]) == pytest.approx(1.0, rel=1e-15)
    # matrices are measured as one vector: ||[[0, 1], [0, 0]]|| / ||[[2, 0], [0, 0]]|| = 1/2
    assert oracle.rel_fro([[2.0, 1.0], [0.0, 0.0]], [[2.0, 0.0], [0.0, 0.0]]) == pytest.approx(0.5)
    # equal arguments: exactly zero; an all-zero reference: the absolute error ||(3, 4)|| = 5
    assert oracle.rel_fro([1.5, -2.0], [1.5, -2.0]) == 0.0
    assert oracle.rel_fro([3.0, 4.0], [0.0, 0.0]) == pytest.approx(5.0, rel=1e-15)
    # the error is not symmetric in its arguments: ||(2)|| / ||(1)|| = 2 but ||(2)|| / ||(3)|| = 2/3
    assert oracle.rel_fro([3.0], [1.0]) == pytest.approx(2.0)
    assert oracle.rel_fro([1.0], [3.0]) == pytest.approx(2.0 / 3.0)


def test_rel_fro_rows_hand_values():
    got = np.array([[1.0, 2.0, 2.0], [3.0, 9.0, 0.0], [0.0, 0.0, 0.0], [3.0, 4.0, 0.0]])
    ref = np.array([[1.0, 0.0, 0.0], [3.0, 4.0, 0.0], [0.0, 0.0, 0.0], [0.0, 0.0, 0.0]])
    np.testing.assert_allclose(oracle.rel_fro_rows(got, ref), [np.sqrt(8.0), 1.0, 0.0, 5.0],
                               rtol=1e-15)
    # one slice per block of a [nb, b, b] stack
    Qg = np.stack([np.eye(2), [[2.0, 1.0], [0.0, 0.0]]])
    Qr = np.stack([np.eye(2), [[2.0, 0.0], [0.0, 0.0]]])
    np.testing.assert_allclose(oracle.rel_fro_rows(Qg, Qr), [0.0, 0.5], rtol=1e-15)


def test_orth_error_hand_values():
    # A = diag(2, 1): A^T A - I = diag(3, 0) -> 3.
    # A = [[1, 1], [0, 1]]: A^T A - I = [[0, 1], [1, 1]] -> sqrt(3); A A - I = [[0, 2], [0, 0]]
    # would give 2 instead.  One value per block.
    A = np.stack([np.diag([2.0, 1.0]), [[1.0, 1.0], [0.0, 1.0]]])
    np.testing.assert_allclose(oracle.orth_error(A), [3.0, np.sqrt(3.0)], rtol=1e-15)
    # an orthogonal matrix (a rotation) has no defect; a zero matrix has ||I||_F = sqrt(b)
    c, s = np.cos(0.3), np.sin(0.3)
    assert oracle.orth_error(np.array([[c, -s], [s, c]])) == pytest.approx(0.0, abs=1e-15)
    assert oracle.orth_error(np.zeros((5, 5))) == pytest.approx(np.sqrt(5.0), rel=1e-15)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_orth_error_closed_form_of_the_neumann_truncation(n):
    # ||Q^T Q - I||_F = ||K^{2n+2}||_F (n even), ||-2K^{n+1} + K^{2n+2}||_F (n odd),
    # with the powers from numpy.linalg.matrix_power.  (Q Q^T gives the same norm for
    # any square Q -- same trace and same Frobenius norm of the Gram matrix -- so the
    # order of the product is pinned by the hand values above, not here.)
    b = 10
    th = rand_theta(3, b, 0.25)
    K = oracle.unpack_skew(th, b)
    want = []
    for j in range(3):
        Kn1 = np.linalg.matrix_power(K[j], n + 1)
        K2n2 = np.linalg.matrix_power(K[j], 2 * n + 2)
        want.append(np.linalg.norm(K2n2 if n % 2 == 0 else -2 * Kn1 + K2n2))
    np.testing.assert_allclose(oracle.orth_error(oracle.cnp(th, b, n)), want, rtol=1e-10)
