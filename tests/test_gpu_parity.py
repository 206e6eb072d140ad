"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bars (relative Frobenius error ||gpu - oracle||_F / ||oracle||_F per output,
and the same bar on each token row / block of it): fp32 paths <= 1e-5;
bf16-input / fp32-accumulate paths <= 2e-2; permutation indices and the merged
weight bit-exact.  The oracle reads exactly the values
the GPU reads (bf16 inputs widened exactly to double) and rounds nothing.
"""
import numpy as np
import pytest
import torch

import oracle
from orthogonal_equivalence_neumann_b300 import TransformedLinear, _lib, inputs

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_BF16 = 2e-2


def to64(t):
    return t.detach().to("cpu", torch.float32).double().numpy()


def tol_for(dtype):
    return TOL_F32 if dtype in ("f32", torch.float32) else TOL_BF16


def assert_close(name, got, ref, tol):
    """The bar on the whole tensor, and the same bar on every slice along the
    first axis (a token row of y or dX, one block of Q, the packed parameters
    of one block), so that a few wrong rows or one wrong tile cannot hide in
    the norm of a large tensor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, "%s: shape %s != %s" % (name, got.shape, ref.shape)
    err = oracle.rel_fro(got, ref)
    assert err <= tol, "%s: relative Frobenius error %.3e > %.1e" % (name, err, tol)
    if ref.ndim >= 2 and ref.shape[0] > 1:
        per = oracle.rel_fro_rows(got, ref)
        worst = int(np.argmax(per))
        assert per[worst] <= tol, "%s: slice %d of %d has relative error %.3e > %.1e" % (
            name, worst, ref.shape[0], per[worst], tol)
    return err


def gpu_layer(case, inp, save_z=True, T=None):
    x = inp["x"].cuda()
    dy = inp["dy"].cuda()
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n,
                            T_max=max(1, x.shape[0]), save_z=save_z)
    y, dX, dtp, dtr = lay.step(x, dy)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    return dict(y=to64(y), dX=to64(dX), dtheta_P=dtp.double().cpu().numpy(),
                dtheta_R=dtr.double().cpu().numpy(), Q_P=to64(lay.Q_P), Q_R=to64(lay.Q_R))


def oracle_inputs(inp):
    return dict(x=to64(inp["x"]), W0=to64(inp["W0"]), dy=to64(inp["dy"]),
                thP=inp["theta_P"].double().numpy(), thR=inp["theta_R"].double().numpy(),
                pi=inp["perm_in"].numpy(), po=inp["perm_out"].numpy())


def oracle_layer(case, inp, rows=None):
    """Oracle outputs; y and dX only for `rows` (all when None); dtheta over all tokens."""
    o = oracle_inputs(inp)
    QP = oracle.cnp(o["thP"], case.b_in, case.n)
    QR = oracle.cnp(o["thR"], case.b_out, case.n)
    xr = o["x"] if rows is None else o["x"][rows]
    y = oracle.forward(xr, o["W0"], QP, QR, o["pi"], o["po"])
    dX, dQP, dQR = oracle.backward(o["x"], o["dy"], o["W0"], QP, QR, o["pi"], o["po"])
    return dict(y=y, dX=dX if rows is None else dX[rows], Q_P=QP, Q_R=QR,
                dtheta_P=oracle.cnp_backward(o["thP"], case.b_in, case.n, dQP),
                dtheta_R=oracle.cnp_backward(o["thR"], case.b_out, case.n, dQR))


def check_layer(case, inp, save_z=True, rows=None):
    g = gpu_layer(case, inp, save_z=save_z)
    r = oracle_layer(case, inp, rows=rows)
    tol = tol_for(case.dtype)
    errs = {}
    for k in ("Q_P", "Q_R", "dtheta_P", "dtheta_R"):
        errs[k] = assert_close(k, g[k], r[k], tol)
    for k in ("y", "dX"):
        got = g[k] if rows is None else g[k][rows]
        errs[k] = assert_close(k, got, r[k], tol)
    return errs


# ------------------------------------------------------------------ Cayley-Neumann

@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_cnp_tiny_config(out):
    th = inputs.make_theta(16, 32, 0.01, 77)
    Q = torch.empty(16, 32, 32, dtype=torch.float32 if out == "f32" else torch.bfloat16,
                    device="cuda")
    _lib.poetx_cayley_neumann(th.cuda(), 32, 4, Q)
    _lib.poetx_stream_status()
    assert_close("Q", to64(Q), oracle.cnp(th.double().numpy(), 32, 4), tol_for(out))


@pytest.mark.parametrize("b", [2, 4, 8, 16])
def test_cnp_small_blocks_fp32(b):
    th = inputs.make_theta(5, b, 0.05, 78 + b)
    Q = torch.empty(5, b, b, dtype=torch.float32, device="cuda")
    _lib.poetx_cayley_neumann(th.cuda(), b, 3, Q)
    _lib.poetx_stream_status()
    assert_close("Q", to64(Q), oracle.cnp(th.double().numpy(), b, 3), TOL_F32)


SWEEP = [(b, s, n, out) for b in inputs.CNP_SWEEP.bs for s in inputs.CNP_SWEEP.sigmas
         for n in inputs.CNP_SWEEP.ns for out in ("f32", "bf16")]


@pytest.mark.parametrize("b,sigma,n,out", SWEEP)
def test_cnp_sweep_full_size_sampled_blocks(b, sigma, n, out):
    """4096 blocks per point at full size; the oracle checks sampled blocks one by one."""
    nb = inputs.CNP_SWEEP.nb
    th = inputs.make_theta(nb, b, sigma, inputs.sweep_seed(b, sigma, n))
    dt = torch.float32 if out == "f32" else torch.bfloat16
    Q = torch.empty(nb, b, b, dtype=dt, device="cuda")
    _lib.poetx_cayley_neumann(th.cuda(), b, n, Q)
    _lib.poetx_stream_status()
    idx = np.array([0, 1, 1234, 2047, 3001, nb - 1])
    ref = oracle.cnp(th[idx].double().numpy(), b, n)
    got = to64(Q[torch.as_tensor(idx, device="cuda")])
    assert_close("Q", got, ref, tol_for(out))
    if out == "f32":
        # orthogonality defect ||Q^T Q - I||_F agrees with the oracle's within the
        # perturbation bound 2 ||Q||_2 ||dQ||_F + ||dQ||_F^2 (plus fp32 rounding of I)
        e_got, e_ref = oracle.orth_error(got), oracle.orth_error(ref)
        dq = np.sqrt(((got - ref) ** 2).sum(axis=(1, 2)))
        q2 = np.linalg.norm(ref, ord=2, axis=(1, 2))
        bound = 2 * q2 * dq + dq ** 2 + 4 * b * 2.0 ** -24
        assert np.all(np.abs(e_got - e_ref) <= bound), (e_got, e_ref, bound)


@pytest.mark.parametrize("b,nb_P,nb_R", [(32, 7, 5), (64, 3, 9), (128, 2, 3), (32, 1, 0),
                                         (64, 0, 1)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_cnp_tile_ragged_tiles_and_both_factors(b, nb_P, nb_R, out):
    """The tile kernel packs 128 / b blocks per 128-row tile and takes both
    factors of a layer in one launch: block counts that leave a partial last
    tile on either factor, every block checked against the oracle."""
    dt = torch.float32 if out == "f32" else torch.bfloat16
    thP = inputs.make_theta(nb_P, b, 0.01, 3100 + b + nb_P)
    thR = inputs.make_theta(nb_R, b, 0.01, 3200 + b + nb_R)
    QP = torch.full((max(nb_P, 1), b, b), float("nan"), dtype=dt, device="cuda")[:nb_P]
    QR = torch.full((max(nb_R, 1), b, b), float("nan"), dtype=dt, device="cuda")[:nb_R]
    _lib.poetx_cayley_neumann_pair(thP.cuda(), b, thR.cuda(), b, 5, QP, QR)
    _lib.poetx_stream_status()
    for name, th, Q in (("Q_P", thP, QP), ("Q_R", thR, QR)):
        if th.shape[0]:
            assert_close(name, to64(Q), oracle.cnp(th.double().numpy(), b, 5), tol_for(out))


def test_cnp_bf16_b128_beyond_the_tensor_core_grid():
    """bf16 Q at b = 128 past 2^16 blocks (the tile kernel walks any number of
    tiles): 65541 blocks (2.1 GB of theta and of Q), blocks sampled at both
    ends and in between against the oracle."""
    nb, b, n = 65541, 128, 3
    th = inputs.make_theta(nb, b, 0.01, 5150)
    Q = torch.empty(nb, b, b, dtype=torch.bfloat16, device="cuda")
    _lib.poetx_cayley_neumann(th.cuda(), b, n, Q)
    _lib.poetx_stream_status()
    idx = np.array([0, 1, 777, 32768, 65534, 65535, 65536, nb - 1])
    ref = oracle.cnp(th[idx].double().numpy(), b, n)
    assert_close("Q", to64(Q[torch.as_tensor(idx, device="cuda")]), ref, TOL_BF16)
    del Q
    torch.cuda.empty_cache()


@pytest.mark.parametrize("b,n", [(2, 1), (4, 3), (32, 4), (64, 2), (128, 3), (256, 3), (256, 6)])
def test_cnp_backward_parity(b, n):
    nb = 6
    th = inputs.make_theta(nb, b, 0.01, 91 + b + n)
    g = torch.Generator().manual_seed(92 + b * 7 + n)
    dQ = torch.randn(nb, b, b, generator=g)
    dth = torch.empty_like(th, device="cuda")
    _lib.poetx_cayley_neumann_backward(th.cuda(), dQ.cuda(), b, n, dth)
    _lib.poetx_stream_status()
    ref = oracle.cnp_backward(th.double().numpy(), b, n, dQ.double().numpy())
    assert_close("dtheta", dth.double().cpu().numpy(), ref, TOL_F32)


# ------------------------------------------------------------------ index maps

@pytest.mark.parametrize("b_P,b_R", [(256, 256), (128, 128), (256, 128), (32, 64)])
def test_cnp_pair_matches_single_calls(b_P, b_R):
    """poetx_cayley_neumann_pair (both factors of a layer, one launch when the
    block sizes agree) computes exactly what two single calls compute."""
    thP = inputs.make_theta(8, b_P, 0.01, 77).cuda()
    thR = inputs.make_theta(6, b_R, 0.01, 78).cuda()
    bf = torch.bfloat16
    QP = torch.empty(8, b_P, b_P, dtype=bf, device="cuda")
    QR = torch.empty(6, b_R, b_R, dtype=bf, device="cuda")
    _lib.poetx_cayley_neumann_pair(thP, b_P, thR, b_R, 3, QP, QR)
    QP1, QR1 = torch.empty_like(QP), torch.empty_like(QR)
    _lib.poetx_cayley_neumann(thP, b_P, 3, QP1)
    _lib.poetx_cayley_neumann(thR, b_R, 3, QR1)
    _lib.poetx_stream_status()
    assert torch.equal(QP, QP1) and torch.equal(QR, QR1)
    ref = oracle.cnp(thR.double().cpu().numpy(), b_R, 3)
    assert_close("Q_R", to64(QR), ref, TOL_BF16)


@pytest.mark.parametrize("d", [1, 7, 256, 2048, 5632])
def test_invert_perm_bit_exact(d):
    perm = torch.randperm(d, generator=torch.Generator().manual_seed(d)).to(torch.int32)
    inv = torch.empty(d, dtype=torch.int32, device="cuda")
    _lib.poetx_invert_perm(perm.cuda(), inv)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(inv.cpu().numpy(), oracle.invert_perm(perm.numpy()))
    scratch = torch.empty(d + 1, dtype=torch.int32, device="cuda")
    assert _lib.poetx_check_perm(perm.cuda(), inv, scratch) == 0


def test_check_perm_rejects_non_permutations():
    scratch = torch.empty(9, dtype=torch.int32, device="cuda")
    for bad in ([0, 0, 1, 2, 3, 4, 5, 6], [0, 1, 2, 3, 4, 5, 6, 8], [-1, 1, 2, 3, 4, 5, 6, 7]):
        p = torch.tensor(bad, dtype=torch.int32, device="cuda")
        assert _lib.poetx_check_perm(p, None, scratch) == 4
    p = torch.arange(8, dtype=torch.int32, device="cuda")
    wrong_inv = torch.tensor([1, 0, 2, 3, 4, 5, 6, 7], dtype=torch.int32, device="cuda")
    assert _lib.poetx_check_perm(p, wrong_inv, scratch) == 4
    assert _lib.poetx_check_perm(p, p, scratch) == 0


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_merge_w0_bit_exact(dt):
    d_out, d_in = 384, 256
    g = torch.Generator().manual_seed(5)
    W0 = torch.randn(d_out, d_in, generator=g).to(dt)
    po = torch.randperm(d_out, generator=g).to(torch.int32)
    pi = torch.randperm(d_in, generator=g).to(torch.int32)
    W0m = torch.empty(d_out, d_in, dtype=dt, device="cuda")
    _lib.poetx_merge_w0(W0.cuda(), W0m, po.cuda(), pi.cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to64(W0m), oracle.merge_w0(to64(W0), po.numpy(), pi.numpy()))


# ------------------------------------------------------------------ end of an inner loop

@pytest.mark.parametrize("dt,d_in,d_out,b_in,b_out", [
    ("f32", 256, 256, 32, 32), ("f32", 96, 64, 8, 16), ("bf16", 256, 384, 32, 64),
    ("bf16", 1024, 1024, 128, 128), ("bf16", 2048, 2048, 256, 256), ("bf16", 64, 128, 4, 8)])
def test_fold_w0_parity(dt, d_in, d_out, b_in, b_out):
    """W0_new = R W0 P from the merged weight, against the oracle's dense product
    (the blocks are seeded random matrices: the fold is linear in them)."""
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(7 * d_in + d_out)
    W0 = (torch.randn(d_out, d_in, generator=g) * d_in ** -0.5).to(tdt)
    QP = (torch.randn(d_in // b_in, b_in, b_in, generator=g) * b_in ** -0.5).to(tdt)
    QR = (torch.randn(d_out // b_out, b_out, b_out, generator=g) * b_out ** -0.5).to(tdt)
    pi = torch.randperm(d_in, generator=g).to(torch.int32)
    po = torch.randperm(d_out, generator=g).to(torch.int32)
    W0m = torch.empty(d_out, d_in, dtype=tdt, device="cuda")
    _lib.poetx_merge_w0(W0.cuda(), W0m, po.cuda(), pi.cuda())
    ws = torch.empty(_lib.poetx_fold_workspace_bytes(d_out, d_in, b_in, b_out, tdt),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(W0m)
    _lib.poetx_fold_w0(W0m, QP.cuda(), QR.cuda(), pi.cuda(), po.cuda(), b_in, b_out, out, ws)
    inplace = W0m.clone()
    _lib.poetx_fold_w0(inplace, QP.cuda(), QR.cuda(), pi.cuda(), po.cuda(), b_in, b_out, inplace,
                       ws)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    ref = oracle.fold_w0(to64(W0), to64(QP), to64(QR), pi.numpy(), po.numpy())
    assert_close("W0_new", to64(out), ref, tol_for(dt))
    assert torch.equal(out, inplace)


def test_fold_w0_rejects_a_small_workspace():
    W0m = torch.zeros(64, 64, device="cuda")
    Q = torch.zeros(4, 16, 16, device="cuda")
    p = torch.arange(64, dtype=torch.int32, device="cuda")
    need = _lib.poetx_fold_workspace_bytes(64, 64, 16, 16, torch.float32)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.PoetxError) as e:
        _lib.poetx_fold_w0(W0m, Q, Q, p, p, 16, 16, W0m, ws)
    assert e.value.code == 2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_merge_and_resample_keeps_the_function(dtype):
    """An inner loop ends: W0 <- R W0 P, theta <- 0, new permutations.  The
    layer's forward is the same function before and after (both against the
    oracle's forward with the original parameters)."""
    case = inputs.LinearCase("resample", 512, 768, 128, 256, 3, 300, 0.05, dtype, 911)
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T)
    x = inp["x"].cuda()
    lay.cayley_neumann()
    y0 = lay.forward(x).clone()
    g = torch.Generator().manual_seed(3)
    pi1 = torch.randperm(case.d_in, generator=g).to(torch.int32)
    po1 = torch.randperm(case.d_out, generator=g).to(torch.int32)
    lay.merge_and_resample(pi1, po1)
    y1 = lay.forward(x)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    assert float(lay.theta_P.abs().max()) == 0.0 and float(lay.theta_R.abs().max()) == 0.0
    assert torch.equal(lay.perm_in.cpu(), pi1) and torch.equal(lay.perm_out.cpu(), po1)
    assert torch.equal(lay.inv_in.cpu()[pi1.long()], torch.arange(case.d_in, dtype=torch.int32))
    eye = torch.eye(case.b_in, dtype=lay.Q_P.dtype, device="cuda")
    assert torch.equal(lay.Q_P, eye.expand_as(lay.Q_P))
    o = oracle_inputs(inp)
    QP = oracle.cnp(o["thP"], case.b_in, case.n)
    QR = oracle.cnp(o["thR"], case.b_out, case.n)
    ref = oracle.forward(o["x"], o["W0"], QP, QR, o["pi"], o["po"])
    tol = tol_for(dtype)
    assert_close("y before", to64(y0), ref, tol)
    assert_close("y after", to64(y1), ref, tol)


# ------------------------------------------------------------------ POET-XQ (INT8 frozen weight)

@pytest.mark.parametrize("dt,d_out,d_in", [(torch.bfloat16, 2048, 2048), (torch.float32, 384, 260),
                                           (torch.bfloat16, 5632, 2048)])
def test_quantize_w0_codes_bit_exact(dt, d_out, d_in):
    g = torch.Generator().manual_seed(d_out + d_in)
    W = (torch.randn(d_out, d_in, generator=g) * torch.rand(d_out, 1, generator=g)).to(dt)
    W[3] = 0                                              # a zero row: scale 0, codes 0
    q = torch.empty(d_out, d_in, dtype=torch.int8, device="cuda")
    sc = torch.empty(d_out, dtype=torch.float32, device="cuda")
    _lib.poetx_quantize_w0(W.cuda(), q, sc)
    Wd = torch.empty(d_out, d_in, dtype=dt, device="cuda")
    _lib.poetx_dequantize_w0(q, sc, Wd)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_rows_int8(W.float().numpy())
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    # dequantised: the fp32 product code * scale, rounded once to the dtype
    want = (torch.from_numpy(q_ref).float() * torch.from_numpy(s_ref)[:, None]).to(dt)
    assert torch.equal(Wd.cpu(), want)


def xq_oracle_layer(case, inp, rows=None):
    """The oracle layer with the weight the GPU multiplies by: the INT8 codes
    of W0 dequantised (in double)."""
    o = oracle_inputs(inp)
    q, s = oracle.quantize_rows_int8(inp["W0"].float().numpy())
    W0 = oracle.dequantize_rows(q, s)
    QP = oracle.cnp(o["thP"], case.b_in, case.n)
    QR = oracle.cnp(o["thR"], case.b_out, case.n)
    xr = o["x"] if rows is None else o["x"][rows]
    y = oracle.forward(xr, W0, QP, QR, o["pi"], o["po"])
    dX, dQP, dQR = oracle.backward(o["x"], o["dy"], W0, QP, QR, o["pi"], o["po"])
    return dict(y=y, dX=dX if rows is None else dX[rows],
                dtheta_P=oracle.cnp_backward(o["thP"], case.b_in, case.n, dQP),
                dtheta_R=oracle.cnp_backward(o["thR"], case.b_out, case.n, dQR))


@pytest.mark.parametrize("name,d,b,T,dtype,save_z", [
    ("xq_tiny", 256, 32, 64, "f32", True), ("xq_tiny", 256, 32, 64, "f32", False),
    ("xq_1024", 1024, 128, 1000, "bf16", True), ("xq_1024", 1024, 128, 1000, "bf16", False),
    ("xq_2048", 2048, 256, 8192, "bf16", True)])
def test_xq_layer_parity(name, d, b, T, dtype, save_z):
    case = inputs.LinearCase(name, d, d, b, b, 3, T, 0.01, dtype, 913)
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], b, b, 3, T_max=T, save_z=save_z, w0_int8=True)
    assert lay.W0m is None and lay.W0q.dtype == torch.int8
    y, dX, dtp, dtr = lay.step(inp["x"].cuda(), inp["dy"].cuda())
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    rows = SAMPLE_ROWS(T) if T > 2048 else None
    r = xq_oracle_layer(case, inp, rows=rows)
    tol = tol_for(dtype)
    got = dict(y=to64(y), dX=to64(dX), dtheta_P=dtp.double().cpu().numpy(),
               dtheta_R=dtr.double().cpu().numpy())
    for k in ("dtheta_P", "dtheta_R"):
        assert_close(k, got[k], r[k], tol)
    for k in ("y", "dX"):
        assert_close(k, got[k] if rows is None else got[k][rows], r[k], tol)


def test_xq_merge_and_resample_keeps_the_function():
    case = inputs.LinearCase("xq_resample", 512, 768, 128, 256, 3, 300, 0.05, "bf16", 914)
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T,
                            w0_int8=True)
    x = inp["x"].cuda()
    lay.cayley_neumann()
    y0 = lay.forward(x).clone()
    g = torch.Generator().manual_seed(4)
    lay.merge_and_resample(torch.randperm(case.d_in, generator=g),
                           torch.randperm(case.d_out, generator=g))
    y1 = lay.forward(x)
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    ref = xq_oracle_layer(case, inp)["y"]
    assert_close("y before", to64(y0), ref, TOL_BF16)
    assert_close("y after", to64(y1), ref, TOL_BF16)


# ------------------------------------------------------------------ the layer

@pytest.mark.parametrize("save_z", [True, False])
def test_layer_tiny_fp32_config(save_z):
    case = inputs.TINY_FP32
    check_layer(case, inputs.make_linear_inputs(case), save_z=save_z)


@pytest.mark.parametrize("b", [2, 4, 8, 16, 64])
def test_layer_fp32_block_sizes_ragged_tokens(b):
    case = inputs.LinearCase("fp32_b%d" % b, 128, 192, b, min(2 * b, 64), 3, 37, 0.02, "f32", 600 + b)
    check_layer(case, inputs.make_linear_inputs(case))


@pytest.mark.parametrize("b_in,b_out", [(32, 64), (64, 32), (128, 128), (256, 256), (256, 128)])
@pytest.mark.parametrize("T", [1, 200, 384])
def test_layer_bf16_tiles_and_ragged_tail(b_in, b_out, T):
    case = inputs.LinearCase("bf16_%d_%d_%d" % (b_in, b_out, T), 512, 768, b_in, b_out, 3, T,
                             0.005, "bf16", 700 + b_in + b_out + T)
    check_layer(case, inputs.make_linear_inputs(case))


@pytest.mark.parametrize("b", [256, 128])
def test_bf16_step_runs_on_the_tensor_core_kernels(b):
    """The 2048-wide bf16 layer takes the sm_103a paths: cluster block applies,
    tcgen05 GEMMs, cluster dQ sums (the permuted operand gathered in flight, no
    permuted copy written) and the tensor-core Cayley-Neumann kernels (a silent
    fall-back to the slab, permute-then-sum or CUDA-core kernels would still
    pass the parity tests, so the launched kernels are checked by name)."""
    case = inputs.LinearCase("paths_%d" % b, 2048, 2048, b, b, 3, 256, 0.005, "bf16", 990 + b)
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], b, b, 3, T_max=case.T)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    lay.step(x, dy)
    torch.cuda.synchronize()
    _lib.poetx_profile_report()
    _lib.poetx_profile_enable(True)
    try:
        lay.step(x, dy)
        torch.cuda.synchronize()
    finally:
        _lib.poetx_profile_enable(False)
    names = set(_lib.poetx_profile_report())
    for k in ("tc_cluster_gather", "tc_cluster_scatter", "tc_gemm_nt", "tc_gemm_nn",
              "tc_cluster_dq", "tc_cnp_fwd" if b == 256 else "tc_cnp_tile", "tc_cnp_bwd"):
        assert k in names, (k, sorted(names))
    assert not any(n.endswith("_simt") for n in names), sorted(names)
    assert "tc_permute_cols" not in names and "tc_dq" not in names, sorted(names)


@pytest.mark.parametrize("d_in,d_out,b,T", [(4352, 512, 128, 333), (512, 5632, 256, 200),
                                           (5632, 256, 256, 131)])
def test_staged_applies_parity(d_in, d_out, b, T):
    """Sides whose blocks do not fit the cluster applies (34 blocks of 128, 22
    of 256: a CTA's share exceeds its tensor memory) run a column permutation
    through the scratch plus the unpermuted block apply; ragged token tiles."""
    case = inputs.LinearCase("staged_%d_%d_%d" % (d_in, d_out, b), d_in, d_out, b, b, 3, T, 0.005,
                             "bf16", 880 + T)
    check_layer(case, inputs.make_linear_inputs(case))


@pytest.mark.parametrize("which", [4, 6])   # gate 2048 -> 5632, down 5632 -> 2048
def test_wide_stack_layers_run_on_the_staged_applies(which):
    """The stack's 5632-wide side (22 blocks of 256) takes the column
    permutation plus the unpermuted apply on the tensor cores, not the slab
    kernel or the CUDA cores (checked by name: parity alone would not show a
    fall-back)."""
    case = inputs.stack_cases(T=256, layers=1)[which]
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    lay.step(x, dy)
    torch.cuda.synchronize()
    _lib.poetx_profile_report()
    _lib.poetx_profile_enable(True)
    try:
        lay.step(x, dy)
        torch.cuda.synchronize()
    finally:
        _lib.poetx_profile_enable(False)
    names = set(_lib.poetx_profile_report())
    for k in ("tc_plain_apply", "tc_permute_cols", "tc_dq", "tc_cluster_gather",
              "tc_cluster_scatter", "tc_cluster_dq", "tc_gemm_nt", "tc_gemm_nn"):
        assert k in names, (k, sorted(names))
    assert not any(n.startswith("tc_blockapply") or n.endswith("_simt") for n in names), sorted(names)


@pytest.mark.parametrize("b", [32, 256])
def test_cnp_fp32_chain_beyond_fp16_range_reports_a_status(b):
    """fp32 Q on the tensor cores holds chain values as two fp16 parts: a
    chain far outside the series' convergent range (sigma = 10, values past
    65504) is reported as POETX_ERR_RANGE by the next status read, and the
    context stays usable (the next call in range is checked against the
    oracle)."""
    Q = torch.empty(4, b, b, dtype=torch.float32, device="cuda")
    _lib.poetx_stream_status()
    _lib.poetx_cayley_neumann(inputs.make_theta(4, b, 10.0, 93).cuda(), b, 3, Q)
    torch.cuda.synchronize()
    with pytest.raises(_lib.PoetxError) as e:
        _lib.poetx_stream_status()
    assert e.value.code == 7
    th = inputs.make_theta(4, b, 1e-2, 94)
    _lib.poetx_cayley_neumann(th.cuda(), b, 3, Q)
    _lib.poetx_stream_status()
    assert_close("Q", to64(Q), oracle.cnp(th.double().numpy(), b, 3), TOL_F32)


@pytest.mark.parametrize("nb_P,nb_R", [(3, 0), (2, 5)])
def test_cnp_fp32_b256_runs_on_the_tensor_cores(nb_P, nb_R):
    """fp32 Q of 256-blocks: the split unpack and the three-term chain on the
    tensor cores (checked by name: parity alone would not show the CUDA-core
    kernel), one factor and both factors of a layer in one call, against the
    oracle block by block."""
    n = 3
    thP = inputs.make_theta(nb_P, 256, 1e-2, 91)
    thR = inputs.make_theta(max(nb_R, 1), 256, 1e-2, 92)[:nb_R]
    QP = torch.empty(nb_P, 256, 256, dtype=torch.float32, device="cuda")
    QR = torch.empty(max(nb_R, 1), 256, 256, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    _lib.poetx_profile_report()
    _lib.poetx_profile_enable(True)
    try:
        if nb_R == 0:
            _lib.poetx_cayley_neumann(thP.cuda(), 256, n, QP)
        else:
            _lib.poetx_cayley_neumann_pair(thP.cuda(), 256, thR.cuda(), 256, n, QP, QR[:nb_R])
        torch.cuda.synchronize()
    finally:
        _lib.poetx_profile_enable(False)
    _lib.poetx_stream_status()
    names = set(_lib.poetx_profile_report())
    assert {"tc_cnp_unpack_f32", "tc_cnp_fwd_f32"} <= names, sorted(names)
    assert not any(k.endswith("_simt") for k in names), sorted(names)
    assert_close("Q_P", to64(QP), oracle.cnp(thP.double().numpy(), 256, n), TOL_F32)
    if nb_R:
        assert_close("Q_R", to64(QR[:nb_R]), oracle.cnp(thR.double().numpy(), 256, n), TOL_F32)


@pytest.mark.parametrize("d_in,d_out,T", [(512, 768, 200), (2048, 2048, 600)])
@pytest.mark.parametrize("b,n", [(256, 1), (256, 2), (256, 5), (128, 1), (128, 4)])
def test_bf16_chain_backward_orders(d_in, d_out, T, b, n):
    """The tensor-core Cayley-Neumann backward at several truncation orders,
    both block sizes: the cluster form (a block split over row halves and
    64-column slabs; n = 1 has no exchange step) and, where the backward runs
    on two streams (the 2048 layer), the two-CTA ring form of the R side."""
    case = inputs.LinearCase("chain_%d_%d_%d" % (d_in, b, n), d_in, d_out, b, b, n, T, 0.005, "bf16",
                             610 + b + n + d_in)
    check_layer(case, inputs.make_linear_inputs(case))


def test_xfast_and_xmem_give_the_same_gradients():
    """POET-Xmem recomputes z with the forward's own kernels, so y and dX are
    bit-identical to POET-Xfast; the block gradients are token sums kept as
    per-range partials that are added in a fixed order (no atomics), so dtheta
    is bit-identical too."""
    case = inputs.LinearCase("xmem", 512, 512, 128, 128, 3, 300, 0.005, "bf16", 801)
    inp = inputs.make_linear_inputs(case)
    a = gpu_layer(case, inp, save_z=True)
    b = gpu_layer(case, inp, save_z=False)
    for k in ("y", "dX", "dtheta_P", "dtheta_R"):
        assert np.array_equal(b[k], a[k]), k


@pytest.mark.parametrize("d,b,T", [(2048, 256, 8192), (1024, 128, 1000)])
def test_bf16_layer_is_run_to_run_deterministic(d, b, T):
    """Every output of the tensor-core step is a fixed function of the inputs:
    two runs agree bit for bit."""
    case = inputs.LinearCase("det", d, d, b, b, 3, T, 0.005, "bf16", 803)
    inp = inputs.make_linear_inputs(case)
    a = gpu_layer(case, inp, save_z=True)
    c = gpu_layer(case, inp, save_z=True)
    for k in ("y", "dX", "dtheta_P", "dtheta_R"):
        assert np.array_equal(c[k], a[k]), k


@pytest.mark.parametrize("save_z", [True, False])
def test_captured_step_replays_the_eager_step(save_z):
    """A step captured into a CUDA graph and replayed on new inputs gives, bit
    for bit, what the eager step gives on those inputs; the profiled capture's
    per-kernel event pairs are readable after a replay."""
    case = inputs.LinearCase("graph", 2048, 2048, 256, 256, 3, 4096, 0.005, "bf16", 804)
    inp = inputs.make_linear_inputs(case)
    dev = torch.device("cuda")
    lay = TransformedLinear(inp["W0"].to(dev), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T,
                            save_z=save_z)
    x, dy = inp["x"].to(dev), inp["dy"].to(dev)
    y = torch.empty(case.T, case.d_out, dtype=torch.bfloat16, device=dev)
    dX = torch.empty(case.T, case.d_in, dtype=torch.bfloat16, device=dev)
    graph = lay.capture_step(x, dy, y, dX)
    gen = torch.Generator(device=dev).manual_seed(5)
    x2 = torch.randn(case.T, case.d_in, generator=gen, device=dev).to(torch.bfloat16)
    dy2 = torch.randn(case.T, case.d_out, generator=gen, device=dev).to(torch.bfloat16)
    ye, dXe, dtpe, dtre = [t.clone() for t in lay.step(x2, dy2)]
    x.copy_(x2)
    dy.copy_(dy2)
    graph.replay()
    _lib.poetx_stream_status()
    torch.cuda.synchronize()
    assert torch.equal(y, ye) and torch.equal(dX, dXe)
    assert torch.equal(lay.dtheta_P, dtpe) and torch.equal(lay.dtheta_R, dtre)
    _lib.poetx_profile_report()
    _lib.poetx_profile_enable(True)
    try:
        pg = lay.capture_step(x, dy, y, dX, warm=False)
    finally:
        _lib.poetx_profile_enable(False)
    pg.replay()
    torch.cuda.synchronize()
    rep = _lib.poetx_profile_report()
    assert "tc_gemm_nt" in rep and all(v[1] > 0 for v in rep.values()), rep


def test_zero_tokens_is_a_no_op_with_zero_gradients():
    case = inputs.LinearCase("empty", 256, 256, 32, 32, 3, 0, 0.01, "f32", 802)
    inp = inputs.make_linear_inputs(case, T=0)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], 32, 32, 3, T_max=1)
    x = torch.empty(0, 256, device="cuda")
    dy = torch.empty(0, 256, device="cuda")
    lay.dtheta_P.fill_(7.0)
    y, dX, dtp, dtr = lay.step(x, dy)
    _lib.poetx_stream_status()
    assert y.shape == (0, 256) and dX.shape == (0, 256)
    assert float(dtp.abs().max()) == 0.0 and float(dtr.abs().max()) == 0.0


def test_small_workspace_is_rejected():
    case = inputs.TINY_FP32
    inp = inputs.make_linear_inputs(case)
    lay = TransformedLinear(inp["W0"].cuda(), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], 32, 32, 4, T_max=64)
    lay.workspace = lay.workspace[:1024]
    lay.cayley_neumann()
    with pytest.raises(_lib.PoetxError) as e:
        lay.forward(inp["x"].cuda())
    assert e.value.code == 2


# ------------------------------------------------------------------ full-size configs

SAMPLE_ROWS = lambda T: np.unique(np.concatenate([[0, 1, T // 2, T - 2, T - 1],
                                                   np.random.default_rng(T).integers(0, T, 27)]))


def test_full_size_square_2048():
    case = inputs.SQUARE_2048
    check_layer(case, inputs.make_linear_inputs(case), rows=SAMPLE_ROWS(case.T))


def test_full_size_upproj_2048x5632():
    case = inputs.UPPROJ
    check_layer(case, inputs.make_linear_inputs(case), rows=SAMPLE_ROWS(case.T))


@pytest.mark.parametrize("which", [0, 4, 6])   # q (2048->2048), gate (2048->5632), down (5632->2048)
def test_full_size_stack_layer_shapes(which):
    case = inputs.stack_cases()[which]
    check_layer(case, inputs.make_linear_inputs(case), rows=SAMPLE_ROWS(case.T))
