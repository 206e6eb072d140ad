"""The data-parallel path on CPU: two `gloo` ranks, no GPU.

Each rank runs the layer (the oracle, in double) on its own token shard with
the replicated weights, permutations and skew parameters, then the packed
gradients are summed over ranks with ``dp.allreduce_dtheta`` -- the one
exchange of the distributed job ("POET-X: Memory-efficient LLM Training by
Scaling Orthogonal Transformation", gist.science summary, section 4: DDP).
The summed gradients must equal the gradients of the whole batch, and each
rank's y and dX rows must equal the whole batch's rows of its shard.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from orthogonal_equivalence_neumann_b300 import dp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(T):
    rng = np.random.default_rng(31)
    d_in, d_out, b_in, b_out, n = 16, 12, 4, 6, 3
    return dict(
        x=rng.standard_normal((T, d_in)), dy=rng.standard_normal((T, d_out)),
        W0=rng.standard_normal((d_out, d_in)) / 4.0,
        thP=rng.standard_normal((d_in // b_in, b_in * (b_in - 1) // 2)) * 0.1,
        thR=rng.standard_normal((d_out // b_out, b_out * (b_out - 1) // 2)) * 0.1,
        pi=rng.permutation(d_in).astype(np.int32), po=rng.permutation(d_out).astype(np.int32),
        b_in=b_in, b_out=b_out, n=n)


def _layer(c, rows):
    import oracle
    return oracle.layer(c["x"][rows], c["W0"], c["thP"], c["thR"], c["n"], c["pi"], c["po"],
                        c["b_in"], c["b_out"], dy=c["dy"][rows])


def _rank_main(rank, port, T, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        c = _case(T)
        sh = dp.token_shard(T, WORLD, rank)
        r = _layer(c, sh)
        dtp = torch.from_numpy(r["dtheta_P"].copy())
        dtr = torch.from_numpy(r["dtheta_R"].copy())
        dp.allreduce_dtheta(dtp, dtr)
        slowest = dp.max_over_ranks(float(rank + 1))
        np.savez(os.path.join(out_dir, "rank%d.npz" % rank), dtheta_P=dtp.numpy(),
                 dtheta_R=dtr.numpy(), y=r["y"], dX=r["dX"], start=sh.start, stop=sh.stop,
                 slowest=slowest)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T", [11, 2])
def test_two_ranks_sum_to_the_whole_batch(T, tmp_path):
    mp.start_processes(_rank_main, args=(_free_port(), T, str(tmp_path)), nprocs=WORLD,
                       join=True, start_method="spawn")
    full = _layer(_case(T), slice(0, T))
    covered = np.zeros(T, dtype=int)
    for rank in range(WORLD):
        g = np.load(tmp_path / ("rank%d.npz" % rank))
        np.testing.assert_allclose(g["dtheta_P"], full["dtheta_P"], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dtheta_R"], full["dtheta_R"], rtol=1e-12, atol=1e-13)
        rows = slice(int(g["start"]), int(g["stop"]))
        np.testing.assert_allclose(g["y"], full["y"][rows], rtol=0, atol=1e-13)
        np.testing.assert_allclose(g["dX"], full["dX"][rows], rtol=0, atol=1e-13)
        covered[rows] += 1
        assert float(g["slowest"]) == WORLD
    np.testing.assert_array_equal(covered, 1)


@pytest.mark.parametrize("T,world", [(0, 3), (7, 1), (7, 3), (8192, 8), (5, 8)])
def test_token_shards_cover_every_token_once(T, world):
    seen = np.zeros(T, dtype=int)
    sizes = []
    for r in range(world):
        s = dp.token_shard(T, world, r)
        seen[s] += 1
        sizes.append(s.stop - s.start)
    np.testing.assert_array_equal(seen, 1)
    assert max(sizes) - min(sizes) <= 1


def test_single_process_exchange_is_a_no_op():
    a, b = torch.ones(3), torch.full((2,), 2.0)
    assert dp.allreduce_dtheta(a, b) is None
    assert dp.max_over_ranks(4.5) == 4.5
    assert torch.equal(a, torch.ones(3)) and torch.equal(b, torch.full((2,), 2.0))


# ---- a three-layer chain with the exchange overlapped: each layer's packed
# gradients are all-reduced asynchronously as soon as its backward has made
# them, and the step waits for all of them at the end.

class _OracleLayer:
    """One layer of a chain for the CPU test: the oracle's forward and backward
    in double, with the gradient buffers the exchange works on in place."""

    def __init__(self, seed, d_in, d_out, b_in, b_out, n=3):
        rng = np.random.default_rng(seed)
        self.W0 = rng.standard_normal((d_out, d_in)) / np.sqrt(d_in)
        self.thP = rng.standard_normal((d_in // b_in, b_in * (b_in - 1) // 2)) * 0.1
        self.thR = rng.standard_normal((d_out // b_out, b_out * (b_out - 1) // 2)) * 0.1
        self.pi = rng.permutation(d_in).astype(np.int32)
        self.po = rng.permutation(d_out).astype(np.int32)
        self.b_in, self.b_out, self.n = b_in, b_out, n

    def forward(self, x):
        import oracle
        return oracle.layer(x, self.W0, self.thP, self.thR, self.n, self.pi, self.po, self.b_in,
                            self.b_out)["y"]

    def backward(self, x, dy):
        import oracle
        r = oracle.layer(x, self.W0, self.thP, self.thR, self.n, self.pi, self.po, self.b_in,
                         self.b_out, dy=dy)
        self.dtheta_P = torch.from_numpy(r["dtheta_P"].copy())
        self.dtheta_R = torch.from_numpy(r["dtheta_R"].copy())
        return r["dX"], self.dtheta_P, self.dtheta_R


def _chain(T):
    layers = [_OracleLayer(41, 16, 12, 4, 6), _OracleLayer(42, 12, 12, 6, 3),
              _OracleLayer(43, 12, 16, 3, 8)]
    rng = np.random.default_rng(44)
    return layers, rng.standard_normal((T, 16)), rng.standard_normal((T, 16))


def _chain_grads(layers, x, dy, exchange=None):
    xs = [x]
    for lay in layers[:-1]:
        xs.append(lay.forward(xs[-1]))
    dX = dp.backward_layers(layers, xs, dy, exchange)
    return dX, [(lay.dtheta_P, lay.dtheta_R) for lay in layers]


def _chain_rank_main(rank, port, T, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        layers, x, dy = _chain(T)
        sh = dp.token_shard(T, WORLD, rank)
        ex = dp.GradientExchange()
        dX, grads = _chain_grads(layers, x[sh], dy[sh], ex)
        issued = ex.pending()
        ex.wait()
        np.savez(os.path.join(out_dir, "chain%d.npz" % rank), dX=dX, start=sh.start,
                 stop=sh.stop, issued=issued, pending=ex.pending(),
                 **{"g%d_%s" % (i, s): t.numpy() for i, g in enumerate(grads)
                    for s, t in zip("PR", g)})
    finally:
        dist.destroy_process_group()


def test_chain_of_three_layers_with_the_exchange_overlapped(tmp_path):
    T = 9
    mp.start_processes(_chain_rank_main, args=(_free_port(), T, str(tmp_path)), nprocs=WORLD,
                       join=True, start_method="spawn")
    layers, x, dy = _chain(T)
    dX_full, full = _chain_grads(layers, x, dy)
    for rank in range(WORLD):
        g = np.load(tmp_path / ("chain%d.npz" % rank))
        # one asynchronous all-reduce per side and layer, all finished by wait()
        assert int(g["issued"]) == 2 * len(layers) and int(g["pending"]) == 0
        for i, (gp, gr) in enumerate(full):
            np.testing.assert_allclose(g["g%d_P" % i], gp.numpy(), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(g["g%d_R" % i], gr.numpy(), rtol=1e-12, atol=1e-13)
        rows = slice(int(g["start"]), int(g["stop"]))
        np.testing.assert_allclose(g["dX"], dX_full[rows], rtol=0, atol=1e-12)
