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
