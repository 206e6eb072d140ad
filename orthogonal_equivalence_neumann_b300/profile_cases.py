"""Small, self-contained workloads for profiling the library's kernels.

    python -m orthogonal_equivalence_neumann_b300.profile_cases layer
        six eager training steps of the square 2048 layer (d_in = d_out = 2048,
        b = 256, n = 3, 8192 bf16 tokens): each step launches the
        Cayley-Neumann kernels, the cluster block applies, the two frozen-weight
        GEMMs and the dQ token sums once or twice; prints the library's
        per-kernel times of the last three steps (CUDA event pairs).
    python -m orthogonal_equivalence_neumann_b300.profile_cases cnp
        three Cayley-Neumann calls at each of four sweep points (4096 blocks,
        n = 3, sigma = 1e-2: b = 128 bf16, b = 128 fp32, b = 32 bf16,
        b = 256 fp32).
    python -m orthogonal_equivalence_neumann_b300.profile_cases gate|down|upproj
        the same six steps as ``layer`` for one of the wide shapes: the MLP
        gate / up projection 2048 -> 5632 and the down projection 5632 -> 2048
        of the 1B-style stack (b = 256, 8192 tokens), or the up-projection
        layer 2048 -> 5632 at b = 128 with 16384 tokens.

Each holds a few hundred MB on the device (the b = 256 fp32 point 1.6 GB)
and runs in seconds, so a profiler can capture one launch of a chosen kernel
(e.g. ``ncu -k regex:<name> -s 2 -c 1``) without replaying a long program.  Inputs are the seeded synthetic
draws of ``inputs``.
"""
import sys

import torch

from . import TransformedLinear, _lib, inputs


def _case(what):
    if what == "layer":
        return inputs.SQUARE_2048
    if what == "upproj":
        return inputs.UPPROJ
    stack = {c.name.split("_")[-1]: c for c in inputs.stack_cases(layers=1)}
    return stack[what]


def layer_steps(what="layer", warm=3, timed=3):
    case = _case(what)
    inp = inputs.make_linear_inputs(case)
    dev = torch.device("cuda")
    lay = TransformedLinear(inp["W0"].to(dev), inp["theta_P"], inp["theta_R"], inp["perm_in"],
                            inp["perm_out"], case.b_in, case.b_out, case.n, T_max=case.T)
    x, dy = inp["x"].to(dev), inp["dy"].to(dev)
    for _ in range(warm):
        lay.step(x, dy)
    torch.cuda.synchronize()
    _lib.poetx_stream_status()
    _lib.poetx_profile_report()
    _lib.poetx_profile_enable(True)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(timed):
        lay.step(x, dy)
    t1.record()
    torch.cuda.synchronize()
    _lib.poetx_profile_enable(False)
    for k, (n, ms) in sorted(_lib.poetx_profile_report().items()):
        print("%-22s %3d launches %8.1f us each" % (k, n, 1000.0 * ms / n))
    print("eager step (event pairs recorded around every kernel) %.1f us" %
          (1000.0 * t0.elapsed_time(t1) / timed))


def cnp_points(calls=3):
    for b, dt in ((128, torch.bfloat16), (128, torch.float32), (32, torch.bfloat16),
                  (256, torch.float32)):
        th = inputs.make_theta(4096, b, 1e-2, inputs.sweep_seed(b, 1e-2, 3)).cuda()
        Q = torch.empty(4096, b, b, dtype=dt, device="cuda")
        for _ in range(calls):
            _lib.poetx_cayley_neumann(th, b, 3, Q)
        torch.cuda.synchronize()
        _lib.poetx_stream_status()
        del th, Q
    print("cnp points ok")


if __name__ == "__main__":
    what = sys.argv[1] if len(sys.argv) > 1 else "layer"
    if what in ("layer", "gate", "down", "upproj"):
        layer_steps(what)
    elif what == "cnp":
        cnp_points()
    else:
        raise SystemExit("usage: python -m orthogonal_equivalence_neumann_b300.profile_cases "
                         "layer|gate|down|upproj|cnp")
