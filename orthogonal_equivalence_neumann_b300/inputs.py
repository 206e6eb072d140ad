"""Seeded synthetic inputs for the transformed linear workloads.

This module is shared by the tests, the benchmark and the smoke check: the same
bytes go to the GPU library and to the CPU oracle.  It holds no arithmetic of
the method -- only random draws (``torch.randn`` scaled to the stated standard
deviation, ``torch.randperm``) and the one rounding of the activations and
weights to bf16, done here once so that both sides read identical values.

The workloads stand in for one 1B-class Llama layer as trained in the POET-X
experiments (the page "POET-X: Memory-efficient LLM Training by Scaling
Orthogonal Transformation", section 4, Llama models on C4); no dataset is
used, only these shapes and distributions.
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch


@dataclass(frozen=True)
class LinearCase:
    """One transformed linear: shapes, block sizes, Neumann terms, distributions."""
    name: str
    d_in: int
    d_out: int
    b_in: int
    b_out: int
    n: int
    T: int
    sigma: float            # std of the packed skew parameters
    dtype: str              # "f32" or "bf16": activations, W0, Q, dy, y, dX
    seed: int
    w0_std: Optional[float] = None   # default 1/sqrt(d_in)

    @property
    def nb_in(self) -> int:
        return self.d_in // self.b_in

    @property
    def nb_out(self) -> int:
        return self.d_out // self.b_out

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_tokens(self, T: int) -> "LinearCase":
        return LinearCase(self.name, self.d_in, self.d_out, self.b_in, self.b_out, self.n, T,
                          self.sigma, self.dtype, self.seed, self.w0_std)


# Tiny fp32 single layer (parity at 1e-5): d=256, 8+8 blocks of b=32, n=4, T=64.
TINY_FP32 = LinearCase("tiny_fp32_d256_b32_n4_T64", 256, 256, 32, 32, 4, 64, 0.01, "f32", 1234)
# Square hidden layer at 1B width: d=2048, 8 blocks of b=256 per side, n=3, 8192 tokens.
SQUARE_2048 = LinearCase("square_d2048_b256_n3_T8192", 2048, 2048, 256, 256, 3, 8192, 0.005,
                         "bf16", 1235)
# MLP up-projection 2048 -> 5632: P 16 x b=128, R 44 x b=128, n=3, 16384 tokens.
UPPROJ = LinearCase("upproj_2048x5632_b128_n3_T16384", 2048, 5632, 128, 128, 3, 16384, 0.005,
                    "bf16", 1236)


@dataclass(frozen=True)
class CnpSweep:
    """Cayley-Neumann generation sweep: 4096 blocks per point."""
    nb: int = 4096
    bs: tuple = (32, 64, 128, 256)
    sigmas: tuple = (1e-3, 1e-2)
    ns: tuple = (1, 2, 3, 4, 5, 6)
    seed: int = 1237


CNP_SWEEP = CnpSweep()


def stack_cases(T: int = 8192, layers: int = 16) -> List[LinearCase]:
    """1B-style stack: 16 layers x (q, k, v, o 2048->2048; gate, up 2048->5632;
    down 5632->2048), b=256, n=3, bf16, fresh activations per linear."""
    shapes = [("q", 2048, 2048), ("k", 2048, 2048), ("v", 2048, 2048), ("o", 2048, 2048),
              ("gate", 2048, 5632), ("up", 2048, 5632), ("down", 5632, 2048)]
    out = []
    for layer in range(layers):
        for li, (nm, di, do) in enumerate(shapes):
            out.append(LinearCase("stack_L%d_%s" % (layer, nm), di, do, 256, 256, 3, T, 0.005,
                                  "bf16", 1238 * 1000 + layer * 16 + li))
    return out


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _sub(case_seed: int, k: int) -> int:
    # sub-seeds for x, W0, theta_P, theta_R, dy, perm_in, perm_out
    return case_seed * 16 + k


def make_linear_inputs(case: LinearCase, T: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """CPU tensors for one case.  ``T`` < case.T returns the first T token rows of
    the same draw (tokens are drawn row by row, so a prefix is the same data)."""
    T_full = case.T
    T = T_full if T is None else T
    dt = case.torch_dtype
    w0_std = case.w0_std if case.w0_std is not None else case.d_in ** -0.5
    p_in = case.b_in * (case.b_in - 1) // 2
    p_out = case.b_out * (case.b_out - 1) // 2
    x = (torch.randn(T_full, case.d_in, generator=_gen(_sub(case.seed, 0)))[:T]).to(dt)
    W0 = (torch.randn(case.d_out, case.d_in, generator=_gen(_sub(case.seed, 1))) * w0_std).to(dt)
    theta_P = torch.randn(case.nb_in, p_in, generator=_gen(_sub(case.seed, 2))) * case.sigma
    theta_R = torch.randn(case.nb_out, p_out, generator=_gen(_sub(case.seed, 3))) * case.sigma
    dy = (torch.randn(T_full, case.d_out, generator=_gen(_sub(case.seed, 4)))[:T]).to(dt)
    perm_in = torch.randperm(case.d_in, generator=_gen(_sub(case.seed, 5))).to(torch.int32)
    perm_out = torch.randperm(case.d_out, generator=_gen(_sub(case.seed, 6))).to(torch.int32)
    return dict(x=x.contiguous(), W0=W0.contiguous(), theta_P=theta_P.float().contiguous(),
                theta_R=theta_R.float().contiguous(), dy=dy.contiguous(),
                perm_in=perm_in, perm_out=perm_out)


def make_theta(nb: int, b: int, sigma: float, seed: int) -> torch.Tensor:
    """Packed skew parameters [nb, b(b-1)/2] ~ N(0, sigma^2), fp32."""
    return (torch.randn(nb, b * (b - 1) // 2, generator=_gen(seed)) * sigma).float().contiguous()


def sweep_seed(b: int, sigma: float, n: int) -> int:
    return CNP_SWEEP.seed * 100000 + b * 100 + int(round(-torch.log10(torch.tensor(sigma)).item())) * 10 + n
