"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and rounds them to bf16; it holds none
of the method's arithmetic.  Both sides receive exactly the same bf16 values
(the oracle widens them to fp64).

Workload shapes follow the CODA write-up ("CODA: Rewriting Transformer Blocks
as GEMM-Epilogue Programs", section on experimental results): the
GEMM-RMSNorm-GEMM pattern at the hidden sizes of LLaMA-style 1B, 7B and 70B
models, plus an LM-head cross-entropy over a 128256-entry vocabulary.

Readings (the write-up gives no distributions; these are the recipe):
  * "N(0, s)" means standard deviation s.
  * Activations X and H are N(0, 1); the residual R is N(0, 1); the RMSNorm
    weight g is U(0.5, 1.5); projection weights are N(0, 0.02) except the tiny
    case, whose weights are N(0, 1/sqrt(512)); upstream gradient dY is N(0, 1).
  * Tensor number t of a workload is drawn from a generator seeded with
    seed*1000 + t, in the fixed order X, W1, R, g, W2, dY, H, W, labels.
  * Weights are stored in nn.Linear layout: W1t[d, K1], W2t[2F, d], Wt[V, d]
    (the contraction dimension is contiguous).
  * W2t rows [0, F) are the gate projection and rows [F, 2F) the up projection.
"""
from __future__ import annotations

import dataclasses
import math

import torch

# order in which tensors draw their seeds
_ORDER = {"X": 0, "W1": 1, "R": 2, "g": 3, "W2": 4, "dY": 5, "H": 6, "W": 7, "labels": 8, "W3": 9, "dYb": 10}


@dataclasses.dataclass(frozen=True)
class BlockShape:
    """One GEMM-Residual-PartialRMS-GEMM problem.

    M tokens, K1 input width of the first projection, d hidden width,
    N2 columns of the second projection (2F for SwiGLU, N for plain).
    """
    name: str
    M: int
    K1: int
    d: int
    N2: int
    swiglu: bool = True
    w_std: float = 0.02
    x_std: float = 1.0
    backward: bool = True
    eps: float = 1e-5

    @property
    def F(self) -> int:
        return self.N2 // 2 if self.swiglu else self.N2

    @property
    def out_cols(self) -> int:
        return self.F if self.swiglu else self.N2

    def fwd_flops(self) -> float:
        return 2.0 * self.M * self.d * self.K1 + 2.0 * self.M * self.N2 * self.d

    def fwdbwd_flops(self) -> float:
        # forward + data-gradient + weight-gradient GEMMs, recompute not counted
        return 3.0 * self.fwd_flops()


@dataclasses.dataclass(frozen=True)
class CEShape:
    """LM-head cross-entropy problem: H[M, d] times W[d, V], labels in [0, V)."""
    name: str
    M: int
    d: int
    V: int
    w_std: float = 0.02

    def gemm_flops(self) -> float:
        return 2.0 * self.M * self.d * self.V


TINY = BlockShape("tiny_fwd_plain", 256, 512, 512, 512, swiglu=False,
                  w_std=1.0 / math.sqrt(512.0), x_std=1.0 / math.sqrt(512.0),
                  backward=False)
B1 = BlockShape("1b_fwd", 8192, 2048, 2048, 16384, backward=False)
B7 = BlockShape("7b_fwdbwd", 8192, 4096, 4096, 28672)
B70 = BlockShape("70b_fwdbwd", 4096, 8192, 8192, 57344)
LMHEAD = CEShape("lmhead_ce", 8192, 2048, 128256)

BLOCK_SHAPES = {s.name: s for s in (TINY, B1, B7, B70)}


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _ORDER[name])
    return g


def normal_bf16(shape, std: float, seed: int, name: str, device="cpu") -> torch.Tensor:
    t = torch.randn(*shape, generator=_gen(seed, name, device), device=device,
                    dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def uniform_bf16(shape, lo: float, hi: float, seed: int, name: str, device="cpu") -> torch.Tensor:
    t = torch.rand(*shape, generator=_gen(seed, name, device), device=device,
                   dtype=torch.float32)
    t.mul_(hi - lo).add_(lo)
    return t.to(torch.bfloat16)


def block_inputs(s: BlockShape, seed: int = 0, device="cpu", with_dy=None) -> dict:
    """X[M,K1], W1t[d,K1], R[M,d], g[d], W2t[N2,d] (+ dY[M,out_cols]) as bf16."""
    x = {
        "X": normal_bf16((s.M, s.K1), s.x_std, seed, "X", device),
        "W1t": normal_bf16((s.d, s.K1), s.w_std, seed, "W1", device),
        "R": normal_bf16((s.M, s.d), 1.0, seed, "R", device),
        "g": uniform_bf16((s.d,), 0.5, 1.5, seed, "g", device),
        "W2t": normal_bf16((s.N2, s.d), s.w_std, seed, "W2", device),
    }
    if with_dy if with_dy is not None else s.backward:
        x["dY"] = normal_bf16((s.M, s.out_cols), 1.0, seed, "dY", device)
    return x


def down_proj_inputs(s: BlockShape, seed: int = 0, device="cpu") -> dict:
    """For a block whose SwiGLU output feeds a down projection y = out W3:
    W3t[d, F] ~ N(0, w_std) (nn.Linear layout) and the upstream gradient
    dYb[M, d] ~ N(0, 1)."""
    return {"W3t": normal_bf16((s.d, s.F), s.w_std, seed, "W3", device),
            "dYb": normal_bf16((s.M, s.d), 1.0, seed, "dYb", device)}


def ce_inputs(s: CEShape, seed: int = 0, device="cpu") -> dict:
    """H[M,d] ~ N(0,1), Wt[V,d] ~ N(0, w_std), labels[M] int32 uniform in [0,V)."""
    lab = torch.randint(0, s.V, (s.M,), generator=_gen(seed, "labels", device),
                        device=device, dtype=torch.int64).to(torch.int32)
    return {
        "H": normal_bf16((s.M, s.d), 1.0, seed, "H", device),
        "Wt": normal_bf16((s.V, s.d), s.w_std, seed, "W", device),
        "labels": lab,
    }


def to_f64(t: torch.Tensor):
    """Exact widening of a bf16/fp32 tensor to a numpy float64 array."""
    return t.detach().to("cpu", torch.float32).numpy().astype("float64")
