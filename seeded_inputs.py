"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and names workload shapes.  It holds none of the
GEMM's or the convolution's arithmetic, and it imports neither the CUDA library nor the
oracle, so both sides can take their inputs from here without sharing anything else.

Recipe (the pages fix no generator; this is the reading used throughout):
  * one ``torch.Generator('cpu')`` seeded with the workload's seed; A is drawn first,
    then B (for the convolution: the input x first, then the weights);
  * "uniform[-1,1]": ``torch.rand(...) * 2 - 1`` in float32;
  * "normal(0,1) rounded to bf16": ``torch.randn(...)`` in float32, then rounded to
    nearest-even bf16 with ``.to(torch.bfloat16)``;
  * the integer-valued copy: ``torch.randint(-4, 5, ...)`` from a fresh generator on the
    same seed (A then B), converted to the input dtype (exact: |v| <= 4).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "gemm" or "conv4d"
    dtype: str           # "f32" or "bf16" (input dtype; C is always fp32)
    M: int
    N: int
    K: int
    seed: int
    dist: str            # "uniform" or "normal"
    conv: dict = field(default_factory=dict)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five configurations: a small parity case, the two headline GEMMs, a skinny
# memory-bound GEMM and a 4-D convolution lowered to a GEMM by im2col.
WORKLOADS = {
    "f32_256": Workload("f32_256", "gemm", "f32", 256, 256, 256, 0, "uniform"),
    "f32_4096": Workload("f32_4096", "gemm", "f32", 4096, 4096, 4096, 1, "uniform"),
    "bf16_8192": Workload("bf16_8192", "gemm", "bf16", 8192, 8192, 8192, 2, "normal"),
    "f32_skinny": Workload("f32_skinny", "gemm", "f32", 16, 16384, 16384, 3, "uniform"),
    "conv4d": Workload("conv4d", "conv4d", "f32", 32, 12 ** 4, 16 * 5 ** 4, 4, "uniform",
                       conv=dict(cin=16, cout=32, ins=(16, 16, 16, 16), ks=(5, 5, 5, 5))),
}


def generator(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def uniform(shape, g: torch.Generator) -> torch.Tensor:
    return torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1


def normal_bf16(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def ints(shape, g: torch.Generator, lo: int = -4, hi: int = 4) -> torch.Tensor:
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int32)


TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _cast(t: torch.Tensor, dtype: str) -> torch.Tensor:
    """Round to the input dtype (nearest-even for bf16/f16)."""
    return t.to(TORCH_DTYPES[dtype])


def gemm_operands(M: int, N: int, K: int, seed: int, dist: str = "uniform", dtype: str = "f32"):
    """(A [M,K], B [K,N]) on the CPU, drawn A first then B from one generator."""
    g = generator(seed)
    if dist == "uniform":
        A, B = uniform((M, K), g), uniform((K, N), g)
    elif dist == "normal":
        A = torch.randn((M, K), generator=g, dtype=torch.float32)
        B = torch.randn((K, N), generator=g, dtype=torch.float32)
    elif dist == "ints":
        A, B = ints((M, K), g).float(), ints((K, N), g).float()
    else:
        raise ValueError(dist)
    return _cast(A, dtype), _cast(B, dtype)


def integer_copy(M: int, N: int, K: int, seed: int, dtype: str = "f32"):
    """Integer-valued operands in [-4, 4] from a fresh generator on ``seed``."""
    return gemm_operands(M, N, K, seed, "ints", dtype)


def workload_operands(w: Workload):
    """CPU tensors of a workload: (A, B) for a GEMM, (x, weights) for the convolution."""
    if w.kind == "gemm":
        return gemm_operands(w.M, w.N, w.K, w.seed, w.dist, w.dtype)
    c = w.conv
    g = generator(w.seed)
    x = uniform((c["cin"],) + tuple(c["ins"]), g)
    wt = uniform((c["cout"], c["cin"]) + tuple(c["ks"]), g)
    return x, wt


def channel_last(x: torch.Tensor, wt: torch.Tensor, dtype: str = "bf16"):
    """The convolution's operands in channel-last order, rounded to a 16-bit dtype:
    x [C_in, I0..I3] -> [I0..I3, C_in] and w [C_out, C_in, R0..R3] -> [C_out, R0..R3, C_in]
    (a copy of the same values; nothing else changes)."""
    return (_cast(x.permute(1, 2, 3, 4, 0).contiguous(), dtype),
            _cast(wt.permute(0, 2, 3, 4, 5, 1).contiguous(), dtype))


def sample_indices(M: int, N: int, seed: int, n_rows: int = 128, n_cols: int = 128, n_rand: int = 65536):
    """Deterministic sample of output positions: full rows, full columns, random entries."""
    g = generator(seed)
    rows = torch.randperm(M, generator=g)[: min(n_rows, M)].sort().values
    cols = torch.randperm(N, generator=g)[: min(n_cols, N)].sort().values
    ri = torch.randint(0, M, (n_rand,), generator=g)
    rj = torch.randint(0, N, (n_rand,), generator=g)
    return rows, cols, ri, rj


def sha256(*tensors: torch.Tensor) -> str:
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()
