"""Seeded synthetic inputs shared by the tests, the oracle checks and bench.py.

This module only draws random numbers; it holds none of the GEMM, schedule or
checksum arithmetic. Every matrix is drawn in fp32 on the CPU from a seeded
``torch.Generator`` and rounded (round-to-nearest-even) to the input dtype,
so the CUDA path and the oracle see identical bytes.

Workload recipes (the shapes and value laws of the GEMM workloads the
Stream-K and fault-tolerance pages evaluate on, restated as synthetic data):

* ``example_384``: 384x384x128 fp16, U[-1,1], seed 0 (the Stream-K page's
  worked example of Figs. 1-2), fp32 output.
* ``square_sweep``: m=n=k in {1024 ... 6144}, bf16, N(0,1)/sqrt(k) for A and
  B, seed 1 (the square range the fault-tolerance page averages over).
* ``hostile``: 128x128-tile shapes whose tile count quantises badly on the
  GPU, fp16, U[-1,1] for A, B and C0, seed 2, alpha=1.5, beta=0.5.
* ``random_sweep``: m, n, k log-uniform on [128, 8192], rounded up to a
  multiple of 128, seed 3 (the Stream-K page's test domain bounds, Fig. 4).
* ``mlp``: transformer-MLP shapes at 8192 tokens, bf16, activations A ~
  N(0,1), weights B ~ N(0, 0.02^2), seed 4.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Tuple

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@dataclass
class Problem:
    m: int
    n: int
    k: int
    A: torch.Tensor            # stored (m, k) row-major, or (k, m) when a_layout == 1
    B: torch.Tensor            # stored (n, k) "K-major", or (k, n) when b_layout == 1
    C0: Optional[torch.Tensor]  # (m, n) in the output dtype, or None
    alpha: float
    beta: float
    in_dtype: str
    out_dtype: str
    a_layout: int = 0
    b_layout: int = 0


def _draw(gen: torch.Generator, shape, law: str, scale: float) -> torch.Tensor:
    if law == "uniform":
        return (torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0) * scale
    if law == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * scale
    if law == "integer":       # small integers: every product and sum is exact in fp32
        return torch.randint(-3, 4, shape, generator=gen).to(torch.float32) * scale
    raise ValueError(law)


def make_problem(m: int, n: int, k: int, *, seed: int, in_dtype: str = "bf16",
                 out_dtype: str = "bf16", law_a: str = "uniform", law_b: str = "uniform",
                 scale_a: float = 1.0, scale_b: float = 1.0, alpha: float = 1.0,
                 beta: float = 0.0, law_c: str = "uniform", a_layout: int = 0,
                 b_layout: int = 0) -> Problem:
    """Draw A, then B, then (if beta != 0) C0 from one generator seeded `seed`."""
    gen = torch.Generator().manual_seed(seed)
    dt = DTYPES[in_dtype]
    A = _draw(gen, (m, k) if a_layout == 0 else (k, m), law_a, scale_a).to(dt)
    B = _draw(gen, (n, k) if b_layout == 0 else (k, n), law_b, scale_b).to(dt)
    C0 = None
    if beta != 0.0:
        C0 = _draw(gen, (m, n), law_c, 1.0).to(DTYPES[out_dtype])
    return Problem(m, n, k, A, B, C0, alpha, beta, in_dtype, out_dtype, a_layout, b_layout)


# ----------------------------------------------------------------------------
# Named workloads
# ----------------------------------------------------------------------------
def example_384() -> Problem:
    return make_problem(384, 384, 128, seed=0, in_dtype="f16", out_dtype="f32")


SQUARE_SIZES = (1024, 2048, 3072, 4096, 5120, 6144)


def square(size: int) -> Problem:
    s = 1.0 / math.sqrt(size)
    return make_problem(size, size, size, seed=1, in_dtype="bf16", out_dtype="bf16",
                        law_a="normal", law_b="normal", scale_a=s, scale_b=s)


HOSTILE_SHAPES = ((1664, 1664, 8192), (2560, 2432, 4096), (256, 256, 65536), (128, 19072, 2048))


def hostile(m: int, n: int, k: int) -> Problem:
    return make_problem(m, n, k, seed=2, in_dtype="f16", out_dtype="f16", alpha=1.5, beta=0.5)


def random_shapes(count: int = 1000, seed: int = 3, lo: int = 128, hi: int = 8192,
                  multiple: int = 128) -> List[Tuple[int, int, int]]:
    """m, n, k each log-uniform on [lo, hi], rounded up to a multiple."""
    gen = torch.Generator().manual_seed(seed)
    u = torch.rand((count, 3), generator=gen, dtype=torch.float64)
    v = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    out = []
    for row in v.tolist():
        out.append(tuple(int(math.ceil(x / multiple) * multiple) for x in row))
    return out


def random_problem(m: int, n: int, k: int, index: int) -> Problem:
    return make_problem(m, n, k, seed=3 * 1_000_003 + index, in_dtype="f16", out_dtype="f16")


MLP_SHAPES = ((8192, 28672, 8192), (8192, 8192, 28672), (8192, 1024, 8192))


def mlp(m: int, n: int, k: int) -> Problem:
    return make_problem(m, n, k, seed=4, in_dtype="bf16", out_dtype="bf16", law_a="normal",
                        law_b="normal", scale_a=1.0, scale_b=0.02)


def fault_plan(launches: int, seed: int = 4, every: int = 100):
    """Launch ids (one per block of `every` launches) that carry an injected
    bit flip, and a generator for the flip's tile/row/column/bit draws."""
    gen = torch.Generator().manual_seed(seed)
    ids = []
    for start in range(0, launches, every):
        span = min(every, launches - start)
        ids.append(start + int(torch.randint(0, span, (1,), generator=gen)))
    return ids, gen
