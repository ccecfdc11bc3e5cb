"""Seeded synthetic inputs for the fused GEMM + reduce-scatter.

This module only draws random numbers and holds the workload recipes.  It
contains none of the method's arithmetic.  The tests, the benchmark, the
oracle checks and the CUDA path all take their inputs from here, so both
sides see the same bytes.

Recipe (every workload is synthetic; the pages use no dataset):
  * Values are drawn in fp32 on the CPU with ``torch.Generator().manual_seed``:
    seed 1 for A, 2 for B, 3 for C.  They are then rounded to bf16 with
    round-to-nearest-even (``Tensor.to(torch.bfloat16)``).
  * "uniform" draws U(-1, 1).  "normal" draws N(0, 0.02), reading 0.02 as the
    standard deviation.  "normal1" draws N(0, 1) (the bias-like C).  "int"
    draws integers in {-2, ..., 2}, for runs whose sums are exact in fp32.
  * A has shape [W, M, K/W]: rank r's K-shard of the activations.  B has shape
    [W, K/W, N]: rank r's K-shard of the row-parallel weight.  C has shape
    [M, N].
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    W: int
    M: int
    N: int
    Kpr: int
    a_dist: str
    b_dist: str
    alpha: float
    beta: float
    c_dist: str | None
    y_dtype: str  # "bf16" or "fp32"
    calls: int = 1

    @property
    def K(self) -> int:
        return self.W * self.Kpr

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads of the fused GEMM+RS path.  The FFN widths are
# 14336/8 = 1792, 28672/8 = 3584 and 13824/4 = 3456 per rank.
WORKLOADS = {
    "tiny_w2": Workload("tiny_w2", 2, 256, 256, 256, "uniform", "uniform",
                        1.0, 0.0, None, "fp32"),
    "ffn_w8_m4096": Workload("ffn_w8_m4096", 8, 4096, 4096, 1792, "normal", "normal",
                             1.0, 0.0, None, "bf16"),
    "ffn_w8_m8192_bias": Workload("ffn_w8_m8192_bias", 8, 8192, 8192, 3584, "normal",
                                  "normal", 0.5, 1.0, "normal1", "bf16"),
    "decode_w8_m64": Workload("decode_w8_m64", 8, 64, 8192, 3584, "normal", "normal",
                              1.0, 0.0, None, "bf16"),
    "ffn_w4_m16384_x20": Workload("ffn_w4_m16384_x20", 4, 16384, 5120, 3456, "uniform",
                                  "normal", 1.0, 0.0, None, "fp32", calls=20),
}
WORKLOAD_ORDER = ["tiny_w2", "ffn_w8_m4096", "ffn_w8_m8192_bias", "decode_w8_m64",
                  "ffn_w4_m16384_x20"]


def _draw(shape, dist: str, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    if dist == "uniform":
        x = torch.empty(shape, dtype=torch.float32).uniform_(-1.0, 1.0, generator=g)
    elif dist == "normal":
        x = torch.empty(shape, dtype=torch.float32).normal_(0.0, 0.02, generator=g)
    elif dist == "normal1":
        x = torch.empty(shape, dtype=torch.float32).normal_(0.0, 1.0, generator=g)
    elif dist == "int":
        x = torch.randint(-2, 3, shape, generator=g).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(torch.bfloat16)


def make_inputs(W: int, M: int, N: int, Kpr: int, a_dist: str = "normal",
                b_dist: str = "normal", c_dist: str | None = None,
                seeds=(1, 2, 3)):
    """CPU bf16 tensors A [W, M, Kpr], B [W, Kpr, N] and C [M, N] (or None)."""
    A = _draw((W, M, Kpr), a_dist, seeds[0])
    B = _draw((W, Kpr, N), b_dist, seeds[1])
    C = None if c_dist is None else _draw((M, N), c_dist, seeds[2])
    return A, B, C


def workload_inputs(w: Workload, exact: bool = False, seeds=(1, 2, 3)):
    """Inputs of a named workload.  With exact=True, every value is an integer
    in {-2..2}: every sum is then exact in fp32, so the result is unique."""
    if exact:
        return make_inputs(w.W, w.M, w.N, w.Kpr, "int", "int",
                           None if w.c_dist is None else "int", seeds)
    return make_inputs(w.W, w.M, w.N, w.Kpr, w.a_dist, w.b_dist, w.c_dist, seeds)


@dataclass(frozen=True)
class AgWorkload:
    """An AG+GEMM workload: H_r = alpha * X @ B1_r, X [M, K], B1 [W, K, N]."""
    name: str
    W: int
    M: int
    N: int  # columns per rank
    K: int
    x_dist: str
    b_dist: str
    alpha: float
    y_dtype: str

    @property
    def flops(self) -> int:
        return 2 * self.W * self.M * self.N * self.K


# The FFN's first GEMM in front of the 4096x4096 W=8 GEMM+RS workload: hidden
# 4096, FFN width 14336 = 8 x 1792 (its output H_r is that workload's A_r).
AG_WORKLOADS = {
    "ag_ffn_w8_m4096": AgWorkload("ag_ffn_w8_m4096", 8, 4096, 1792, 4096, "normal", "normal",
                                  1.0, "bf16"),
}


def make_ag_inputs(W: int, M: int, N: int, K: int, x_dist: str = "normal", b_dist: str = "normal",
                   seeds=(11, 12)):
    """CPU bf16 tensors X [M, K] and B1 [W, K, N]."""
    return _draw((M, K), x_dist, seeds[0]), _draw((W, K, N), b_dist, seeds[1])


def bf16_bits(t: torch.Tensor):
    """The raw bit patterns of a CPU bf16 tensor as a numpy uint16 array."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(M: int, W: int, BM: int = 128, n_random: int = 64, seed: int = 7,
                n_boundaries: int | None = None):
    """A row sample for full-size checks: the first and last row of every
    chunk, row-tile boundary rows (the first row of a tile and the row before
    it; all boundaries, or n_boundaries evenly spaced ones), and n_random
    seeded random rows.  Returned sorted and unique."""
    R = M // W
    rows = set()
    for c in range(W):
        rows.add(c * R)
        rows.add(c * R + R - 1)
    bounds = list(range(BM, M, BM))
    if n_boundaries is not None and len(bounds) > n_boundaries:
        step = len(bounds) / n_boundaries
        bounds = [bounds[int(i * step)] for i in range(n_boundaries)]
    for b in bounds:
        rows.add(b)
        rows.add(b - 1)
    g = torch.Generator().manual_seed(seed)
    if M > 0 and n_random > 0:
        for v in torch.randint(0, M, (n_random,), generator=g).tolist():
            rows.add(int(v))
    return sorted(r for r in rows if 0 <= r < M)
