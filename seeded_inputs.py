"""Seeded synthetic inputs shared by the oracle side and the CUDA side of the tests and bench.

This module only draws numbers; it holds none of the chain's arithmetic. Every workload is a
synthetic GEMM chain (the CTA-Pipelining paper evaluates synthetic multi-layer GEMMs, section IV,
Fig. 3-5; no dataset is involved).

Recipe: one ``torch.Generator('cpu')`` seeded with ``seed`` draws, in the order X, W1, W2, ...,
each tensor as ``randn(float32) * std`` and then casts it to bfloat16 (round to nearest even).
A gated chain draws X, W_gate, W_up, W2, ... (gate and up share the first stage's std).
``N(0, 1/d)`` in a workload description means variance 1/d, i.e. ``std = 1/sqrt(d)``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMM chain: Y = stage_{S-1}( ... stage_0(X) ... ), stage_s(A) = epi(A @ W_s)."""

    name: str
    M: int
    dims: Tuple[int, ...]          # K, N1, N2, ... (num_gemms + 1 entries)
    x_std: float
    w_std: Tuple[float, ...]       # one per weight
    gelu: bool = False             # GeLU(tanh) on every GEMM's fp32 accumulator
    residual: bool = False         # add X to the last stage before rounding
    tile_m: int = 0                # 0: library default
    tile_n: int = 0
    description: str = ""
    gated: bool = False            # first stage from two weights: SiLU(X Wg) * (X Wu)

    @property
    def num_gemms(self) -> int:
        return len(self.dims) - 1

    @property
    def flops(self) -> int:
        f = sum(2 * self.M * self.dims[i] * self.dims[i + 1] for i in range(self.num_gemms))
        return f + (2 * self.M * self.dims[0] * self.dims[1] if self.gated else 0)

    @property
    def algorithmic_bytes(self) -> int:
        """X + every W + Y, plus each intermediate written once and read once (bf16)."""
        b = self.M * self.dims[0] * 2
        b += sum(self.dims[i] * self.dims[i + 1] * 2 for i in range(self.num_gemms))
        if self.gated:
            b += self.dims[0] * self.dims[1] * 2
        b += self.M * self.dims[-1] * 2
        b += sum(2 * self.M * d * 2 for d in self.dims[1:-1])
        if self.residual:
            b += self.M * self.dims[0] * 2
        return b


def _sq(d: int) -> float:
    return 1.0 / math.sqrt(d)


# The five synthetic chain workloads this library is exercised on.
WORKLOADS = {
    "tiny_m64_d256": Workload(
        "tiny_m64_d256", 64, (256, 256, 256), _sq(256), (_sq(256), _sq(256)),
        tile_m=64, tile_n=64,
        description="X[64x256], W1,W2[256x256], entries N(0,1)/sqrt(256); 64x64 tiles"),
    "decode_m128_d4096": Workload(
        "decode_m128_d4096", 128, (4096, 4096, 4096), 1.0, (_sq(4096), _sq(4096)),
        description="M=128, K=N1=N2=4096, X~N(0,1), W~N(0,1/4096)"),
    "prefill_m2048_d8192": Workload(
        "prefill_m2048_d8192", 2048, (8192, 8192, 8192), 1.0, (_sq(8192), _sq(8192)),
        description="M=2048, K=N1=N2=8192, X~N(0,1), W~N(0,1/8192)"),
    "llama_m256_4096_14336": Workload(
        "llama_m256_4096_14336", 256, (4096, 14336, 4096), 1.0, (_sq(4096), _sq(14336)),
        description="X[256x4096] W1[4096x14336] W2[14336x4096], W1~N(0,1/4096), W2~N(0,1/14336)"),
    "llama_swiglu_m256_4096_14336": Workload(
        "llama_swiglu_m256_4096_14336", 256, (4096, 14336, 4096), 1.0, (_sq(4096), _sq(14336)),
        gated=True,
        description="Llama-style gated MLP: X[256x4096], Wg,Wu[4096x14336]~N(0,1/4096), "
                    "H = SiLU(X Wg) * (X Wu), W2[14336x4096]~N(0,1/14336)"),
    "gelu4_m512_d8192": Workload(
        "gelu4_m512_d8192", 512, (8192,) * 5, 1.0, (_sq(8192),) * 4, gelu=True, residual=True,
        description="4 GEMMs d=8192, GeLU(tanh) after each, residual X at the end, M=512"),
}


def make_workload(name: str, M: int, dims: Sequence[int], x_std: float = 1.0,
                  w_std: Optional[Sequence[float]] = None, gelu: bool = False,
                  residual: bool = False, tile_m: int = 0, tile_n: int = 0, gated: bool = False) -> Workload:
    dims = tuple(int(d) for d in dims)
    if w_std is None:
        w_std = tuple(_sq(d) for d in dims[:-1])
    return Workload(name, int(M), dims, float(x_std), tuple(w_std), gelu, residual, tile_m, tile_n,
                    gated=gated)


def draw(w: Workload, seed: int = 0) -> Tuple[torch.Tensor, List[torch.Tensor]]:
    """X and the weights as CPU bfloat16 tensors, drawn in the order X, W1, W2, ..."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = (torch.randn(w.M, w.dims[0], generator=g, dtype=torch.float32) * w.x_std).to(torch.bfloat16)
    ws = []
    for i in ([0] if w.gated else []) + list(range(w.num_gemms)):
        t = torch.randn(w.dims[i], w.dims[i + 1], generator=g, dtype=torch.float32) * w.w_std[i]
        ws.append(t.to(torch.bfloat16))
    return x, ws


def draw_integer(M: int, dims: Sequence[int], seed: int = 0, values=(-1, 0, 1), gated: bool = False):
    """Integer-valued bf16 inputs: every entry drawn uniformly from ``values``.

    With small integers every partial sum is an integer; while the sums stay below 2**24 in
    magnitude, fp32 represents them exactly, so any summation order gives the same result.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    vals = torch.tensor(values, dtype=torch.float32)
    x = vals[torch.randint(0, len(values), (M, dims[0]), generator=g)].to(torch.bfloat16)
    ws = [vals[torch.randint(0, len(values), (dims[i], dims[i + 1]), generator=g)].to(torch.bfloat16)
          for i in ([0] if gated else []) + list(range(len(dims) - 1))]
    return x, ws


def permutation_matrix(n: int, seed: int = 0, scale: float = 1.0) -> Tuple[torch.Tensor, torch.Tensor]:
    """(P, perm) with P[k, perm[k]] = scale; so (A @ P)[:, perm[k]] = scale * A[:, k]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(n, generator=g)
    p = torch.zeros(n, n, dtype=torch.float32)
    p[torch.arange(n), perm] = scale
    return p.to(torch.bfloat16), perm


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> contiguous numpy uint16 array of its bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor (CPU)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def sample_rows(M: int, count: int = 64, seed: int = 0) -> np.ndarray:
    """First row, last row and seeded random rows in between, ascending and unique."""
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    if M > 2:
        rows.update(int(r) for r in rng.choice(np.arange(1, M - 1), size=min(count - 2, M - 2),
                                               replace=False))
    return np.array(sorted(rows), dtype=np.int64)
