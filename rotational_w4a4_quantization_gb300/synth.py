"""Seeded synthetic inputs shared by the CUDA-path tests, the oracle tests and the bench.

This module draws numbers only: it holds none of the rotation, quantization or
GEMM arithmetic, so both sides can use it without sharing any of the method.

Recipe (the outlier model of the pages: a small, fixed set of hidden channels,
under 0.1% of them, up to 100x the typical magnitude, in the same channels for
every token; "Rotational Quantization ..." §The Activation Outlier Bottleneck in
Low-Bit Serving):

* values are drawn in fp64 from a ``torch.Generator`` on the CPU, then cast
  (round-to-nearest-even) to the stated dtype; the CUDA path and the oracle read
  the same cast tensor;
* outlier channels are distinct, drawn with ``randperm`` from the same
  generator, and multiplied by the stated factor in every row;
* weights are drawn directly in the transposed, output-channel-major layout
  W^T (N x K), which is the layout the offline fold reads.
"""
from __future__ import annotations

import dataclasses

import torch

SIGN_SEED = 0x5EED


@dataclasses.dataclass(frozen=True)
class Workload:
    """One shape set of the hot path (activation rotation+quant, GEMM, KV)."""
    name: str
    rows: int = 0            # tokens of the activation X
    n: int = 0               # hidden size = GEMM K = Hadamard size
    x_dtype: torch.dtype = torch.bfloat16
    n_outliers: int = 0      # outlier channels in X
    outlier_factor: float = 1.0
    gemm_n: int = 0          # GEMM output channels
    w_std: float = 0.02
    kv_tokens: int = 0
    kv_heads: int = 0
    kv_head_dim: int = 0
    kv_outliers_per_head: int = 0
    kv_outlier_factor: float = 1.0
    data_seed: int = 0

    @property
    def weight_seed(self) -> int:
        return 100 + self.data_seed


def _n_outliers(n: int) -> int:
    """0.1% of the channels, rounded, at least one."""
    return max(1, round(0.001 * n))


TINY = Workload("tiny", rows=64, n=1024, x_dtype=torch.float32, n_outliers=4,
                outlier_factor=50.0, gemm_n=1024, data_seed=1)
DECODE = Workload("decode", rows=16, n=4096, n_outliers=_n_outliers(4096),
                  outlier_factor=100.0, gemm_n=4096, data_seed=2)
PREFILL = Workload("prefill", rows=2048, n=4096, n_outliers=_n_outliers(4096),
                   outlier_factor=100.0, gemm_n=14336, data_seed=3)
KV = Workload("kv", kv_tokens=8192, kv_heads=32, kv_head_dim=128, kv_outliers_per_head=2,
              kv_outlier_factor=30.0, data_seed=4)
LARGE = Workload("large", rows=4096, n=8192, n_outliers=_n_outliers(8192),
                 outlier_factor=100.0, gemm_n=28672, data_seed=5)

WORKLOADS = {w.name: w for w in (TINY, DECODE, PREFILL, KV, LARGE)}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def outlier_channels(n: int, count: int, seed: int) -> torch.Tensor:
    g = generator(seed * 7919 + 17)
    return torch.randperm(n, generator=g)[:count].sort().values


def activations(rows: int, n: int, dtype: torch.dtype, seed: int, n_outliers: int = 0,
                factor: float = 1.0) -> torch.Tensor:
    """X (rows x n): N(0,1) with `n_outliers` fixed channels scaled by `factor`."""
    g = generator(seed)
    x = torch.randn(rows, n, dtype=torch.float64, generator=g)
    if n_outliers:
        ch = outlier_channels(n, n_outliers, seed)
        x[:, ch] *= factor
    return x.to(dtype)


def weights_t(n_out: int, k: int, seed: int, std: float = 0.02,
              dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """W^T (n_out x k): N(0, std^2), one output channel per row."""
    g = generator(seed)
    w = torch.randn(n_out, k, dtype=torch.float64, generator=g)
    w *= std
    return w.to(dtype)


def kv_pair(tokens: int, heads: int, head_dim: int, seed: int, outliers_per_head: int = 0,
            factor: float = 1.0, dtype: torch.dtype = torch.bfloat16):
    """K and V ([tokens][heads][head_dim]), N(0,1), each head with its own fixed
    outlier dimensions (chosen separately for K and V) scaled by `factor`."""
    out = []
    for which in range(2):
        g = generator(seed * 2 + which)
        t = torch.randn(tokens, heads, head_dim, dtype=torch.float64, generator=g)
        if outliers_per_head:
            for h in range(heads):
                dims = outlier_channels(head_dim, outliers_per_head, seed * 1000 + which * 100 + h)
                t[:, h, dims] *= factor
        out.append(t.to(dtype))
    return out[0], out[1]


def random_codes(rows: int, k: int, seed: int):
    """Uniform random packed INT4 operands: (rows x k/2 uint8 bytes, rows fp32
    positive scales).  Every byte value is equally likely, so every 4-bit code,
    -8 included, appears."""
    g = generator(seed)
    q = torch.randint(0, 256, (rows, k // 2), dtype=torch.int32, generator=g).to(torch.uint8)
    s = (torch.rand(rows, dtype=torch.float64, generator=g) * 0.99 + 0.01).to(torch.float32)
    return q, s


def extreme_codes(rows: int, k: int, byte: int):
    """Every byte equal to `byte` (e.g. 0x77 = all +7, 0x88 = all -8)."""
    return torch.full((rows, k // 2), byte, dtype=torch.uint8)
