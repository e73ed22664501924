"""Seeded synthetic inputs for the MoE routed-expert workloads.

This module is the only code shared by the tests, the oracle checks and the
benchmark.  It draws random numbers and group sizes and holds none of the
quantization or GEMM arithmetic.

Every workload is synthetic: the pages measure on Llama4 Scout training runs
(C4 / FineWeb data, trained checkpoints), which are not available, so tensors
of those shapes with the value distributions below stand in for them.

Workloads (all bf16, tokens sorted by expert, ``offs`` = cumulative end rows):

* ``tiny``      G=2, A[256,256]~N(0,1), offs [128,256], W[2,128,256]~N(0,0.02).
* ``scout``     Llama4-Scout-like routed experts: G=8, K=5120, N=8192,
                M=16384; group sizes 32 * Multinomial(512, p_i ~ i^-1.1) over a
                seeded permutation of the experts (empty groups possible);
                A~N(0,1), W~N(0,0.02), dOut~N(0,1e-3).
* ``swiglu``    SwiGLU expert: G=2, M=65600 split 39360/26240 (60/40 in
                32-row chunks), gate/up W[2,8192,5120], down W[2,5120,8192],
                x~N(0,1), W~N(0,0.02), dY~N(0,1e-3).
* ``imbalanced`` G=16, K=7168, N=2048, M=32768; group 1 holds 13120 tokens,
                groups 0, 7, 15 are empty, the other 19648 tokens go to the
                remaining 12 groups by Zipf(1.1) in 32-token chunks;
                A~N(0,1) with 1% of elements scaled by 100, W~N(0,0.02).
* ``sweep``     quantization bandwidth sweep: [M,K] for M in
                {8192..131072} x K in {5120, 8192}, values N(0,1) * 10^U(-4,4)
                per row; 3D weights [16,8192,5120].
"""
from __future__ import annotations

import numpy as np
import torch

SWEEP_M = (8192, 16384, 32768, 65536, 131072)
SWEEP_K = (5120, 8192)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def offsets_from_sizes(sizes) -> torch.Tensor:
    """Cumulative end offsets (int32) from group sizes."""
    return torch.tensor(np.cumsum(np.asarray(sizes, dtype=np.int64)), dtype=torch.int32)


def zipf_chunk_sizes(total: int, G: int, s: float, seed: int, chunk: int = 32) -> list[int]:
    """Sizes of G groups summing to ``total`` (a multiple of ``chunk``): the
    total/chunk chunks are drawn multinomially with p_i ~ i^-s, then the experts
    are permuted (seeded).  Zero-sized groups are possible."""
    assert total % chunk == 0
    rng = np.random.default_rng(seed)
    p = np.arange(1, G + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    counts = rng.multinomial(total // chunk, p)
    counts = counts[rng.permutation(G)]
    return [int(c) * chunk for c in counts]


def scout_group_sizes(seed: int = 0, M: int = 16384, G: int = 8) -> list[int]:
    return zipf_chunk_sizes(M, G, 1.1, seed)


def imbalanced_group_sizes(seed: int = 0) -> list[int]:
    G, M = 16, 32768
    sizes = [0] * G
    sizes[1] = 13120
    rest = [g for g in range(G) if g not in (0, 1, 7, 15)]
    # Zipf over the 12 remaining groups, no permutation (keeps 0/7/15 empty).
    rng = np.random.default_rng(seed)
    p = np.arange(1, len(rest) + 1, dtype=np.float64) ** (-1.1)
    p /= p.sum()
    counts = rng.multinomial((M - 13120) // 32, p)
    for g, c in zip(rest, counts):
        sizes[g] = int(c) * 32
    assert sum(sizes) == M
    return sizes


def swiglu_group_sizes() -> list[int]:
    return [39360, 26240]


def outlier_activations(shape, seed: int, frac: float = 0.01, factor: float = 100.0, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    mask = torch.rand(shape, generator=g, device=device) < frac
    x = torch.where(mask, x * factor, x)
    return x.to(torch.bfloat16)


def log_uniform_rows(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """N(0,1) * 10^U(-4,4), one magnitude per row."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    mag = torch.pow(10.0, torch.rand((M, 1), generator=g, device=device) * 8.0 - 4.0)
    return (x * mag).to(torch.bfloat16)


def workload(name: str, seed: int = 0, device="cpu") -> dict:
    """Inputs of one workload as tensors on ``device`` (CPU by default)."""
    if name == "tiny":
        sizes = [128, 128]
        M, N, K, G = 256, 128, 256, 2
        return dict(name=name, G=G, M=M, N=N, K=K, sizes=sizes, offs=offsets_from_sizes(sizes),
                    A=randn_bf16((M, K), 1.0, seed + 1, device), W=randn_bf16((G, N, K), 0.02, seed + 2, device),
                    dOut=randn_bf16((M, N), 1e-3, seed + 3, device))
    if name == "scout":
        G, M, N, K = 8, 16384, 8192, 5120
        sizes = scout_group_sizes(seed, M, G)
        return dict(name=name, G=G, M=M, N=N, K=K, sizes=sizes, offs=offsets_from_sizes(sizes),
                    A=randn_bf16((M, K), 1.0, seed + 1, device), W=randn_bf16((G, N, K), 0.02, seed + 2, device),
                    dOut=randn_bf16((M, N), 1e-3, seed + 3, device))
    if name == "imbalanced":
        G, M, N, K = 16, 32768, 2048, 7168
        sizes = imbalanced_group_sizes(seed)
        return dict(name=name, G=G, M=M, N=N, K=K, sizes=sizes, offs=offsets_from_sizes(sizes),
                    A=outlier_activations((M, K), seed + 1, device=device),
                    W=randn_bf16((G, N, K), 0.02, seed + 2, device),
                    dOut=randn_bf16((M, N), 1e-3, seed + 3, device))
    if name == "swiglu":
        G, M, D, H = 2, 65600, 5120, 8192
        sizes = swiglu_group_sizes()
        return dict(name=name, G=G, M=M, D=D, H=H, sizes=sizes, offs=offsets_from_sizes(sizes),
                    x=randn_bf16((M, D), 1.0, seed + 1, device),
                    Wg=randn_bf16((G, H, D), 0.02, seed + 2, device),
                    Wu=randn_bf16((G, H, D), 0.02, seed + 3, device),
                    Wd=randn_bf16((G, D, H), 0.02, seed + 4, device),
                    dY=randn_bf16((M, D), 1e-3, seed + 5, device))
    raise KeyError(name)
