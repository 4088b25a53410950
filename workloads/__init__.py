"""Seeded synthetic inputs for the W4A16 matmul and the Q4 block-32 GEMV.

This module only draws random numbers and names shapes. It holds none of the
quantization or matmul arithmetic, so both the CUDA path's tests and the CPU
oracle's tests can take their inputs from it without sharing method code.

Recipe (the same for every consumer):
  * weights: fp32 [N, K] drawn from N(0, 0.02^2) with a CPU ``torch.Generator``
    seeded with ``seed``;
  * optional outliers: exactly ``round(frac * N * K)`` positions chosen without
    replacement (``torch.randperm`` on the same generator, after the normal
    draw) are multiplied by ``mult``;
  * activations: fp32 N(0, 1) from a second generator seeded with
    ``seed + X_SEED_OFFSET``, then cast to BF16 (or FP16) with PyTorch's
    round-to-nearest-even conversion.

Shapes follow the pages' workloads: a tiny correctness case, the Llama-3-8B MLP
up-projection (4096 -> 14336), a 16384 x 16384 Q4 matrix, the M = 1..4096 batch
sweep on the Llama shape with 0.1 % outliers x10, and the 196 linear layers of a
Qwen2.5-1.5B-shaped decoder (28 blocks x {q, k, v, o, gate, up, down}).
"""
from __future__ import annotations

import torch

X_SEED_OFFSET = 1_000_003
WEIGHT_STD = 0.02

TINY = dict(name="tiny_m1_n256_k512_g128", M=1, N=256, K=512, group=128)
LLAMA_UP = dict(name="llama3_8b_up_proj_m1_n14336_k4096_g128", M=1, N=14336, K=4096, group=128)
Q4_SQUARE = dict(name="q4b32_gemv_n16384_k16384", N=16384, K=16384)
BATCH_SWEEP = dict(name="llama3_8b_up_proj_batch_sweep_n14336_k4096_g128", N=14336, K=4096, group=128,
                   Ms=(1, 2, 4, 8, 16, 32, 64, 128, 256, 1024, 4096), outlier_frac=0.001,
                   outlier_mult=10.0)
# (name, N = out_features, K = in_features) for one decoder block
QWEN_BLOCK = (("q", 1536, 1536), ("k", 256, 1536), ("v", 256, 1536), ("o", 1536, 1536),
              ("gate", 8960, 1536), ("up", 8960, 1536), ("down", 1536, 8960))
QWEN_STACK = dict(name="qwen2_5_1_5b_decode_stack_m1_28x7_g128", layers=28, block=QWEN_BLOCK,
                  group=128)


def weights(N: int, K: int, seed: int = 0, std: float = WEIGHT_STD, outlier_frac: float = 0.0,
            outlier_mult: float = 10.0) -> torch.Tensor:
    """fp32 [N, K] (CPU) ~ N(0, std^2), optionally with round(frac*N*K) outliers x mult."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    w = torch.randn(N, K, generator=g, dtype=torch.float32) * std
    n_out = int(round(outlier_frac * N * K))
    if n_out > 0:
        idx = torch.randperm(N * K, generator=g)[:n_out]
        flat = w.view(-1)
        flat[idx] = flat[idx] * outlier_mult
    return w


def activations_bf16(M: int, K: int, seed: int = 0) -> torch.Tensor:
    """BF16 [M, K] (CPU) ~ N(0, 1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + X_SEED_OFFSET)
    return torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)


def activations_fp16(K: int, seed: int = 0) -> torch.Tensor:
    """FP16 [K] (CPU) ~ N(0, 1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + X_SEED_OFFSET)
    return torch.randn(K, generator=g, dtype=torch.float32).to(torch.float16)


def bits16(t: torch.Tensor):
    """The uint16 bit patterns of a BF16/FP16 CPU tensor, as a numpy array."""
    import numpy as np

    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_indices(n: int, count: int, seed: int = 0) -> torch.Tensor:
    """``count`` distinct sorted indices in [0, n) (always including 0 and n-1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7)
    count = min(count, n)
    idx = torch.randperm(n, generator=g)[:count]
    idx = torch.cat([idx, torch.tensor([0, n - 1])]).unique(sorted=True)
    return idx
