"""Seeded synthetic inputs shared by the oracle side and the CUDA side of the tests and the bench.

This module only draws random numbers with the distributions of the workloads; it holds none of
the quantization, packing or GEMM arithmetic. Every array it returns is an *input*: float32 weights
before quantization, float32 or bf16 activations, top-k expert ids and router logits.

Workloads (shapes of a Kimi-K2-class MoE decoder, the model the pages build the engine for):

  tiny     M=1,  K=256,   N=512                   x ~ N(0,1), W ~ N(0, 0.02)
  swiglu   M in {1,4,16}, K=7168, N=2*18432       gate and up columns side by side
  down     M in {1,4,16}, K=18432, N=7168         x ~ 0.1 N(0,1); 1 % of W entries x10 (outliers)
  moe      T=64 tokens, E=384 experts, top-8 without replacement, router logits ~ N(0,1);
           per expert gate/up W [7168, 2*2048] and down W [2048, 7168]
  prefill  M=4096, K=7168, N=18432, x bf16 ~ N(0,1)

Two generator families draw the same distributions: numpy ``default_rng`` (host, small and
medium sizes) and ``torch.Generator`` on a CUDA device (full-size weights, which would take
minutes to draw on the host). They produce different streams; a test uses one family for both
the oracle and the CUDA path.
"""
from __future__ import annotations

import numpy as np

W_STD = 0.02          # weight standard deviation
OUTLIER_P = 0.01      # probability that a weight is an outlier (down projection workload)
OUTLIER_MUL = 10.0    # outlier magnification
DOWN_X_STD = 0.1      # activation scale for the down projection workload

# workload shapes
TINY = dict(M=1, K=256, N=512)
SWIGLU = dict(K=7168, I=18432)            # N = 2 * I
DOWN = dict(K=18432, N=7168)
MOE = dict(T=64, E=384, topk=8, K=7168, I=2048)
PREFILL = dict(M=4096, K=7168, N=18432)


def _rng(seed: int, stream: int) -> np.random.Generator:
    """Independent numpy stream per (seed, tensor id)."""
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream)]))


# ----------------------------------------------------------------------------- host (numpy)

def normal(shape, std=1.0, seed=0, stream=0) -> np.ndarray:
    """float32 N(0, std^2) array."""
    a = _rng(seed, stream).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def weights(K: int, N: int, seed=0, stream=1, outliers=False) -> np.ndarray:
    """float32 [K, N] weights ~ N(0, 0.02^2); with ``outliers`` each entry independently
    (probability 1 %) is multiplied by 10."""
    W = normal((K, N), W_STD, seed, stream)
    if outliers:
        mask = _rng(seed, stream + 1000).random((K, N), dtype=np.float32) < OUTLIER_P
        W[mask] *= np.float32(OUTLIER_MUL)
    return W


def activations(M: int, K: int, seed=0, stream=2, std=1.0) -> np.ndarray:
    """float32 [M, K] activations ~ N(0, std^2)."""
    return normal((M, K), std, seed, stream)


def packed_codes(K: int, N: int, seed=0, stream=6) -> np.ndarray:
    """int32 [K/8, N] words of uniformly random bits: every packed 4-bit code uniform in 0..15."""
    words = _rng(seed, stream).integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64)
    return words.astype(np.uint32).view(np.int32)


def group_scales(K: int, N: int, seed=0, stream=7, lo=0.002, hi=0.006) -> np.ndarray:
    """float32 [K/32, N] positive scales drawn uniformly from [lo, hi)."""
    return _rng(seed, stream).uniform(lo, hi, size=(K // 32, N)).astype(np.float32)


def bf16_activations(M: int, K: int, seed=0, stream=3) -> np.ndarray:
    """bf16 activations ~ N(0,1), returned as their uint16 bit patterns [M, K].

    The float32 draw is cut to bf16 with round-to-nearest-even by a torch CPU cast (a library
    conversion); the bit patterns are then the input both sides consume."""
    import torch
    x = torch.from_numpy(normal((M, K), 1.0, seed, stream))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def routing(T: int, E: int, topk: int, seed=0, stream=4):
    """Top-k routing lists: for each token ``topk`` distinct experts drawn uniformly without
    replacement, and ``topk`` router logits ~ N(0,1).  Returns (topk_ids int32 [T,topk],
    logits float32 [T,topk])."""
    rng = _rng(seed, stream)
    ids = np.stack([rng.choice(E, size=topk, replace=False) for _ in range(T)]).astype(np.int32)
    logits = rng.standard_normal((T, topk), dtype=np.float32)
    return ids, logits


def moe_expert_weights(e: int, K: int, I: int, seed=0):
    """Host draw of one expert's float32 gate/up [K, 2I] and down [I, K] weights."""
    gu = normal((K, 2 * I), W_STD, seed, 10_000 + 2 * e)
    dn = normal((I, K), W_STD, seed, 10_001 + 2 * e)
    return gu, dn


# ----------------------------------------------------------------------------- device (torch)

def _tgen(seed: int, stream: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(stream))
    return g


def cuda_normal(shape, std=1.0, seed=0, stream=0, device="cuda"):
    """float32 N(0, std^2) tensor drawn on the device."""
    import torch
    t = torch.randn(shape, generator=_tgen(seed, stream, device), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def cuda_weights(K: int, N: int, seed=0, stream=1, outliers=False, device="cuda"):
    """Device draw of float32 [K, N] weights, same distribution as :func:`weights`."""
    import torch
    W = cuda_normal((K, N), W_STD, seed, stream, device)
    if outliers:
        u = torch.rand((K, N), generator=_tgen(seed, stream + 1000, device), device=device)
        W[u < OUTLIER_P] *= OUTLIER_MUL
        del u
    return W


def cuda_moe_expert_weights(e: int, K: int, I: int, seed=0, device="cuda"):
    """Device draw of one expert's float32 gate/up [K, 2I] and down [I, K] weights.

    Each expert has its own generator stream, so any expert can be redrawn on its own."""
    gu = cuda_normal((K, 2 * I), W_STD, seed, 10_000 + 2 * e, device)
    dn = cuda_normal((I, K), W_STD, seed, 10_001 + 2 * e, device)
    return gu, dn


def cuda_bf16_activations(M: int, K: int, seed=0, stream=3, device="cuda"):
    """bf16 [M, K] activations ~ N(0,1) drawn on the device."""
    import torch
    return cuda_normal((M, K), 1.0, seed, stream, device).to(torch.bfloat16)
