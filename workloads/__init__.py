"""Seeded synthetic inputs for the ragged_dot (MoE grouped GEMM) workloads.

This module only draws random numbers and builds group-size vectors with the
structure of the routed-expert workloads (top-k router counts, a Zipf-skewed
packed buffer, empty groups).  It holds none of the grouped-GEMM or GLU
arithmetic, so both the CPU oracle and the CUDA path can take their inputs
from here without sharing any of the method's code.

Notation: ``N(0, v)`` means a normal with variance ``v`` (standard deviation
``sqrt(v)``).  Small tensors come from ``numpy.random.default_rng(seed)``
(bit-reproducible on every machine); full-size tensors come from a seeded
``torch.Generator`` on the target device, which is fast and reproducible on a
given device and torch build.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "topk_counts",
    "zipf_sizes",
    "tiny_fwd",
    "mixtral_fwd",
    "packed_glu_fwd",
    "backward_pair",
    "decode_fwd",
    "expert_ffn",
    "normal_bf16",
    "normal_bf16_np",
    "random_sizes",
    "WORKLOADS",
]


@dataclasses.dataclass
class Workload:
    """Shapes, group sizes and the seed of one synthetic workload."""

    name: str
    m: int            # rows of the token buffer
    k: int            # hidden width of lhs / contraction of the forward
    n: int            # output width of rhs (before any GLU halving)
    g_total: int      # number of groups in group_sizes
    group_sizes: np.ndarray   # int32 [g_total]
    group_offset: int = 0
    g_local: Optional[int] = None
    limit: Optional[int] = None
    glu: bool = False
    lhs_var: float = 1.0
    rhs_var: float = 1.0
    seed: int = 0

    def __post_init__(self):
        if self.g_local is None:
            self.g_local = self.g_total


# --------------------------------------------------------------------------
# group-size structure
# --------------------------------------------------------------------------
def topk_counts(logits: np.ndarray, topk: int) -> np.ndarray:
    """Count how many rows pick each column among their ``topk`` largest logits.

    The counts are the group sizes of a token buffer sorted by expert after
    top-k routing (each token appears once per selected expert).
    """
    t, g = logits.shape
    picks = np.argpartition(-logits, topk - 1, axis=1)[:, :topk]
    return np.bincount(picks.ravel(), minlength=g).astype(np.int32)


def zipf_sizes(total: int, groups: int, s: float) -> np.ndarray:
    """Deterministic Zipf(s) apportionment of ``total`` rows over ``groups``.

    Group e gets a share proportional to (e+1)^-s; rounding uses the
    largest-remainder rule so the sizes sum exactly to ``total``.
    """
    w = np.arange(1, groups + 1, dtype=np.float64) ** (-s)
    quota = total * w / w.sum()
    base = np.floor(quota).astype(np.int64)
    rest = total - int(base.sum())
    order = np.argsort(-(quota - base), kind="stable")
    base[order[:rest]] += 1
    return base.astype(np.int32)


def random_sizes(rng: np.random.Generator, m: int, g: int, n_empty: int = 0) -> np.ndarray:
    """Multinomial split of ``m`` rows over ``g`` groups, ``n_empty`` forced to 0."""
    sizes = np.zeros(g, np.int32)
    empty = rng.choice(g, size=n_empty, replace=False) if n_empty else np.array([], np.int64)
    live = np.setdiff1d(np.arange(g), empty)
    if len(live):
        sizes[live] = rng.multinomial(m, np.full(len(live), 1.0 / len(live)))
    return sizes


# --------------------------------------------------------------------------
# tensors
# --------------------------------------------------------------------------
def normal_bf16_np(rng: np.random.Generator, shape, var: float = 1.0):
    """CPU bf16 torch tensor with N(0, var) entries drawn by numpy."""
    import torch

    x = rng.standard_normal(shape, dtype=np.float32)
    if var != 1.0:
        x *= np.float32(math.sqrt(var))
    return torch.from_numpy(x).to(torch.bfloat16)


def normal_bf16(shape, var: float, seed: int, device):
    """bf16 tensor with N(0, var) entries from a seeded torch generator on ``device``."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    chunk = 1 << 28
    std = math.sqrt(var)
    for lo in range(0, flat.numel(), chunk):
        hi = min(flat.numel(), lo + chunk)
        tmp = torch.randn(hi - lo, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[lo:hi].copy_(tmp)
        del tmp
    return out


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------
def tiny_fwd() -> Workload:
    """Tiny forward: lhs [256,128] N(0,1), rhs [4,128,256] N(0,1/128), one empty group."""
    rng = np.random.default_rng(1)
    g = 4
    empty = int(rng.integers(g))
    live = [i for i in range(g) if i != empty]
    sizes = np.zeros(g, np.int32)
    sizes[live] = rng.multinomial(256, np.full(3, 1.0 / 3))
    return Workload("tiny_fwd_256x128x256_g4", 256, 128, 256, g, sizes,
                    lhs_var=1.0, rhs_var=1.0 / 128, seed=1)


def mixtral_fwd() -> Workload:
    """Mixtral-shaped forward: 16384 tokens, top-2 of 8 experts, skewed router.

    Router logits N(0,1) [16384, 8] plus a per-expert bias N(0, 0.5); the
    top-2 counts are the group sizes of the 32768-row sorted buffer.
    """
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((16384, 8)) + rng.normal(0.0, math.sqrt(0.5), 8)
    sizes = topk_counts(logits, 2)
    return Workload("mixtral_fwd_32768x4096x14336_g8", 32768, 4096, 14336, 8, sizes,
                    lhs_var=1.0, rhs_var=1.0 / 4096, seed=2)


def packed_glu_fwd() -> Workload:
    """Packed expert buffer with a valid-row limit and a fused SiLU-GLU epilogue.

    225280-row buffer, 126156 valid rows split Zipf(1.1) over 64 experts;
    this shard owns experts 16..31 (group_offset 16, 16 local groups) with a
    fused [gate|up] rhs of width 2048.
    """
    sizes = zipf_sizes(126156, 64, 1.1)
    return Workload("packed_glu_225280x4096x2048_g64_local16", 225280, 4096, 2048, 64, sizes,
                    group_offset=16, g_local=16, limit=126156, glu=True,
                    lhs_var=1.0, rhs_var=1.0 / 4096, seed=3)


def backward_pair() -> Workload:
    """Backward pair: x [65536,4096], do [65536,1024], w [64,4096,1024], 8 empty groups."""
    rng = np.random.default_rng(4)
    sizes = random_sizes(rng, 65536, 64, n_empty=8)
    return Workload("backward_65536x4096x1024_g64", 65536, 4096, 1024, 64, sizes,
                    lhs_var=1.0, rhs_var=1.0 / 4096, seed=4)


def decode_fwd(skewed: bool = True) -> Workload:
    """Decode-shaped forward: 256 tokens, top-8 of 128 experts (2048 rows).

    The up projection is rhs [128,4096,1536] with the GLU epilogue; the down
    projection is rhs [128,768,4096].  ``skewed`` adds a per-expert router
    bias N(0,1), which gives many groups of 0-3 rows; without it the routing
    is uniform.
    """
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((256, 128))
    bias = rng.standard_normal(128)
    if skewed:
        logits = logits + bias
    sizes = topk_counts(logits, 8)
    tag = "skewed" if skewed else "uniform"
    return Workload(f"decode_{tag}_2048x4096x1536_g128", 2048, 4096, 1536, 128, sizes,
                    glu=True, lhs_var=1.0, rhs_var=1.0 / 4096, seed=5)


def expert_ffn(tokens: int) -> Workload:
    """Expert FFN forward at a batch of ``tokens`` tokens, top-8 of 128 experts.

    The same layer as ``decode_fwd`` (up rhs [128,4096,1536] with the GLU
    epilogue, down rhs [128,768,4096]) at larger batches, from weight-bound
    (a few hundred tokens) to compute-bound (tens of thousands): the router
    logits are N(0,1) plus a per-expert bias N(0,1), seeded by ``tokens``.
    """
    rng = np.random.default_rng(tokens)
    logits = rng.standard_normal((tokens, 128)) + rng.standard_normal(128)
    sizes = topk_counts(logits, 8)
    return Workload(f"expert_ffn_{tokens}tok_top8_g128", int(sizes.sum()), 4096, 1536, 128,
                    sizes, glu=True, lhs_var=1.0, rhs_var=1.0 / 4096, seed=tokens)


WORKLOADS = {
    "tiny": tiny_fwd,
    "mixtral": mixtral_fwd,
    "packed_glu": packed_glu_fwd,
    "backward": backward_pair,
    "decode": decode_fwd,
}
