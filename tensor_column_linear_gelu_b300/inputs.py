"""Seeded synthetic inputs for the tensor-parallel linear path.

This module is shared by the tests, the benchmark and the oracle's callers.
It draws random numbers and rounds them to the storage dtype; it holds none of
the method's arithmetic (no products, no activations, no sharding).

Recipe
------
* Every tensor has its own generator, seeded ``seed + offset`` with the
  offsets below; activations are N(0, 1), weights and biases N(0, 0.02)
  (0.02 is the standard deviation).
* Values are drawn in fp32 and rounded to bf16 with round-to-nearest-even
  (``Tensor.to(torch.bfloat16)``) when the storage dtype is bf16.  Biases stay
  fp32.
* Tensors with at most 2**24 elements are drawn on the CPU (torch's
  mt19937 generator).  Larger tensors (the Llama-2-70B-shaped weights) are
  drawn on the CUDA device with torch's Philox generator, because a CPU draw
  of 235 M values takes tens of seconds; the oracle then receives a host copy
  of the very same bits.
* The worked example of "Tensor parallel serving" ("Simulating the split, and
  proving it is correct") is drawn exactly as the page does: one generator
  seeded 0, then x [1, 8], W [6, 8], b [6] in that order, fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

# per-tensor seed offsets
OFF_X, OFF_W1, OFF_WUP, OFF_W2, OFF_B1, OFF_B2, OFF_CTX = 0, 1, 2, 3, 4, 5, 6

WEIGHT_STD = 0.02
CPU_DRAW_LIMIT = 1 << 24


def normal(shape, std: float, seed: int, dtype=torch.bfloat16, device=None,
           gen_device: Optional[str] = None) -> torch.Tensor:
    """N(0, std^2) tensor drawn from its own seeded generator.

    ``gen_device`` picks where the draw happens ("cpu" or "cuda"); by default
    small tensors are drawn on the CPU and large ones on CUDA.  The result is
    moved to ``device`` (default: where it was drawn).
    """
    numel = 1
    for s in shape:
        numel *= int(s)
    if gen_device is None:
        gen_device = "cpu" if numel <= CPU_DRAW_LIMIT else "cuda"
    g = torch.Generator(device=gen_device)
    g.manual_seed(int(seed))
    t = torch.randn(tuple(shape), generator=g, device=gen_device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    t = t.to(dtype)
    if device is not None:
        t = t.to(device)
    return t


def worked_example():
    """x [1, 8], W [6, 8], b [6], fp32, drawn in page order from seed 0."""
    g = torch.Generator(device="cpu")
    g.manual_seed(0)
    x = torch.randn(1, 8, generator=g)
    W = torch.randn(6, 8, generator=g)
    b = torch.randn(6, generator=g)
    return x, W, b


@dataclass
class FFNInputs:
    X: torch.Tensor                 # [M, d_model]
    W1: torch.Tensor                # [d_ff, d_model]  (gate weight for SwiGLU)
    W2: torch.Tensor                # [d_model, d_ff]
    W_up: Optional[torch.Tensor] = None   # [d_ff, d_model] (SwiGLU only)
    b1: Optional[torch.Tensor] = None     # [d_ff] fp32
    b2: Optional[torch.Tensor] = None     # [d_model] fp32
    meta: dict = field(default_factory=dict)


def ffn(seed: int, M: int, d_model: int, d_ff: int, act: str, bias: bool,
        device=None, dtype=torch.bfloat16, x_std: float = 1.0) -> FFNInputs:
    """FFN block inputs: X N(0,1), weights N(0,0.02), fp32 biases N(0,0.02)."""
    X = normal((M, d_model), x_std, seed + OFF_X, dtype, device)
    W1 = normal((d_ff, d_model), WEIGHT_STD, seed + OFF_W1, dtype, device)
    W2 = normal((d_model, d_ff), WEIGHT_STD, seed + OFF_W2, dtype, device)
    W_up = None
    if act == "swiglu":
        W_up = normal((d_ff, d_model), WEIGHT_STD, seed + OFF_WUP, dtype, device)
    b1 = b2 = None
    if bias:
        b1 = normal((d_ff,), WEIGHT_STD, seed + OFF_B1, torch.float32, device)
        b2 = normal((d_model,), WEIGHT_STD, seed + OFF_B2, torch.float32, device)
    return FFNInputs(X, W1, W2, W_up, b1, b2,
                     dict(seed=seed, M=M, d_model=d_model, d_ff=d_ff, act=act))


def gelu_ffn_small(seed: int = 1234, device=None) -> FFNInputs:
    """GELU FFN block, tp=2: X bf16 [16,512]; W1 [2048,512]; W2 [512,2048]; fp32 biases."""
    return ffn(seed, 16, 512, 2048, "gelu", True, device)


def llama70b_ffn(seed: int, M: int, device=None) -> FFNInputs:
    """Llama-2-70B-shaped SwiGLU FFN: d_model 8192, d_ff 28672, no bias."""
    return ffn(seed, M, 8192, 28672, "swiglu", False, device)


@dataclass
class AttnInputs:
    X: torch.Tensor        # [M, d_model]
    Wqkv: torch.Tensor     # [(H + 2 Hkv) hd, d_model], rows [Q heads; K heads; V heads]
    Wo: torch.Tensor       # [d_model, H hd]
    ctx: torch.Tensor      # [M, H hd]  stands in for the attention core's output
    bqkv: Optional[torch.Tensor] = None
    bo: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)


def attn(seed: int, M: int, d_model: int, n_heads: int, n_kv_heads: int,
         head_dim: int, bias: bool = False, device=None,
         dtype=torch.bfloat16) -> AttnInputs:
    """Attention-projection inputs: X, ctx N(0,1); Wqkv, Wo N(0,0.02)."""
    nq = (n_heads + 2 * n_kv_heads) * head_dim
    X = normal((M, d_model), 1.0, seed + OFF_X, dtype, device)
    Wqkv = normal((nq, d_model), WEIGHT_STD, seed + OFF_W1, dtype, device)
    Wo = normal((d_model, n_heads * head_dim), WEIGHT_STD, seed + OFF_W2, dtype, device)
    ctx = normal((M, n_heads * head_dim), 1.0, seed + OFF_CTX, dtype, device)
    bqkv = bo = None
    if bias:
        bqkv = normal((nq,), WEIGHT_STD, seed + OFF_B1, torch.float32, device)
        bo = normal((d_model,), WEIGHT_STD, seed + OFF_B2, torch.float32, device)
    return AttnInputs(X, Wqkv, Wo, ctx, bqkv, bo,
                      dict(seed=seed, M=M, d_model=d_model, n_heads=n_heads,
                           n_kv_heads=n_kv_heads, head_dim=head_dim))


def llama70b_attn(seed: int, M: int, device=None) -> AttnInputs:
    """64 query heads, 8 KV heads of dim 128 (GQA), d_model 8192, no bias."""
    return attn(seed, M, 8192, 64, 8, 128, False, device)


def sample_rows(M: int, count: int, seed: int) -> torch.Tensor:
    """Sorted distinct row indices: always 0 and M-1, the rest seeded-random."""
    count = min(count, M)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    rows = {0, M - 1}
    perm = torch.randperm(M, generator=g).tolist()
    for r in perm:
        if len(rows) >= count:
            break
        rows.add(r)
    return torch.tensor(sorted(rows), dtype=torch.long)
