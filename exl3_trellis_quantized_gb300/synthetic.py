"""Seeded synthetic inputs for the EXL3 linear layer.

This module only draws random numbers.  It holds none of the layer's
arithmetic, so both the CUDA path's tests and the CPU oracle can consume
the same inputs without sharing any of the method.

Distributions follow the workloads quoted for the layer:

* trellis words: uniform over all 2^16 int16 bit patterns, shape
  ``[K/16, N/16, 16*bits]`` (cuda-exl3 README, "VRAM"; TensorFold PR,
  "What it adds");
* suh / svh: fp16 ``sign * U(0.8, 1.2)`` with a fair random sign;
* activations x: bf16 draws of N(0, 1).

Everything is generated on the CPU with ``torch.Generator`` so that a
given seed yields the same bytes on every machine; callers move tensors
to the device themselves.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence

import torch


@dataclass
class Layer:
    """Host copies of one (possibly fused) EXL3 linear layer."""

    k: int
    shard_cols: List[int]  # column offsets, len S+1, shard s owns [c_s, c_{s+1})
    bits: int
    codebook: int  # 0 = 3inst, 1 = mcg, 2 = mul1
    trellis: torch.Tensor  # int16 [K/16, N/16, 16*bits]
    suh: torch.Tensor  # fp16 [S, K]
    svh: torch.Tensor  # fp16 [N]

    @property
    def n(self) -> int:
        return self.shard_cols[-1]

    @property
    def num_shards(self) -> int:
        return len(self.shard_cols) - 1


def _signed_uniform(g: torch.Generator, shape: Sequence[int]) -> torch.Tensor:
    mag = torch.rand(shape, generator=g, dtype=torch.float64) * 0.4 + 0.8
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.int64) * 2 - 1
    return (mag * sign).to(torch.float16)


def random_trellis(k: int, n: int, bits: int, g: torch.Generator) -> torch.Tensor:
    """Uniform random int16 words, every bit pattern equally likely."""
    if k % 16 or n % 16:
        raise ValueError("k and n must be multiples of 16")
    words = torch.randint(-(1 << 15), 1 << 15, (k // 16, n // 16, 16 * bits), generator=g, dtype=torch.int32)
    return words.to(torch.int16)


def make_layer(k: int, shard_widths: Sequence[int], bits: int, codebook: int, seed: int) -> Layer:
    g = torch.Generator().manual_seed(seed)
    cols = [0]
    for w in shard_widths:
        cols.append(cols[-1] + int(w))
    n = cols[-1]
    trellis = random_trellis(k, n, bits, g)
    suh = _signed_uniform(g, (len(shard_widths), k))
    svh = _signed_uniform(g, (n,))
    return Layer(k=k, shard_cols=cols, bits=bits, codebook=codebook, trellis=trellis, suh=suh, svh=svh)


def make_x(m: int, k: int, seed: int) -> torch.Tensor:
    """bf16 activations drawn from N(0, 1); smaller batches take a prefix."""
    g = torch.Generator().manual_seed(seed + 7919)
    return torch.randn((m, k), generator=g, dtype=torch.float32).to(torch.bfloat16)


def random_words(count: int, seed: int) -> torch.Tensor:
    """Uniform int16 words (used for tile-level unpack tests)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-(1 << 15), 1 << 15, (count,), generator=g, dtype=torch.int32).to(torch.int16)


# ---------------------------------------------------------------------------
# Mixture-of-experts inputs
# ---------------------------------------------------------------------------


@dataclass
class MoeLayer:
    """Host copies of one EXL3 expert layer: E experts of the same shape."""

    k: int
    shard_cols: List[int]
    bits: int
    codebook: int
    trellis: torch.Tensor  # int16 [E, K/16, N/16, 16*bits] (experts stacked)
    suh: torch.Tensor  # fp16 [E, S, K]
    svh: torch.Tensor  # fp16 [E, N]

    @property
    def n(self) -> int:
        return self.shard_cols[-1]

    @property
    def num_experts(self) -> int:
        return self.trellis.shape[0]


def make_moe_layer(k: int, shard_widths: Sequence[int], bits: int, codebook: int, num_experts: int,
                   seed: int) -> MoeLayer:
    layers = [make_layer(k, shard_widths, bits, codebook, seed * 1009 + e) for e in range(num_experts)]
    return MoeLayer(k=k, shard_cols=layers[0].shard_cols, bits=bits, codebook=codebook,
                    trellis=torch.stack([l.trellis for l in layers]), suh=torch.stack([l.suh for l in layers]),
                    svh=torch.stack([l.svh for l in layers]))


@dataclass
class Routing:
    """Routed (token, expert) pairs in the block-aligned order a grouped GEMM
    consumes (the layout vLLM's moe_align_block_size produces, cuda-exl3 README,
    "What is supported" and "MoE notes"): pairs sorted by expert, each expert's
    run padded to whole blocks of ``block`` rows.

    sorted_ids[r] is the pair index token * topk + slot of padded row r, or
    num_tokens * topk for a padding row; block_expert[b] is the expert of rows
    [b * block, (b + 1) * block), or -1 for a block that belongs to no expert
    (such blocks also sit between live ones, not only at the end).
    """

    num_tokens: int
    topk: int
    block: int
    topk_ids: torch.Tensor  # int32 [num_tokens, topk], distinct experts per token
    sorted_ids: torch.Tensor  # int32 [rows]
    block_expert: torch.Tensor  # int32 [rows / block]

    @property
    def rows(self) -> int:
        return self.sorted_ids.numel()


def make_routing(num_tokens: int, num_experts: int, topk: int, block: int, seed: int,
                 empty_blocks: int = 2) -> Routing:
    """Random top-k choices (distinct experts per token), aligned to blocks,
    with ``empty_blocks`` blocks of -1 inserted at random positions."""
    g = torch.Generator().manual_seed(seed)
    topk_ids = torch.stack([torch.randperm(num_experts, generator=g)[:topk] for _ in range(num_tokens)]).to(torch.int32)
    pad = num_tokens * topk
    ids: List[int] = []
    blocks: List[int] = []
    flat = topk_ids.reshape(-1).tolist()
    for e in range(num_experts):
        run = [i for i, x in enumerate(flat) if x == e]
        if not run:
            continue
        nb = -(-len(run) // block)
        run += [pad] * (nb * block - len(run))
        ids += run
        blocks += [e] * nb
    for _ in range(empty_blocks):
        at = int(torch.randint(0, len(blocks) + 1, (1,), generator=g))
        blocks.insert(at, -1)
        ids[at * block:at * block] = [pad] * block
    return Routing(num_tokens=num_tokens, topk=topk, block=block, topk_ids=topk_ids,
                   sorted_ids=torch.tensor(ids, dtype=torch.int32), block_expert=torch.tensor(blocks, dtype=torch.int32))


def make_topk_weights(num_tokens: int, topk: int, seed: int) -> torch.Tensor:
    """Router weights of each token's top-k slots: float32 [num_tokens, topk],
    positive and normalised to sum to 1 per token."""
    g = torch.Generator().manual_seed(seed)
    w = torch.rand((num_tokens, topk), generator=g, dtype=torch.float32) + 0.05
    return w / w.sum(dim=1, keepdim=True)
