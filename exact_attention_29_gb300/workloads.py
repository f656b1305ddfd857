"""Seeded synthetic workloads: named shapes and the input generators.

This module holds no attention arithmetic. It only names the workload shapes
and draws their inputs from seeds, so that the CUDA path, the fp64 oracle and
the benchmark all see the very same bf16 values.

Input recipe
------------
* Prefill: one ``torch.Generator`` seeded with ``seed`` draws Q, then K, then V
  as standard-normal fp32 of shape [B, H, N, d]; each is rounded to bf16
  (round-to-nearest-even). Standard normal entries make the raw dot products
  q.k have variance d, the regime the 1/sqrt(d) scale is meant for (CMU
  15-779 Lecture 5 notes §2.3 and Exercise 2).
* Decode: the same generator draws q [B, H, d], then the K cache, then the V
  cache [B, H, L, d]. Ragged lengths come from a second generator seeded with
  ``seed + 1``: uniform integers in [1024, L].
* Row subsets (long-context checks): a generator seeded with ``seed + 2``
  draws ``randperm(N)[:n_rows]`` independently for each (b, h) in order.
* Inputs of more than ``GPU_GEN_THRESHOLD`` elements are drawn on the GPU by a
  CUDA ``torch.Generator`` (same seed, different stream of numbers than the
  CPU generator) in slices of one batch entry, because drawing gigabytes on
  the host takes minutes. The oracle then reads back only the heads it checks.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

GPU_GEN_THRESHOLD = 1 << 25  # elements per tensor


@dataclass(frozen=True)
class Prefill:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    @property
    def flops(self) -> float:
        """Matmul FLOPs: 4 B H N^2 d, half of that under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f


@dataclass(frozen=True)
class Decode:
    name: str
    B: int
    H: int
    L: int
    d: int
    ragged: bool


PREFILL = {
    "pr1": Prefill("pr1", 1, 1, 128, 64, False),
    "gpt2_small": Prefill("gpt2_small", 8, 12, 1024, 64, False),
    "gpt2_small_causal": Prefill("gpt2_small_causal", 8, 12, 1024, 64, True),
    "llama3_8b_prefill": Prefill("llama3_8b_prefill", 2, 32, 4096, 128, True),
    "llama3_8b_prefill_noncausal": Prefill("llama3_8b_prefill_noncausal", 2, 32, 4096, 128, False),
    "long_16k": Prefill("long_16k", 1, 32, 16384, 128, True),
    "long_64k": Prefill("long_64k", 1, 32, 65536, 128, True),
}

DECODE = {
    "decode_32k": Decode("decode_32k", 16, 32, 32768, 128, False),
    "decode_32k_ragged": Decode("decode_32k_ragged", 16, 32, 32768, 128, True),
}

DECODE_SPLITS = (8, 16, 32)

# Block-sparse prefill: the Llama-3-8B-shaped problem (non-causal) under a
# band + global + random block mask (block_mask_bigbird, 128-key blocks).
SPARSE_PREFILL = Prefill("llama3_8b_prefill_bigbird", 2, 32, 4096, 128, False)


@dataclass(frozen=True)
class DecodeGQA:
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    d: int
    ragged: bool

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv


# Grouped K/V heads (Lecture 5 notes, Exercise 7): g = 8 is the 64-query-head,
# 8-K/V-head grouping the exercise takes; g = 4 groups 32 query heads over 8
# K/V heads; MQA puts 32 query heads on one K/V head.
DECODE_GQA = {
    "decode_gqa8_32k": DecodeGQA("decode_gqa8_32k", 16, 64, 8, 32768, 128, False),
    "decode_gqa8_32k_ragged": DecodeGQA("decode_gqa8_32k_ragged", 16, 64, 8, 32768, 128, True),
    "decode_gqa4_32k": DecodeGQA("decode_gqa4_32k", 16, 32, 8, 32768, 128, False),
    "decode_mqa_32k": DecodeGQA("decode_mqa_32k", 16, 32, 1, 32768, 128, False),
}


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    numel = 1
    for s in shape:
        numel *= s
    if numel <= GPU_GEN_THRESHOLD or str(device) == "cpu":
        return torch.randn(shape, generator=gen, dtype=torch.float32, device=gen.device).to(torch.bfloat16).to(device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for b in range(shape[0]):
        out[b].copy_(torch.randn(shape[1:], generator=gen, dtype=torch.float32, device=gen.device))
    return out


def _generator(seed: int, numel: int, device) -> torch.Generator:
    gdev = "cuda" if (numel > GPU_GEN_THRESHOLD and str(device) != "cpu") else "cpu"
    g = torch.Generator(device=gdev)
    g.manual_seed(seed)
    return g


def prefill_inputs(B: int, H: int, N: int, d: int, seed: int = 0, device="cpu"):
    """Q, K, V bf16 [B, H, N, d] drawn in that order from one seeded generator."""
    shape = (B, H, N, d)
    g = _generator(seed, B * H * N * d, device)
    q = _randn_bf16(shape, g, device)
    k = _randn_bf16(shape, g, device)
    v = _randn_bf16(shape, g, device)
    return q, k, v


def backward_inputs(B: int, H: int, N: int, d: int, seed: int = 0, device="cpu"):
    """The upstream gradient dO, bf16 [B, H, N, d], from its own seeded stream
    (independent of the Q, K, V drawn by prefill_inputs with the same seed)."""
    g = _generator(seed + 7919, B * H * N * d, device)
    return _randn_bf16((B, H, N, d), g, device)


def decode_inputs(B: int, H: int, L: int, d: int, seed: int = 0, ragged: bool = False,
                  device="cpu", lo: int = 1024):
    """q [B,H,d], K/V caches [B,H,L,d] (bf16) and seqlens [B] (int32)."""
    g = _generator(seed, B * H * L * d, device)
    q = _randn_bf16((B, H, d), g, device)
    k = _randn_bf16((B, H, L, d), g, device)
    v = _randn_bf16((B, H, L, d), g, device)
    return q, k, v, decode_seqlens(B, L, seed, ragged, lo).to(device)


def decode_seqlens(B: int, L: int, seed: int = 0, ragged: bool = False, lo: int = 1024) -> torch.Tensor:
    """Cache lengths [B] (int32, on the host): all L, or (ragged) uniform
    integers in [min(lo, L), L] from a generator seeded with ``seed + 1``."""
    if not ragged:
        return torch.full((B,), L, dtype=torch.int32)
    gl = torch.Generator(device="cpu")
    gl.manual_seed(seed + 1)
    return torch.randint(min(lo, L), L + 1, (B,), generator=gl, dtype=torch.int64).to(torch.int32)


def decode_gqa_inputs(B: int, Hq: int, Hkv: int, L: int, d: int, seed: int = 0, ragged: bool = False,
                      device="cpu", lo: int = 1024):
    """q [B,Hq,d], K/V caches [B,Hkv,L,d] (bf16) and seqlens [B] (int32), drawn
    in that order; lengths as in decode_inputs."""
    g = _generator(seed, B * Hkv * L * d, device)
    q = _randn_bf16((B, Hq, d), g, device)
    k = _randn_bf16((B, Hkv, L, d), g, device)
    v = _randn_bf16((B, Hkv, L, d), g, device)
    return q, k, v, decode_seqlens(B, L, seed, ragged, lo).to(device)


def block_mask_bigbird(T: int, heads: int = 1, window: int = 1, globals_: int = 1, random: int = 2,
                       seed: int = 0) -> torch.Tensor:
    """A seeded block mask [heads, T, T] (uint8) of the kind block-sparse
    attention serves: a band of +-window blocks, the first `globals_` block rows
    and columns, and `random` extra blocks per block row."""
    g = torch.Generator().manual_seed(seed + 3)
    m = torch.zeros((heads, T, T), dtype=torch.uint8)
    idx = torch.arange(T)
    band = (idx[:, None] - idx[None, :]).abs() <= window
    m[:, band] = 1
    m[:, :globals_, :] = 1
    m[:, :, :globals_] = 1
    for h in range(heads):
        for i in range(T):
            m[h, i, torch.randint(0, T, (random,), generator=g)] = 1
    return m


def row_subsets(B: int, H: int, N: int, n_rows: int, seed: int = 0):
    """Per-(b, h) random query-row subsets, as a [B, H, n_rows] int64 tensor."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 2)
    out = torch.empty((B, H, min(n_rows, N)), dtype=torch.int64)
    for b in range(B):
        for h in range(H):
            out[b, h] = torch.randperm(N, generator=g)[: min(n_rows, N)]
    return out
