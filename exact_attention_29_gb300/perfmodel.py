"""Work and traffic models used to report throughput and roofline fractions.

FLOPs count only the two matrix products: 2 N^2 d each per head, 4 N^2 d in
all, half of that under the causal mask (CMU 15-779 Lecture 5 notes §3.1;
"FlashAttention 完全拆解（一）", background section: 4 N^2 d for one forward).

HBM traffic of the tiled forward in elements, per head, with Q tiles of B_r
rows and K/V re-read once per Q tile: 2Nd (read Q, write O) + 2Nd * N/B_r
(K and V re-reads) + N (the LSE) (Lecture 5 notes §5.4 and Exercise 4;
"已有的几种大模型上下文支持情况" §3.3). When K/V stay in L2 the re-reads
collapse to one read, leaving the algorithmic minimum 4Nd + N.

The backward with recomputation (Lecture 5 notes §7.2-7.3) makes five
N x N x d products per head: S = Q K^T again, dP = dO V^T, dV = P^T dO,
dK = dS^T Q and dQ = dS K, 10 N^2 d FLOPs, half under the causal mask (a
count derived from those products; the pages print no figure for it).

Decode reads every cached K and V element of every visible position once
(arithmetic intensity about 1, Lecture 5 notes §8.3).
"""
from __future__ import annotations


def fwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def bwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 10.0 * B * H * N * N * d
    return f / 2 if causal else f


def fwd_hbm_elements_tiled(N: int, d: int, B_r: int) -> int:
    """Per-head forward traffic with every K/V tile re-read from HBM once per Q tile."""
    return 2 * N * d + 2 * N * d * ((N + B_r - 1) // B_r) + N


def fwd_algorithmic_bytes(B: int, H: int, N: int, d: int, elem_bytes: int = 2, lse_bytes: int = 4) -> int:
    """Minimum traffic: read Q, K, V once, write O once (bf16), write the LSE (fp32)."""
    return B * H * (4 * N * d * elem_bytes + N * lse_bytes)


def decode_kv_bytes(H: int, d: int, seqlens, elem_bytes: int = 2) -> int:
    """K and V bytes a decode step must read: 2 * H * d * elem_bytes per visible position."""
    return 2 * H * d * elem_bytes * int(sum(int(x) for x in seqlens))


def decode_algorithmic_bytes(B: int, H: int, d: int, seqlens, elem_bytes: int = 2) -> int:
    """Decode traffic: the K/V reads plus q read, o and lse written."""
    return decode_kv_bytes(H, d, seqlens, elem_bytes) + B * H * (2 * d * elem_bytes + 4)
