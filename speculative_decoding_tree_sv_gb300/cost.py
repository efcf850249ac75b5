"""Algorithmic work of the verification path (host logic, no GPU needed).

The attention accounting follows the roofline argument of "Dynamic
Speculative Decoding" (Roofline Model Perspective Analysis, Attention
Analysis): per KV token and query row, one multiply-add pair for QK^T and one
for PV over the head dimension (4 * D FLOPs per head), and every KV byte is
read once.  Speculation shares the KV cache across the N proposed tokens, so
the intensity grows by N; grouped-query attention shares it across the G
query heads of a KV head, so it also grows by G.

Bytes are the compulsory HBM traffic of one launch: context K and V (2 bytes
per bf16 element), tree K and V, Q read once, the bf16 output written once,
plus the page indices and tree arrays.  FLOPs count the context part for
every node and, inside the tree, only the (depth + 1) visible tree keys of
each node (not the masked N x N block).
"""

from __future__ import annotations

from typing import Iterable, Optional, Sequence

BF16 = 2


def context_keys(ctx_len: int, page_size: int = 16, pages: Optional[Sequence[int]] = None) -> int:
    """Number of context keys a sequence attends to (L' in the text)."""
    if pages is None:
        return int(ctx_len)
    n = 0
    for p in pages:
        lo = int(p) * page_size
        n += max(0, min(lo + page_size, ctx_len) - lo)
    return n


def attention_bytes(ctx_keys: Iterable[int], nodes: Iterable[int], num_q_heads: int,
                    num_kv_heads: int, head_dim: int, page_size: int = 16,
                    with_lse: bool = False) -> int:
    ctx_keys = [int(x) for x in ctx_keys]
    nodes = [int(x) for x in nodes]
    kv_row = 2 * num_kv_heads * head_dim * BF16           # K and V of one token
    total = sum(ctx_keys) * kv_row                          # context cache
    total += sum(nodes) * kv_row                            # tree K/V
    total += 2 * sum(nodes) * num_q_heads * head_dim * BF16  # Q in, O out
    if with_lse:
        total += sum(nodes) * num_q_heads * 4
    pages = sum(-(-k // page_size) for k in ctx_keys)
    total += pages * 4 + sum(nodes) * 4 + 4 * 3 * len(nodes)  # indices, parents, lens
    return total


def attention_flops(ctx_keys: Iterable[int], depths_per_seq: Iterable[Sequence[int]],
                    num_q_heads: int, head_dim: int) -> int:
    total = 0
    for L, depths in zip(ctx_keys, depths_per_seq):
        n = len(depths)
        total += 4 * num_q_heads * head_dim * (n * int(L) + sum(int(d) + 1 for d in depths))
    return total


def per_context_token(num_q_heads: int, num_kv_heads: int, head_dim: int, nodes: int):
    """(FLOPs, bytes) that one context token adds to a launch: the form the
    roofline argument uses, with arithmetic intensity nodes * G."""
    flops = 4 * num_q_heads * head_dim * nodes
    bytes_ = 2 * num_kv_heads * head_dim * BF16
    return flops, bytes_


def accept_bytes(total_nodes: int, vocab: int, batch: int, max_depth: int) -> int:
    """Logits read once, plus tree arrays and the small outputs."""
    return total_nodes * vocab * 4 + total_nodes * 4 * 3 + batch * 4 * (3 + max_depth + 1)


def commit_bytes(accepted_per_seq: Iterable[int], num_layers: int, num_kv_heads: int,
                 head_dim: int) -> int:
    """Each committed slot: K and V read from the tree buffer and written to
    the cache, on every layer."""
    slots = sum(int(a) + 1 for a in accepted_per_seq)
    return slots * num_layers * 2 * num_kv_heads * head_dim * BF16 * 2
