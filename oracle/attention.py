"""Oracle for tree-verification attention (float64, explicit mask).

What is computed (one layer):

* SpecBlock, Appendix A.5 "Inference procedure": the verifier scores every
  drafted tree node in one parallel forward.
* SpecBlock, Appendix A.2 "Attention Mask for SpecBlock": a drafted position
  sees the verified prefix and the positions on its own branch path; off-path
  positions are masked.  For the verifier this is the ancestor-or-self mask
  over tree nodes, with the whole committed context visible.
* SpecPV, section 3.2 "Partial Verification": with a partial cache the
  retained blocks (sink, retrieved, local window, buffer) are treated as one
  continuous KV segment.  Here the retained set is a list of 16-token pages.

Readings where the pages are silent: softmax scale 1/sqrt(D); query head h
uses KV head floor(h / G) with G = Hq / Hkv; Q and K arrive with positions
already applied; the root (node 0) is the last accepted token, its K/V is
the tree's node 0 and it is not part of the context length L.

The oracle is test infrastructure: only tests, the smoke check and the CPU
baseline of the benchmark use it.
"""

from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def ancestor_or_self_mask(parents: Sequence[int]) -> np.ndarray:
    """mask[i, j] is True iff tree node j lies on the path from the root to i
    (j is an ancestor of i, or j == i).  ``parents[0] == -1`` is the root."""
    n = len(parents)
    mask = np.zeros((n, n), dtype=bool)
    for i in range(n):
        j = i
        steps = 0
        while j != -1:
            mask[i, j] = True
            j = int(parents[j])
            steps += 1
            if steps > n:
                raise ValueError("parent array has a cycle")
    return mask


def context_positions(ctx_len: int, page_size: int,
                      pages: Optional[Sequence[int]] = None) -> np.ndarray:
    """Logical token positions of the context keys a sequence attends to.

    Full verification: 0 .. L-1.  Partial verification: the tokens of each
    listed logical page, 16p .. min(16p + 15, L - 1), concatenated in list
    order (the list is ascending and unique)."""
    if pages is None:
        return np.arange(ctx_len, dtype=np.int64)
    out = []
    for p in pages:
        lo = int(p) * page_size
        hi = min(lo + page_size, ctx_len)
        out.extend(range(lo, hi))
    return np.asarray(out, dtype=np.int64)


def gather_context(cache_layer: np.ndarray, table_row: np.ndarray,
                   positions: np.ndarray, page_size: int) -> np.ndarray:
    """K or V of the listed logical positions: cache [pages, Hkv, P, D] ->
    [len(positions), Hkv, D] (bf16 bits)."""
    phys = table_row[positions // page_size]
    slot = positions % page_size
    return cache_layer[phys, :, slot, :]


def visibility_mask(parents: Sequence[int], num_ctx: int) -> np.ndarray:
    """Explicit N x (L' + N) boolean mask: every context column is visible;
    tree column j is visible from row i iff j is an ancestor of i or i."""
    n = len(parents)
    mask = np.ones((n, num_ctx + n), dtype=bool)
    mask[:, num_ctx:] = ancestor_or_self_mask(parents)
    return mask


def tree_verify_attention(q, tree_k, tree_v, k_cache, v_cache, block_table,
                          ctx_lens, cu_nodes, parents, *, page_size: int = 16,
                          kv_pages=None, cu_kv_pages=None,
                          sm_scale: Optional[float] = None,
                          seqs: Optional[Sequence[int]] = None,
                          kv_heads: Optional[Sequence[int]] = None):
    """Tree-verification attention for one layer.

    Arguments (bf16 arrays are uint16 bit patterns):
      q        [T, Hq, D]            queries of all tree nodes of all sequences
      tree_k/v [T, Hkv, D]           this step's K/V of the tree nodes
      k/v_cache [num_pages, Hkv, P, D]  paged context cache
      block_table [B, max_pages]     logical page -> physical page
      ctx_lens [B], cu_nodes [B+1], parents [T] (sequence-local, root -1)
      kv_pages / cu_kv_pages         optional partial page lists
      seqs / kv_heads                optional subsets (others are left NaN)

    Returns ``(out, lse)``: out float64 [T, Hq, D] and lse float64 [T, Hq],
    the natural log of the softmax denominator sum_j exp(scale * q . k_j).
    """
    q = np.asarray(q)
    T, Hq, D = q.shape
    Hkv = tree_k.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    B = len(ctx_lens)
    seqs = range(B) if seqs is None else seqs
    kv_heads = range(Hkv) if kv_heads is None else kv_heads
    for b in seqs:
        n0, n1 = int(cu_nodes[b]), int(cu_nodes[b + 1])
        n = n1 - n0
        if n == 0:
            continue
        L = int(ctx_lens[b])
        pages = None
        if kv_pages is not None:
            pages = kv_pages[int(cu_kv_pages[b]): int(cu_kv_pages[b + 1])]
        pos = context_positions(L, page_size, pages)
        k_ctx = gather_context(k_cache, block_table[b], pos, page_size)
        v_ctx = gather_context(v_cache, block_table[b], pos, page_size)
        mask = visibility_mask(parents[n0:n1], len(pos))
        for g in kv_heads:
            K = np.concatenate([bf16_to_f64(k_ctx[:, g, :]), bf16_to_f64(tree_k[n0:n1, g, :])])
            V = np.concatenate([bf16_to_f64(v_ctx[:, g, :]), bf16_to_f64(tree_v[n0:n1, g, :])])
            for h in range(g * G, (g + 1) * G):
                Q = bf16_to_f64(q[n0:n1, h, :])
                s = (Q @ K.T) * scale
                s = np.where(mask, s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                p = np.exp(s - m)
                l = p.sum(axis=1, keepdims=True)
                out[n0:n1, h, :] = (p @ V) / l
                lse[n0:n1, h] = (m + np.log(l))[:, 0]
    return out, lse


def attention_probabilities(q_rows, keys, mask, scale):
    """Softmax probabilities of rows ``q_rows`` [N, D] over ``keys`` [K, D]
    under boolean ``mask`` [N, K] (used by invariant checks)."""
    s = np.where(mask, (q_rows @ keys.T) * scale, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return p / p.sum(axis=1, keepdims=True)
