"""Oracle for committing the accepted path's K/V into the paged cache.

SpecBlock, Appendix A.5: the longest accepted prefix is committed before the
next iteration; "Dynamic Speculative Decoding", Implementation Details: the
KV cache must stay consistent with the committed tokens.

Reading: the root (the last accepted token of the previous step) and the a
accepted nodes get cache slots L .. L + a of their sequence, in path order,
on every layer; slot s lives in logical page s // P at offset s % P.  The
bonus token has no K/V yet (it becomes the next step's root).  The new
context length is L + a + 1.  All other cache bytes are unchanged.

Test infrastructure only.
"""

from __future__ import annotations

import numpy as np


def kv_commit(k_cache, v_cache, tree_k, tree_v, block_table, ctx_lens, cu_nodes,
              accepted_nodes, accept_len, page_size: int = 16):
    """Arrays carry a leading layer axis:
      k/v_cache [layers, pages, Hkv, P, D] (any dtype; copied bit for bit)
      tree_k/v  [layers, T, Hkv, D]
      accepted_nodes: per sequence, local node ids root first (len a + 1)
    Returns ``(k_new, v_new, new_ctx_lens)``; inputs are not modified."""
    k_new = np.array(k_cache, copy=True)
    v_new = np.array(v_cache, copy=True)
    B = len(ctx_lens)
    new_lens = np.zeros(B, dtype=np.int64)
    for b in range(B):
        L = int(ctx_lens[b])
        a = int(accept_len[b])
        base = int(cu_nodes[b])
        for j in range(a + 1):
            node = int(accepted_nodes[b][j])
            slot = L + j
            page = int(block_table[b][slot // page_size])
            off = slot % page_size
            for layer in range(k_new.shape[0]):
                k_new[layer, page, :, off, :] = tree_k[layer, base + node]
                v_new[layer, page, :, off, :] = tree_v[layer, base + node]
        new_lens[b] = L + a + 1
    return k_new, v_new, new_lens
