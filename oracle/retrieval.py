"""Oracle for SpecPV block retrieval (float64) — TEST INFRASTRUCTURE ONLY.

What is computed, from SpecPV:

* section 3.2 "Partial Verification": the partial KV cache keeps the initial
  sink blocks, query-dependent retrieved blocks, a fixed-size local window
  and a buffer, attended as one continuous segment; key-state summaries of
  every block are cached to speed up retrieval, and they are the
  element-wise maximum and minimum of the block's key states; blocks are
  scored against several candidate tokens' query states and the per-query
  scores are reduced to one block-importance score by a reduction such as
  max, mean or last;
* Appendix C: mean reduction works best;  Appendix D: blocks of 16 tokens.

Readings where the pages are silent (also listed in the design notes):

* The score of a block for one query q (query head h, KV head h // G) is the
  largest value q . k can take for a key k lying element-wise between the
  block's minimum and maximum key: sum_d max(q_d * kmax_d, q_d * kmin_d).  It
  bounds q . k from above for every key of the block.
* A block's importance reduces those scores over all candidate tokens (the
  tree's nodes) and all query heads: their mean ("mean"), their maximum
  ("max"), or the mean over query heads for the last node in index order
  ("last").
* A block is one 16-token page (logical page p holds tokens 16p .. 16p+15;
  the last page of a context may be partial and its summary covers only its
  valid tokens).
* Sink pages are the first ceil(sink_tokens / 16) pages; window pages are
  those holding the last window_tokens tokens.  The other pages are the
  candidates; the topk most important (ties: lower page id first) are
  retrieved.  The partial list is sink, retrieved and window pages in
  ascending order.  (SpecPV's buffer of partially verified tokens lies at
  the end of the context and is covered by the window.)

Only the test suite may import this module.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from .attention import bf16_to_f64

REDUCTIONS = ("mean", "max", "last")


def page_summaries(k_cache: np.ndarray, block_table: np.ndarray, ctx_lens: Sequence[int],
                   page_size: int = 16) -> Tuple[np.ndarray, np.ndarray]:
    """Element-wise max and min of the valid keys of every page in use.

    k_cache: bf16 bits [num_pages, Hkv, page_size, D].  Returns
    (summary float64 [num_pages, Hkv, 2, D] with [:, :, 0] = max and
    [:, :, 1] = min, defined bool [num_pages]).  Pages no sequence uses stay
    zero and undefined."""
    num_pages, hkv, ps, d = k_cache.shape
    assert ps == page_size
    summ = np.zeros((num_pages, hkv, 2, d), dtype=np.float64)
    defined = np.zeros(num_pages, dtype=bool)
    for b, L in enumerate(ctx_lens):
        L = int(L)
        for lp in range((L + page_size - 1) // page_size):
            phys = int(block_table[b, lp])
            valid = min(page_size, L - lp * page_size)
            keys = bf16_to_f64(k_cache[phys, :, :valid, :])  # [Hkv, valid, D]
            summ[phys, :, 0, :] = keys.max(axis=1)
            summ[phys, :, 1, :] = keys.min(axis=1)
            defined[phys] = True
    return summ, defined


def query_block_score(q: np.ndarray, kmax: np.ndarray, kmin: np.ndarray) -> float:
    """Largest q . k for any key k with kmin <= k <= kmax element-wise."""
    return float(np.sum(np.maximum(q * kmax, q * kmin)))


def page_regions(ctx_len: int, sink_tokens: int, window_tokens: int,
                 page_size: int = 16) -> Tuple[int, int, int]:
    """(n_pages, number of sink pages, first window page) of a context."""
    n_pages = (int(ctx_len) + page_size - 1) // page_size
    sink = min(n_pages, (int(sink_tokens) + page_size - 1) // page_size)
    first_window = min(n_pages, max(0, int(ctx_len) - int(window_tokens)) // page_size)
    first_window = max(first_window, sink)
    return n_pages, sink, first_window


def block_importance(q_seq: np.ndarray, summ: np.ndarray, phys_pages: Sequence[int], num_kv_heads: int,
                     reduce: str) -> np.ndarray:
    """Importance of each listed physical page for one sequence.

    q_seq: query values float64 [N, Hq, D] (post-RoPE) of the sequence's tree
    nodes; summ as returned by page_summaries."""
    n, hq, _ = q_seq.shape
    g = hq // num_kv_heads
    out = np.zeros(len(phys_pages), dtype=np.float64)
    nodes = [n - 1] if reduce == "last" else list(range(n))
    for pi, phys in enumerate(phys_pages):
        scores = []
        for i in nodes:
            for h in range(hq):
                kv = h // g
                scores.append(query_block_score(q_seq[i, h], summ[phys, kv, 0], summ[phys, kv, 1]))
        if reduce == "max":
            out[pi] = max(scores)
        elif reduce in ("mean", "last"):
            out[pi] = float(np.mean(scores))
        else:
            raise ValueError(reduce)
    return out


def retrieve_pages(q: np.ndarray, k_cache: np.ndarray, block_table: np.ndarray, ctx_lens: Sequence[int],
                   cu_nodes: Sequence[int], sink_tokens: int, window_tokens: int, topk: int,
                   reduce: str = "mean", page_size: int = 16
                   ) -> Tuple[np.ndarray, np.ndarray, List[Dict[int, float]]]:
    """Partial page lists of every sequence.

    q: bf16 bits [T, Hq, D].  Returns (kv_pages int32, cu_kv_pages int32
    [B+1], per sequence a dict logical candidate page -> importance)."""
    if reduce not in REDUCTIONS:
        raise ValueError(reduce)
    num_kv_heads = k_cache.shape[1]
    summ, _ = page_summaries(k_cache, block_table, ctx_lens, page_size)
    qf = bf16_to_f64(q)
    lists, scores_all = [], []
    for b, L in enumerate(ctx_lens):
        n_pages, sink, first_window = page_regions(int(L), sink_tokens, window_tokens, page_size)
        cand = list(range(sink, first_window))
        imp = block_importance(qf[cu_nodes[b]:cu_nodes[b + 1]], summ, [int(block_table[b, p]) for p in cand],
                               num_kv_heads, reduce)
        scores_all.append({p: float(s) for p, s in zip(cand, imp)})
        order = sorted(range(len(cand)), key=lambda i: (-imp[i], cand[i]))
        chosen = {cand[i] for i in order[:min(int(topk), len(cand))]}
        keep = set(range(sink)) | chosen | set(range(first_window, n_pages))
        lists.append(sorted(keep))
    cu = np.zeros(len(lists) + 1, dtype=np.int32)
    for b, lst in enumerate(lists):
        cu[b + 1] = cu[b] + len(lst)
    flat = np.array([p for lst in lists for p in lst], dtype=np.int32)
    return flat, cu, scores_all


def extend_partial_lists(ref_pages: Sequence[int], ref_cu: Sequence[int], ref_ctx_lens: Sequence[int],
                         ctx_lens: Sequence[int], page_size: int = 16) -> Tuple[np.ndarray, np.ndarray]:
    """SpecPV section 3.3: between refreshes a sequence attends its refresh
    list plus the pages its buffer of partially verified tokens has grown
    into (the buffer follows the window at the end of the context)."""
    lists = []
    for b in range(len(ctx_lens)):
        lst = [int(x) for x in ref_pages[ref_cu[b]:ref_cu[b + 1]]]
        first_new = (int(ref_ctx_lens[b]) + page_size - 1) // page_size
        now = (int(ctx_lens[b]) + page_size - 1) // page_size
        lists.append(lst + list(range(first_new, now)))
    cu = np.zeros(len(lists) + 1, dtype=np.int32)
    for b, lst in enumerate(lists):
        cu[b + 1] = cu[b] + len(lst)
    return np.array([p for lst in lists for p in lst], dtype=np.int32), cu


def specpv_schedule(step_commits: Sequence[int], step_tokens: int, buffer_limit: int,
                    ctx_len0: int) -> List[str]:
    """Kinds of verification a sequence runs (SpecPV section 3.3): full until
    a partial cache exists; partial while the buffer of tokens committed by
    partial steps, plus what the next step can commit, fits the limit; full
    (refreshing the cache, emptying the buffer) otherwise.  step_commits[i]
    is what step i commits."""
    kinds, has_cache, refresh_len, ctx = [], False, 0, int(ctx_len0)
    for c in step_commits:
        buffered = ctx - refresh_len
        if not has_cache or buffered + step_tokens > buffer_limit:
            kinds.append("full")
            ctx += int(c)
            has_cache, refresh_len = True, ctx
        else:
            kinds.append("partial")
            ctx += int(c)
    return kinds


def specpv_full_tree(cand_parents: Sequence[int], cand_tokens: Sequence[int],
                     buffer_tokens: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """The tree of a full verification that follows partial ones, for one
    sequence (SpecPV section 3.3, "Rectified with Full Verification": before
    the full verification, the partially verified tokens are prepended to the
    new candidates; the full KV cache is used and the partial cache is
    refreshed).

    ``buffer_tokens`` are the tokens committed since the last full
    verification, in order: positions R .. L-1, R being the context length at
    that refresh.  ``cand_parents`` / ``cand_tokens`` are this step's
    candidate tree (sequence-local ids, root = node 0 = the last accepted
    token, at position L).  The result puts the buffered tokens in a chain
    from the root (node j is the token at position R + j, its parent j - 1)
    and hangs the candidate tree below the chain's last node: candidate node
    i becomes node nb + i (nb = number of buffered tokens), with parent
    nb + parent[i], and the candidate root's parent is nb - 1.  Reading of
    the pages: the step is verified at context length R, so every buffered
    token is checked again like a candidate (node j is accepted when its
    token is the target's choice after node j - 1), and the commit writes
    slots R .. R + a, rewriting the buffered slots with the K/V of this
    forward.  With no buffered token the result is the candidate tree.

    Returns (parents int32 [nb + N], tokens int32 [nb + N])."""
    nb = len(buffer_tokens)
    n = len(cand_parents)
    parents = np.empty(nb + n, dtype=np.int32)
    tokens = np.empty(nb + n, dtype=np.int32)
    for j in range(nb):
        parents[j] = j - 1
        tokens[j] = int(buffer_tokens[j])
    for i in range(n):
        if i == 0:
            parents[nb] = nb - 1  # -1 when nothing is buffered
        else:
            parents[nb + i] = nb + int(cand_parents[i])
        tokens[nb + i] = int(cand_tokens[i])
    return parents, tokens


def specpv_full_step_trees(cand_parents: Sequence[int], cand_tokens: Sequence[int], cand_cu: Sequence[int],
                           buffer_tokens: Sequence[int], buffer_cu: Sequence[int]
                           ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """specpv_full_tree for every sequence of a batch: candidate trees packed
    with offsets cand_cu [B+1], buffered tokens packed with offsets
    buffer_cu [B+1].  Returns (parents, tokens, cu_nodes) of the combined
    trees, packed in sequence order."""
    par_all, tok_all, cu = [], [], [0]
    for b in range(len(cand_cu) - 1):
        c0, c1 = int(cand_cu[b]), int(cand_cu[b + 1])
        b0, b1 = int(buffer_cu[b]), int(buffer_cu[b + 1])
        par, tok = specpv_full_tree(cand_parents[c0:c1], cand_tokens[c0:c1], buffer_tokens[b0:b1])
        par_all.append(par)
        tok_all.append(tok)
        cu.append(cu[-1] + len(par))
    cat = (lambda xs: np.concatenate(xs).astype(np.int32)) if par_all else (lambda xs: np.zeros(0, np.int32))
    return cat(par_all), cat(tok_all), np.asarray(cu, dtype=np.int32)
