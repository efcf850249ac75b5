"""Oracle for stochastic (temperature > 0) acceptance of a verified draft tree
-- TEST INFRASTRUCTURE ONLY.

What the pages fix:

* SpecPV section 2 (related work): speculative sampling (Leviathan et al.,
  2023) lets a target verify draft tokens so that the emitted tokens follow
  the target's own sampling distribution; SpecInfer organises the candidates
  as a token tree.
* SpecBlock section 4 evaluates at temperature 1.0 as well as 0; SpecPV
  Appendix E at 0.7 and 1.0.

The pages give no rule for a tree.  Reading (listed in the design notes):
SpecInfer's multi-step speculative sampling, node by node.

* The target distribution at node u is p_u = softmax(logits_u / T).  The draft
  distribution q_u (an input, one probability vector per node) is the one the
  children of u were drawn from.
* The children c_1 .. c_k of u are tried in index order with a residual R that
  starts as p_u: child c_i (token x_i, uniform r_i) is accepted when
  r_i < min(1, R(x_i) / q_u(x_i)) (a zero q_u(x_i) accepts); otherwise
  R <- max(R - q_u, 0) / sum(max(R - q_u, 0)) (unchanged when that sum is 0,
  which needs R <= q_u everywhere, i.e. R = q_u, where every test accepts).
* The walk starts at the root and moves to the accepted child while there is
  one; it ends at node z.  accept_len is the depth of z, the path its root
  path, and the bonus token is drawn from R at z (p_z for a leaf, the residual
  after all of z's children were rejected otherwise) by inverse CDF with z's
  second uniform v_z: the smallest x with R(0) + ... + R(x) > v_z.

The uniforms are inputs (u_accept[n] for the test of node n at its parent,
u_bonus[n] for a draw at n), so both sides are deterministic.  Everything
here is float64; the decisions are returned with their margins so that a
float32 implementation can be compared where the decision is not within
rounding of its threshold.
"""

from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np


def target_probs(logits_row: np.ndarray, temperature: float) -> np.ndarray:
    """softmax(logits / T) in float64."""
    z = np.asarray(logits_row, dtype=np.float64) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def node_verify(p: np.ndarray, q: np.ndarray, child_tokens: Sequence[int], child_uniforms: Sequence[float]):
    """Tries the children of one node in order.

    Returns (index of the accepted child or -1, the residual R when the try
    stopped, the margins |r_i - a_i| of the tests made)."""
    R = np.asarray(p, dtype=np.float64).copy()
    q = np.asarray(q, dtype=np.float64)
    margins = []
    for i, (x, r) in enumerate(zip(child_tokens, child_uniforms)):
        x = int(x)
        a = 1.0 if q[x] <= 0.0 else min(1.0, R[x] / q[x])
        margins.append(abs(float(r) - a))
        if float(r) < a:
            return i, R, margins
        rest = np.maximum(R - q, 0.0)
        z = rest.sum()
        if z > 0.0:
            R = rest / z
    return -1, R, margins


def inverse_cdf(R: np.ndarray, v: float):
    """Smallest x with R[0] + ... + R[x] > v, and the distance of v from the
    two cumulative sums around it (its margin)."""
    c = np.cumsum(np.asarray(R, dtype=np.float64))
    x = int(np.searchsorted(c, float(v), side="right"))
    if x >= len(c):  # v at or beyond the total after rounding: the last token with mass
        nz = np.nonzero(np.asarray(R) > 0)[0]
        x = int(nz[-1]) if len(nz) else len(c) - 1
        return x, 0.0
    lo = c[x - 1] if x > 0 else 0.0
    return x, float(min(abs(float(v) - lo), abs(c[x] - float(v))))


def speculative_tree_accept(logits, draft_probs, tokens, parents, cu_nodes, temperature: float,
                            u_accept, u_bonus) -> Dict[str, object]:
    """Returns a dict with
      ``accepted_child`` int64 [T]: per node, the local index of its accepted
                         child, or -1 (leaves, and nodes whose children were all
                         rejected)
      ``accept_len``     int64 [B]
      ``accepted_nodes`` list of B lists of local node ids, root first
      ``bonus``          int64 [B]
      ``walk_margin``    float64 [B]: the smallest margin of the acceptance
                         tests made at the nodes of the walk
      ``bonus_margin``   float64 [B]: the distance of the bonus uniform from
                         the cumulative sums around the drawn token
      ``node_margin``    float64 [T]: per node the smallest margin of its
                         acceptance tests (inf for leaves)
      ``residual_z``     list of B float64 arrays: the distribution the bonus
                         was drawn from
    """
    logits = np.asarray(logits)
    T = logits.shape[0]
    B = len(cu_nodes) - 1
    acc_child = np.full(T, -1, dtype=np.int64)
    node_margin = np.full(T, np.inf)
    acc_len = np.zeros(B, dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    walk_margin = np.full(B, np.inf)
    bonus_margin = np.full(B, np.inf)
    residual_z = []
    paths: List[List[int]] = []
    for b in range(B):
        n0, n1 = int(cu_nodes[b]), int(cu_nodes[b + 1])
        n = n1 - n0
        par = [int(x) for x in parents[n0:n1]]
        children = [[] for _ in range(n)]
        for c in range(1, n):
            children[par[c]].append(c)
        residual = {}
        node_margins = {}
        for u in range(n):
            if not children[u]:
                continue
            p = target_probs(logits[n0 + u], temperature)
            i, R, m = node_verify(p, draft_probs[n0 + u], [tokens[n0 + c] for c in children[u]],
                                  [u_accept[n0 + c] for c in children[u]])
            if i >= 0:
                acc_child[n0 + u] = children[u][i]
            residual[u] = R
            node_margins[u] = m
            node_margin[n0 + u] = min(m)
        z = 0
        path = [0]
        mg = np.inf
        while True:
            if z in node_margins:
                mg = min(mg, min(node_margins[z]))
            nxt = int(acc_child[n0 + z])
            if nxt < 0:
                break
            z = nxt
            path.append(z)
        R = residual.get(z)
        if R is None:
            R = target_probs(logits[n0 + z], temperature)
        x, m = inverse_cdf(R, u_bonus[n0 + z])
        paths.append(path)
        acc_len[b] = len(path) - 1
        bonus[b] = x
        walk_margin[b] = mg
        bonus_margin[b] = m
        residual_z.append(R)
    return dict(accepted_child=acc_child, accept_len=acc_len, accepted_nodes=paths, bonus=bonus,
                walk_margin=walk_margin, bonus_margin=bonus_margin, node_margin=node_margin, residual_z=residual_z)
