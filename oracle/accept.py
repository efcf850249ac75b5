"""Oracle for greedy (temperature 0) acceptance of a verified draft tree.

* SpecBlock, Appendix A.5 "Inference procedure": the longest accepted prefix
  is committed before the next verifier iteration.
* Temperature 0 (SpecBlock section 4 "Evaluation setup"; SpecPV Appendix D):
  the target's choice at a node is the arg-max of its logits.  Ties go to the
  lowest vocabulary index; -0.0 and +0.0 compare equal.  NaN is unsupported.
* "Dynamic Speculative Decoding", Implementation Details: the scheduler keeps
  ``accept_length + 1`` tokens per request, so the reported accept length
  excludes the bonus token the target emits after the last accepted node.

Reading of "longest accepted prefix" on a tree: a non-root node c matches when
its token equals the arg-max at its parent; it is accepted when it and every
non-root ancestor match.  The result is the accepted node of greatest depth;
among equally deep ones the root path that is lexicographically smallest as a
sequence of node indices wins.  ``accept_len`` is that depth (root and bonus
excluded) and the bonus token is the arg-max at that node.

Test infrastructure only.
"""

from __future__ import annotations

import numpy as np


def greedy_accept(logits, tokens, parents, cu_nodes):
    """Returns a dict with
      ``argmax``         int64 [T]  per-node arg-max (lowest index on ties)
      ``accept_len``     int64 [B]
      ``accepted_nodes`` list of B lists of local node ids, root first
      ``bonus``          int64 [B]
    """
    logits = np.asarray(logits)
    am = np.argmax(logits, axis=1)   # first occurrence of the maximum
    B = len(cu_nodes) - 1
    acc_len = np.zeros(B, dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    paths = []
    for b in range(B):
        n0, n1 = int(cu_nodes[b]), int(cu_nodes[b + 1])
        n = n1 - n0
        par = [int(x) for x in parents[n0:n1]]
        tok = [int(x) for x in tokens[n0:n1]]
        a = [int(x) for x in am[n0:n1]]
        depth = [0] * n
        accepted = [False] * n
        accepted[0] = True
        for c in range(1, n):
            p = par[c]
            depth[c] = depth[p] + 1
            accepted[c] = accepted[p] and tok[c] == a[p]

        def root_path(c):
            path = [c]
            while path[-1] != 0:
                path.append(par[path[-1]])
            return path[::-1]

        cands = [c for c in range(n) if accepted[c]]
        best = min(cands, key=lambda c: (-depth[c], root_path(c)))
        paths.append(root_path(best))
        acc_len[b] = depth[best]
        bonus[b] = a[best]
    return dict(argmax=am.astype(np.int64), accept_len=acc_len,
                accepted_nodes=paths, bonus=bonus)
