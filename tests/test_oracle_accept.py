"""Pins for the acceptance oracle (CPU only): brute-force enumeration of every
root-to-leaf path on thousands of tiny random trees (duplicate sibling tokens
and tied logits included), planted accepted paths of the generated
workloads, explicit arg-max tie cases and the accept-length convention of
"Dynamic Speculative Decoding"."""

import os

import numpy as np
import pytest

import oracle
from synth import make_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _first_max(row):
    # independent arg-max: the first position holding the row maximum
    best = max(row)
    for i, x in enumerate(row):
        if x == best:
            return i
    raise AssertionError


def _brute_force(logits, tokens, parents):
    """Enumerate root-to-leaf paths; walk each from the root while the next
    node's token equals the target's choice; keep the longest walk, ties to
    the lexicographically smallest node sequence."""
    n = len(parents)
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[parents[i]].append(i)
    best = None
    for leaf in range(n):
        if kids[leaf]:
            continue
        path = [leaf]
        while path[-1] != 0:
            path.append(parents[path[-1]])
        path.reverse()
        k = 0
        while k + 1 < len(path) and tokens[path[k + 1]] == _first_max(list(logits[path[k]])):
            k += 1
        cand = (-k, tuple(path[: k + 1]))
        if best is None or cand < best:
            best = cand
    depth, nodes = -best[0], list(best[1])
    return depth, nodes, _first_max(list(logits[nodes[-1]]))


def _random_tree(rng, n):
    return [-1] + [int(rng.integers(0, i)) for i in range(1, n)]


@pytest.mark.parametrize("seed_block", range(4))
def test_matches_brute_force_on_tiny_trees(seed_block):
    rng = np.random.default_rng(1000 + seed_block)
    for _ in range(800):
        B = int(rng.integers(1, 4))
        parents, tokens, rows, cu = [], [], [], [0]
        V = int(rng.integers(2, 5))
        for _b in range(B):
            n = int(rng.integers(1, 10))
            par = _random_tree(rng, n)
            tok = rng.integers(0, V, size=n).tolist()  # duplicate siblings allowed
            lg = rng.integers(-1, 2, size=(n, V)).astype(np.float32)  # many ties
            lg[lg == 0] = np.where(rng.random(int((lg == 0).sum())) < 0.5, -0.0, 0.0)
            parents += par
            tokens += tok
            rows.append(lg)
            cu.append(cu[-1] + n)
        logits = np.concatenate(rows)
        res = oracle.greedy_accept(logits, np.array(tokens), np.array(parents), np.array(cu))
        for b in range(B):
            sl = slice(cu[b], cu[b + 1])
            d, nodes, bonus = _brute_force(logits[sl], tokens[sl], parents[sl])
            assert res["accept_len"][b] == d
            assert res["accepted_nodes"][b] == nodes
            assert res["bonus"][b] == bonus
        for i in range(len(tokens)):
            assert res["argmax"][i] == _first_max(list(logits[i]))


def test_argmax_ties_and_signed_zero():
    logits = np.array([[1, 3, 3, 2], [-0.0, 0.0, -1, -2], [0.0, -0.0, -1, -2],
                       [-5, -4, -4, -9]], dtype=np.float32)
    res = oracle.greedy_accept(logits, np.array([0, 0, 0, 0]), np.array([-1, -1, -1, -1]),
                               np.array([0, 1, 2, 3, 4]))
    assert list(res["argmax"]) == [1, 0, 0, 1]


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("llama8b_eagle", dict(layers=1, ctx=16)),
    ("serving_mix", dict(batch=5, ctx=(20, 40), vocab=4000)),
    ("long_partial", dict(ctx=64, with_partial=False)),
    ("specblock", dict(batch=6, ctx=16, vocab=3000)),
])
def test_planted_paths_are_recovered(name, kw):
    case = make_case(name, **kw)
    res = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    np.testing.assert_array_equal(res["accept_len"], case.planted_len)
    for b in range(case.batch):
        assert res["accepted_nodes"][b] == case.planted_path[b]
    np.testing.assert_array_equal(res["bonus"], case.planted_bonus)


def test_duplicate_sibling_tokens_pick_longest_then_smallest_indices():
    # root has two children with the same token; only the second continues.
    parents = [-1, 0, 0, 2, 1]
    tokens = [9, 5, 5, 7, 3]
    logits = np.zeros((5, 10), dtype=np.float32)
    logits[0, 5] = 1  # root -> token 5 (matches nodes 1 and 2)
    logits[1, 0] = 1  # node 1 -> token 0 (node 4 has token 3: no match)
    logits[2, 7] = 1  # node 2 -> token 7 (node 3 matches)
    logits[3, 4] = 1
    logits[4, 2] = 1
    res = oracle.greedy_accept(logits, np.array(tokens), np.array(parents), np.array([0, 5]))
    assert res["accepted_nodes"][0] == [0, 2, 3]
    assert res["accept_len"][0] == 2 and res["bonus"][0] == 4
    # equal depth: the smaller node index wins
    logits[1, 3] = 2  # now node 4 (token 3) also matches under node 1
    res = oracle.greedy_accept(logits, np.array(tokens), np.array(parents), np.array([0, 5]))
    assert res["accepted_nodes"][0] == [0, 1, 4]


def test_root_only_tree():
    logits = np.array([[0.5, 2.0, 2.0]], dtype=np.float32)
    res = oracle.greedy_accept(logits, np.array([1]), np.array([-1]), np.array([0, 1]))
    assert res["accept_len"][0] == 0 and res["accepted_nodes"][0] == [0] and res["bonus"][0] == 1


def test_accept_length_convention_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "accept_length_convention.txt")) as f:
        for line in f:
            t = line.split()
            if t and not t[0].startswith("#"):
                vals[t[0]] = [int(x) for x in t[1:]]
    acc = vals["accept_length"]
    kept = [a + 1 for a in acc] + [1] * (vals["batch"][0] - len(acc))
    assert kept == vals["kept"]
    assert list(np.cumsum(kept) - 1) == vals["last_index"]
    # our convention: a step emits accept_len draft tokens plus the bonus
    case = make_case("tiny")
    res = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    path = res["accepted_nodes"][0]
    emitted = [int(case.tokens[n]) for n in path[1:]] + [int(res["bonus"][0])]
    assert len(emitted) == res["accept_len"][0] + 1
