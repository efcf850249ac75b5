"""Pins for the stochastic-acceptance oracle (oracle/sampling.py).

* The defining property of speculative sampling (SpecPV section 2: output
  distributed as the target's own samples): at one node whose k children are
  drawn independently from q, the emitted token (the accepted child's token,
  or the draw from the residual when all are rejected) follows p exactly.
  The test treats the oracle as a black box: each acceptance probability is
  recovered by bisection on the child's uniform and the residual by forcing
  every rejection, then the emitted distribution is summed over all child
  tuples and compared with p.
* A whole tree by Monte Carlo: the first emitted token after the root follows
  p_root.
* Temperature -> 0 with distinct sibling tokens reduces to the greedy rule
  (oracle.greedy_accept, pinned separately).
* q = p accepts the first child; a draft that only proposes a token the
  target cannot emit is always rejected and the bonus is drawn from p.
* Inverse CDF on a hand-computed distribution.
"""

import itertools

import numpy as np
import pytest

import oracle
from oracle.sampling import inverse_cdf, node_verify, speculative_tree_accept, target_probs


def test_inverse_cdf_hand_values():
    R = np.array([0.125, 0.25, 0.0, 0.375, 0.25])  # cumulative 0.125, 0.375, 0.375, 0.75, 1 (exact)
    assert inverse_cdf(R, 0.0)[0] == 0
    assert inverse_cdf(R, 0.1)[0] == 0
    assert inverse_cdf(R, 0.2)[0] == 1
    assert inverse_cdf(R, 0.375)[0] == 3      # not above 0.375 before index 3; index 2 has no mass
    assert inverse_cdf(R, 0.7)[0] == 3
    assert inverse_cdf(R, 0.76)[0] == 4
    assert inverse_cdf(R, 0.9999999)[0] == 4
    x, m = inverse_cdf(R, 0.2)
    assert x == 1 and abs(m - 0.075) < 1e-15


def test_target_probs_is_tempered_softmax():
    lg = np.array([1.0, 2.0, -1.0, 0.5])
    for T in (0.5, 1.0, 2.0):
        e = np.exp(lg / T)
        np.testing.assert_allclose(target_probs(lg, T), e / e.sum(), rtol=1e-14)


def _threshold(p, q, xs, i):
    """Acceptance probability of child i after children 0 .. i-1 were
    rejected, found by bisection on its uniform."""
    lo, hi = 0.0, 1.0
    rs = [1.0] * len(xs)
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        rs[i] = mid
        got, _, _ = node_verify(p, q, xs[: i + 1], rs[: i + 1])
        if got == i:
            lo = mid
        else:
            hi = mid
    return lo


def _emitted_distribution(p, q, k):
    V = len(p)
    out = np.zeros(V)
    for xs in itertools.product(range(V), repeat=k):
        w = float(np.prod([q[x] for x in xs]))
        if w == 0.0:
            continue
        surv = 1.0
        for i, x in enumerate(xs):
            a = _threshold(p, q, list(xs), i)
            out[x] += w * surv * a
            surv *= 1.0 - a
        _, R, _ = node_verify(p, q, list(xs), [1.0] * k)  # every child rejected
        out += w * surv * R
    return out


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_one_node_emits_the_target_distribution_exactly(k, seed):
    rng = np.random.default_rng(seed)
    V = 4
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.7)
    np.testing.assert_allclose(_emitted_distribution(p, q, k), p, atol=1e-9)


def test_one_node_with_draft_zeros_and_target_zeros():
    p = np.array([0.5, 0.0, 0.3, 0.2])
    q = np.array([0.0, 0.6, 0.1, 0.3])
    for k in (1, 2, 3):
        np.testing.assert_allclose(_emitted_distribution(p, q, k), p, atol=1e-9)


def test_tree_first_token_follows_the_root_target_by_monte_carlo():
    # root with 3 children, each child with 2 children; children drawn from
    # their parent's draft distribution; the first emitted token (the root's
    # accepted child token, else the bonus) must follow p_root
    rng = np.random.default_rng(7)
    V, T, trials = 5, 0.8, 20000
    parents = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)
    n = len(parents)
    logits = rng.normal(size=(n, V))
    q = rng.dirichlet(np.ones(V), size=n)
    p_root = target_probs(logits[0], T)
    counts = np.zeros(V)
    cu = np.array([0, n], np.int32)
    for _ in range(trials):
        tokens = np.zeros(n, np.int64)
        for c in range(1, n):
            tokens[c] = rng.choice(V, p=q[parents[c]])
        res = speculative_tree_accept(logits, q, tokens, parents, cu, T, rng.random(n), rng.random(n))
        path = res["accepted_nodes"][0]
        first = tokens[path[1]] if len(path) > 1 else res["bonus"][0]
        counts[first] += 1
    freq = counts / trials
    sigma = np.sqrt(p_root * (1 - p_root) / trials)
    assert np.all(np.abs(freq - p_root) <= 5 * sigma + 1e-9), (freq, p_root)


def _random_tree(rng, n):
    par = [-1]
    for i in range(1, n):
        par.append(int(rng.integers(0, i)))
    return np.array(par, np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_low_temperature_reduces_to_greedy(seed):
    rng = np.random.default_rng(100 + seed)
    V, B = 40, 3
    parts, toks, lgs = [], [], []
    cu = [0]
    for _ in range(B):
        n = int(rng.integers(1, 12))
        par = _random_tree(rng, n)
        lg = np.stack([rng.permutation(V) for _ in range(n)]).astype(np.float64)  # a unique arg-max per row
        tok = np.zeros(n, np.int64)
        for u in range(n):
            kids = [c for c in range(1, n) if par[c] == u]
            # distinct sibling tokens; the arg-max of u among them half of the time
            choice = rng.choice(V, size=len(kids), replace=False)
            if kids and rng.random() < 0.5 and int(np.argmax(lg[u])) not in choice:
                choice[int(rng.integers(0, len(kids)))] = int(np.argmax(lg[u]))
            for c, x in zip(kids, choice):
                tok[c] = x
        parts.append(par)
        toks.append(tok)
        lgs.append(lg)
        cu.append(cu[-1] + n)
    parents = np.concatenate(parts)
    tokens = np.concatenate(toks)
    logits = np.concatenate(lgs)
    T = len(tokens)
    q = np.full((T, V), 1.0 / V)
    res = speculative_tree_accept(logits, q, tokens, parents, np.array(cu), 0.01, rng.random(T) * 0.999,
                                  rng.random(T) * 0.999)
    ref = oracle.greedy_accept(logits, tokens, parents, np.array(cu))
    np.testing.assert_array_equal(res["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(res["bonus"], ref["bonus"])
    assert res["accepted_nodes"] == ref["accepted_nodes"]


def test_draft_equal_to_target_accepts_the_first_child():
    rng = np.random.default_rng(3)
    V, T = 30, 0.7
    parents = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    logits = rng.normal(size=(6, V))
    q = np.stack([target_probs(l, T) for l in logits])
    tokens = rng.integers(0, V, size=6)
    res = speculative_tree_accept(logits, q, tokens, parents, np.array([0, 6]), T, rng.random(6), rng.random(6))
    assert res["accepted_nodes"][0] == [0, 1, 3]  # always the first child: 0 -> 1 -> 3 (a leaf)


def test_draft_proposing_an_impossible_token_is_rejected():
    rng = np.random.default_rng(4)
    V, T = 16, 1.0
    parents = np.array([-1, 0, 0, 0], np.int32)
    logits = rng.normal(size=(4, V))
    logits[0, 5] = -1e30                      # the target cannot emit token 5
    q = np.zeros((4, V))
    q[:, 5] = 1.0                             # the draft only proposes it
    tokens = np.array([0, 5, 5, 5])
    for v in (0.01, 0.37, 0.93):
        ub = np.full(4, v)
        res = speculative_tree_accept(logits, q, tokens, parents, np.array([0, 4]), T, np.full(4, 0.5), ub)
        assert res["accept_len"][0] == 0
        assert res["bonus"][0] == inverse_cdf(target_probs(logits[0], T), v)[0]
