"""Parity of sv_sample_accept (CUDA, through the C ABI) with the stochastic
acceptance oracle on the same seeded inputs: drafts near the target and flat,
temperatures 0.3 to 1.5, every workload's tree shape at full vocabulary, the
root-only tree, and the low-temperature limit against the greedy oracle.

Decisions are compared exactly where the oracle's float64 margin (distance of
the uniform from the acceptance threshold, or from the cumulative sums
around the bonus draw) exceeds what float32 sums over the vocabulary can move;
closer decisions may go either way, so there only validity is checked."""

import numpy as np
import pytest
import torch

import oracle
from synth import make_case, make_sampling_inputs
from tests.gpu_support import ensure_lib, i32

from speculative_decoding_tree_sv_gb300 import binding

pytestmark = pytest.mark.gpu

TOL_ACCEPT = 1e-4  # acceptance tests closer than this to their threshold may differ (float32 vs float64)
TOL_CDF = 2e-5     # float32 cumulative sums over the vocabulary move a draw by less than this


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _run(case, q, tokens, ua, ub, temperature, ws=None):
    dev = "cuda"
    T, V, B = case.total_nodes, case.vocab, case.batch
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    acc_child = torch.full((T,), -7, dtype=torch.int32, device=dev)
    alen = torch.full((B,), -7, dtype=torch.int32, device=dev)
    anodes = torch.full((B, case.max_depth + 1), -7, dtype=torch.int32, device=dev)
    bonus = torch.full((B,), -7, dtype=torch.int32, device=dev)
    if ws is None:
        ws = torch.zeros(binding.sv_sample_accept_workspace_size(B, T), dtype=torch.uint8, device=dev)
    binding.sv_sample_accept(f32(case.logits), f32(q), V, temperature, i32(tokens), i32(case.parents),
                             i32(case.cu_nodes), B, T, case.max_nodes, case.max_depth, f32(ua), f32(ub), acc_child,
                             alen, anodes, bonus, ws)
    torch.cuda.synchronize()
    return dict(acc_child=acc_child.cpu().numpy(), accept_len=alen.cpu().numpy(),
                accepted_nodes=anodes.cpu().numpy(), bonus=bonus.cpu().numpy(),
                err=binding.sv_get_device_error(ws), ws=ws)


def _compare(case, res, ref, ub, max_ambiguous=0.25):
    assert res["err"] == 0
    ambiguous = 0
    for b in range(case.batch):
        n0, n1 = int(case.cu_nodes[b]), int(case.cu_nodes[b + 1])
        # per node: the accepted child wherever its tests were clear
        for t in range(n0, n1):
            if ref["node_margin"][t] > TOL_ACCEPT:
                assert res["acc_child"][t] == ref["accepted_child"][t], (b, t - n0)
        path = [int(x) for x in res["accepted_nodes"][b][: res["accept_len"][b] + 1]]
        assert path[0] == 0 and (res["accepted_nodes"][b][len(path):] == -1).all()
        for a_, c_ in zip(path, path[1:]):      # a valid walk: every step is to a child
            assert int(case.parents[n0 + c_]) == a_
        x = int(res["bonus"][b])
        assert 0 <= x < case.vocab
        if ref["walk_margin"][b] <= TOL_ACCEPT:
            ambiguous += 1
            continue
        assert path == ref["accepted_nodes"][b], b
        assert res["accept_len"][b] == ref["accept_len"][b]
        if ref["bonus_margin"][b] > TOL_CDF:
            assert x == ref["bonus"][b], b
        else:
            # a draw within rounding of a boundary: the token's interval of the
            # float64 distribution must hold the uniform, up to that rounding
            c = np.cumsum(ref["residual_z"][b])
            v = float(ub[n0 + path[-1]])
            lo_c = c[x - 1] if x > 0 else 0.0
            assert lo_c - TOL_CDF <= v <= c[x] + TOL_CDF, (b, x, ref["bonus"][b])
    assert ambiguous <= max(1, max_ambiguous * case.batch), ambiguous


def _oracle(case, q, tokens, ua, ub, temperature):
    return oracle.speculative_tree_accept(case.logits, q.astype(np.float64), tokens, case.parents, case.cu_nodes,
                                          temperature, ua.astype(np.float64), ub.astype(np.float64))


@pytest.mark.parametrize("name,kw", [
    ("tiny", dict(batch=6)),
    ("llama8b_eagle", dict(layers=1, ctx=16)),
    ("specblock", dict(ctx=16, batch=4)),
])
@pytest.mark.parametrize("temperature", [0.7, 1.0])
@pytest.mark.parametrize("draft", ["near", "flat"])
def test_matches_oracle(name, kw, temperature, draft):
    case = make_case(name, **kw)
    for seed in range(2):
        q, tokens, ua, ub = make_sampling_inputs(case, seed=seed, draft=draft, sharpness=1.0 / temperature)
        res = _run(case, q, tokens, ua, ub, temperature)
        _compare(case, res, _oracle(case, q, tokens, ua, ub, temperature), ub)


def test_serving_mix_batch_and_temperatures():
    case = make_case("serving_mix", ctx=16)
    for temperature, seed in ((0.3, 5), (1.5, 6)):
        q, tokens, ua, ub = make_sampling_inputs(case, seed=seed, sharpness=1.0 / temperature)
        res = _run(case, q, tokens, ua, ub, temperature)
        _compare(case, res, _oracle(case, q, tokens, ua, ub, temperature), ub)


def test_root_only_trees_draw_from_the_target():
    case = make_case("tiny", batch=5, parents_list=[[-1]] * 5)
    q, tokens, ua, ub = make_sampling_inputs(case, seed=9)
    res = _run(case, q, tokens, ua, ub, 0.9)
    ref = _oracle(case, q, tokens, ua, ub, 0.9)
    assert (res["accept_len"] == 0).all()
    _compare(case, res, ref, ub)


def test_low_temperature_matches_greedy_acceptance():
    # planted paths, sibling tokens distinct, a flat draft: at T = 0.002 only
    # the target's arg-max can pass, so the walk is the greedy one
    case = make_case("llama8b_eagle", layers=1, ctx=16)
    q, _, ua, ub = make_sampling_inputs(case, seed=3, draft="flat")
    ua = np.minimum(ua, np.float32(0.999))
    ub = np.minimum(ub, np.float32(0.999))
    res = _run(case, q, case.tokens, ua, ub, 0.002)
    ref = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    np.testing.assert_array_equal(res["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(res["accept_len"], case.planted_len)
    np.testing.assert_array_equal(res["bonus"], ref["bonus"])
    for b in range(case.batch):
        assert list(res["accepted_nodes"][b][: res["accept_len"][b] + 1]) == ref["accepted_nodes"][b]


def test_workspace_reused_without_clearing():
    case = make_case("tiny", batch=4)
    q, tokens, ua, ub = make_sampling_inputs(case, seed=11)
    first = _run(case, q, tokens, ua, ub, 1.0)
    q2, tokens2, ua2, ub2 = make_sampling_inputs(case, seed=12)
    second = _run(case, q2, tokens2, ua2, ub2, 1.0, ws=first["ws"])
    _compare(case, second, _oracle(case, q2, tokens2, ua2, ub2, 1.0), ub2)


def test_bad_inputs_are_reported_not_trapped():
    # a walk deeper than max_depth, and a child token outside the vocabulary:
    # both are recorded in the error word; the call still returns
    case = make_case("tiny", batch=2)
    q = np.full((case.total_nodes, case.vocab), 1.0 / case.vocab, dtype=np.float32)
    ua = np.zeros(case.total_nodes, np.float32)        # every test passes (flat draft, r = 0)
    ub = np.full(case.total_nodes, 0.5, np.float32)
    tokens = np.zeros(case.total_nodes, np.int32)
    res = _run(case, q, tokens, ua, ub, 1.0)
    assert res["err"] == 0
    deep = int(res["accept_len"].max())
    assert deep >= 1
    # the same inputs with max_depth below the walk's depth
    short = make_case("tiny", batch=2)
    short.max_depth = deep - 1
    res = _run(short, q, tokens, ua, ub, 1.0)
    assert res["err"] == binding.SV_DEVERR_DEPTH
    # a token outside [0, vocab) is never accepted and is reported
    bad = tokens.copy()
    bad[1] = case.vocab + 5
    res = _run(case, q, bad, ua, ub, 1.0)
    assert res["err"] == binding.SV_DEVERR_BAD_TREE


def test_empty_tree_in_a_batch_is_reported_with_defined_outputs():
    case = make_case("tiny", batch=3)
    q, tokens, ua, ub = make_sampling_inputs(case, seed=21)
    # make the last sequence empty: its nodes are dropped from cu_nodes
    n_last = int(case.cu_nodes[3] - case.cu_nodes[2])
    T = int(case.cu_nodes[2])
    trimmed = make_case("tiny", batch=3)
    trimmed.cu_nodes = case.cu_nodes.copy()
    trimmed.cu_nodes[3] = trimmed.cu_nodes[2]   # total_nodes follows cu_nodes
    trimmed.logits = case.logits[:T]
    trimmed.parents = case.parents[:T]
    res = _run(trimmed, q[:T], tokens[:T], ua[:T], ub[:T], 1.0)
    assert res["err"] == binding.SV_DEVERR_BAD_TREE
    assert res["accept_len"][2] == 0 and res["bonus"][2] == -1
    assert (res["accepted_nodes"][2] == -1).all()
    two = make_case("tiny", batch=3)
    two.cu_nodes, two.batch = case.cu_nodes[:3].copy(), 2
    two.logits, two.parents = case.logits[:T], case.parents[:T]
    ref = _oracle(two, q[:T], tokens[:T], ua[:T], ub[:T], 1.0)
    for b in range(2):  # the other sequences are unaffected
        if ref["walk_margin"][b] > TOL_ACCEPT:
            assert list(res["accepted_nodes"][b][: res["accept_len"][b] + 1]) == ref["accepted_nodes"][b]
    assert n_last >= 1
