"""Bit-exact parity of sv_greedy_accept and sv_kv_commit (CUDA, through the
C ABI) with the oracle: every workload's planted path, thousands of tiny
random trees with duplicate sibling tokens and tied logits, large trees
(60..128 nodes, depth up to 127) whose accepted paths tie for depth, ties across
vocabulary chunks, signed zeros, repeated calls on one workspace, and the
commit of every layer checked byte for byte with sentinel-filled caches."""

import numpy as np
import pytest
import torch

import oracle
from synth import make_case
from tests.gpu_support import DeviceCase, bf16, ensure_lib, i32, run_accept

from speculative_decoding_tree_sv_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _assert_accept_equal(res, ref, case):
    assert res["err"] == 0
    np.testing.assert_array_equal(res["argmax"], ref["argmax"])
    np.testing.assert_array_equal(res["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(res["bonus"], ref["bonus"])
    for b in range(case.batch):
        path = ref["accepted_nodes"][b]
        row = res["accepted_nodes"][b]
        assert list(row[: len(path)]) == path
        assert (row[len(path):] == -1).all()


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("llama8b_eagle", dict(layers=1, ctx=16)),
    ("serving_mix", dict(ctx=16)),
    ("long_partial", dict(ctx=64, with_partial=False)),
    ("specblock", dict(ctx=16)),
])
def test_workload_planted_paths(name, kw):
    case = make_case(name, **kw)
    ref = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    res = run_accept(case)
    _assert_accept_equal(res, ref, case)
    np.testing.assert_array_equal(res["accept_len"], case.planted_len)
    # the workspace was left ready: a second call gives the same answer
    res2 = run_accept(case)
    _assert_accept_equal(res2, ref, case)


class _Tiny:
    pass


def _tiny_batch(rng, B, V, int_logits=True):
    parents, tokens, rows, cu = [], [], [], [0]
    for _ in range(B):
        n = int(rng.integers(1, 10))
        par = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        parents += par
        tokens += rng.integers(0, V, size=n).tolist()
        if int_logits:
            lg = rng.integers(-1, 2, size=(n, V)).astype(np.float32)
            z = lg == 0
            lg[z] = np.where(rng.random(int(z.sum())) < 0.5, -0.0, 0.0)
        else:
            lg = rng.standard_normal((n, V)).astype(np.float32)
        rows.append(lg)
        cu.append(cu[-1] + n)
    c = _Tiny()
    c.logits = np.concatenate(rows)
    c.tokens = np.array(tokens, np.int32)
    c.parents = np.array(parents, np.int32)
    c.cu_nodes = np.array(cu, np.int32)
    c.batch, c.vocab = B, V
    c.total_nodes = cu[-1]
    c.max_nodes = int(np.diff(cu).max())
    c.max_depth = 8
    return c


@pytest.mark.parametrize("V", [3, 4, 8, 13])
def test_tiny_random_trees_with_ties_and_duplicates(V):
    rng = np.random.default_rng(V)
    for _ in range(40):
        c = _tiny_batch(rng, 64, V)
        ref = oracle.greedy_accept(c.logits, c.tokens, c.parents, c.cu_nodes)
        _assert_accept_equal(run_accept(c), ref, c)


def _big_batch(rng, B, V, shape):
    # trees of 60..128 nodes over a tiny vocabulary, so many accepted paths
    # tie for the greatest depth; "deep" trees hang each node up to three
    # places below the previous one (depth ~60) and match their parent's
    # arg-max nine times in ten, "chain" is a 128-node path whose every node
    # matches
    parents, tokens, rows, cu = [], [], [], [0]
    for _ in range(B):
        if shape == "chain":
            n = 128
            par = [-1] + list(range(n - 1))
        else:
            n = int(rng.integers(60, 129))
            if shape == "deep":
                par = [-1] + [max(0, i - 1 - int(rng.integers(0, 3))) for i in range(1, n)]
            else:
                par = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        lg = rng.standard_normal((n, V)).astype(np.float32)
        tok = rng.integers(0, V, size=n)
        if shape in ("chain", "deep"):
            best = np.argmax(lg[np.array(par[1:])], axis=1)
            keep = rng.random(n - 1) < (1.0 if shape == "chain" else 0.9)
            tok[1:] = np.where(keep, best, tok[1:])
        parents += par
        tokens += tok.tolist()
        rows.append(lg)
        cu.append(cu[-1] + n)
    c = _Tiny()
    c.logits = np.concatenate(rows)
    c.tokens = np.array(tokens, np.int32)
    c.parents = np.array(parents, np.int32)
    c.cu_nodes = np.array(cu, np.int32)
    c.batch, c.vocab = B, V
    c.total_nodes = cu[-1]
    c.max_nodes = int(np.diff(cu).max())
    depth = []
    for b in range(B):
        par = c.parents[cu[b]:cu[b + 1]]
        d = np.zeros(len(par), np.int64)
        for i in range(1, len(par)):
            d[i] = d[par[i]] + 1
        depth.append(int(d.max()))
    c.max_depth = max(depth)
    return c


@pytest.mark.parametrize("shape,V", [("random", 2), ("random", 3), ("deep", 2), ("deep", 3), ("chain", 5)])
def test_large_trees_with_many_tied_accepted_paths(shape, V):
    rng = np.random.default_rng(1000 + V + len(shape))
    for _ in range(4):
        c = _big_batch(rng, 16, V, shape)
        ref = oracle.greedy_accept(c.logits, c.tokens, c.parents, c.cu_nodes)
        if shape == "chain":
            assert (ref["accept_len"] == 127).all()
        _assert_accept_equal(run_accept(c), ref, c)


def test_ties_across_vocabulary_chunks_and_signed_zero():
    V = 20000
    lg = np.full((4, V), -3.0, dtype=np.float32)
    lg[0, [8191, 8192, 12345]] = 7.0        # lowest index wins across chunks
    lg[1, [19999, 16384]] = 2.0
    lg[2, :] = -0.0
    lg[2, [5, 9000]] = 0.0                 # all zeros: index 0
    lg[3, [3, 16383, 16384]] = 1.5
    c = _Tiny()
    c.logits, c.vocab, c.batch = lg, V, 4
    c.tokens = np.zeros(4, np.int32)
    c.parents = np.full(4, -1, np.int32)
    c.cu_nodes = np.arange(5, dtype=np.int32)
    c.total_nodes, c.max_nodes, c.max_depth = 4, 1, 0
    res = run_accept(c)
    assert list(res["argmax"]) == [8191, 16384, 0, 3]
    ref = oracle.greedy_accept(lg, c.tokens, c.parents, c.cu_nodes)
    _assert_accept_equal(res, ref, c)


def test_full_size_logits_planted_paths():
    for name in ("llama8b_eagle", "serving_mix", "specblock"):
        case = make_case(name, layers=1, ctx=16)
        ref = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
        _assert_accept_equal(run_accept(case), ref, case)


def test_workspace_reused_across_calls_and_unaligned_rows():
    """One workspace serves consecutive calls (the kernel resets its keys and
    tickets), and logits whose rows do not start on a 16-byte boundary take
    the plain-load path with the same answers."""
    case = make_case("serving_mix", ctx=16)
    ref = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    T, V, B = case.total_nodes, case.vocab, case.batch
    dev = "cuda"
    tokens, parents, cu = i32(case.tokens), i32(case.parents), i32(case.cu_nodes)
    ws = torch.zeros(binding.sv_greedy_accept_workspace_size(B, T), dtype=torch.uint8, device=dev)
    flat = torch.empty(T * V + 1, dtype=torch.float32, device=dev)
    flat[1:] = torch.from_numpy(case.logits).reshape(-1).to(dev)
    aligned = torch.from_numpy(case.logits).to(dev)
    for logits in (aligned, flat[1:].view(T, V), aligned):
        am = torch.full((T,), -7, dtype=torch.int32, device=dev)
        alen = torch.full((B,), -7, dtype=torch.int32, device=dev)
        anodes = torch.full((B, case.max_depth + 1), -7, dtype=torch.int32, device=dev)
        bonus = torch.full((B,), -7, dtype=torch.int32, device=dev)
        binding.sv_greedy_accept(logits, V, tokens, parents, cu, B, T, case.max_nodes, case.max_depth, am, alen,
                                 anodes, bonus, ws)
        torch.cuda.synchronize()
        res = dict(argmax=am.cpu().numpy(), accept_len=alen.cpu().numpy(), accepted_nodes=anodes.cpu().numpy(),
                   bonus=bonus.cpu().numpy(), err=binding.sv_get_device_error(ws))
        _assert_accept_equal(res, ref, case)
    # keys and tickets are back to zero after the last call
    assert int(ws[256:].count_nonzero()) == 0


def _commit_check(case, paths, alens, layers):
    dc = DeviceCase(case, layers=layers)
    L_ = len(layers)
    T, Hkv, D = case.total_nodes, case.num_kv_heads, case.head_dim
    md = case.max_depth
    anodes = np.full((case.batch, md + 1), -1, np.int32)
    for b, p in enumerate(paths):
        anodes[b, : len(p)] = p
    k_before = dc.k_cache.clone()
    new_lens = torch.full((case.batch,), -1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.sv_kv_commit(dc.tree_k, dc.tree_v, T * Hkv * D, dc.k_cache, dc.v_cache,
                         case.num_pages * Hkv * case.page_size * D, L_, case.num_pages, dc.block_table,
                         case.max_pages_per_seq, dc.ctx_lens, dc.cu_nodes, i32(anodes), i32(alens),
                         case.batch, md, Hkv, D, case.page_size, new_lens, ws)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 0
    k_ref, v_ref, lens_ref = oracle.kv_commit(case.k_cache[layers], case.v_cache[layers], case.tree_k[layers],
                                              case.tree_v[layers], case.block_table, case.ctx_lens,
                                              case.cu_nodes, paths, alens, case.page_size)
    got_k = dc.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    got_v = dc.v_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got_k, k_ref)
    np.testing.assert_array_equal(got_v, v_ref)
    np.testing.assert_array_equal(new_lens.cpu().numpy(), lens_ref)
    assert not torch.equal(k_before, dc.k_cache)


def test_commit_all_layers_llama_eagle():
    case = make_case("llama8b_eagle", layers=32, ctx=4096 - 3)  # slots cross a page boundary
    ref = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    _commit_check(case, ref["accepted_nodes"], ref["accept_len"], list(range(32)))


def test_commit_serving_mix_ragged():
    case = make_case("serving_mix", layers=1)
    ref = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    _commit_check(case, ref["accepted_nodes"], ref["accept_len"], [0])


def test_commit_bad_path_is_reported():
    case = make_case("tiny")
    dc = DeviceCase(case)
    T, Hkv, D = case.total_nodes, case.num_kv_heads, case.head_dim
    anodes = np.full((1, case.max_depth + 1), -1, np.int32)
    anodes[0, :3] = [0, 99, 1]  # node 99 does not exist
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    before = dc.k_cache.clone()
    binding.sv_kv_commit(dc.tree_k, dc.tree_v, T * Hkv * D, dc.k_cache, dc.v_cache,
                         case.num_pages * Hkv * 16 * D, 1, case.num_pages, dc.block_table,
                         case.max_pages_per_seq, dc.ctx_lens, dc.cu_nodes, i32(anodes), i32([2]), 1,
                         case.max_depth, Hkv, D, 16, None, ws)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 4
    # slots 0 and 2 of the path were written, slot 1 was skipped
    changed = (before != dc.k_cache).any(dim=-1).any(dim=2).sum().item()
    assert changed == 2


def _accept_call(case, cu_nodes, T, ws, max_depth=None):
    dev = "cuda"
    B, V = len(cu_nodes) - 1, case.vocab
    md = case.max_depth if max_depth is None else max_depth
    am = torch.full((T,), -7, dtype=torch.int32, device=dev)
    alen = torch.full((B,), -7, dtype=torch.int32, device=dev)
    anodes = torch.full((B, md + 1), -7, dtype=torch.int32, device=dev)
    bonus = torch.full((B,), -7, dtype=torch.int32, device=dev)
    binding.sv_greedy_accept(torch.from_numpy(case.logits[:T]).to(dev), V, i32(case.tokens[:T]),
                             i32(case.parents[:T]), i32(cu_nodes), B, T, case.max_nodes, md, am, alen, anodes,
                             bonus, ws)
    torch.cuda.synchronize()
    return dict(argmax=am.cpu().numpy(), accept_len=alen.cpu().numpy(), accepted_nodes=anodes.cpu().numpy(),
                bonus=bonus.cpu().numpy(), err=binding.sv_get_device_error(ws))


def test_empty_tree_in_a_batch_gets_defined_outputs():
    """A sequence with no nodes owns no row of the grid; it still gets
    accept_len 0, bonus -1 and a path of -1, the call reports a bad tree, and
    the other sequences keep the oracle's answers."""
    case = make_case("tiny", batch=3)
    cu = case.cu_nodes.copy()
    T = int(cu[2])
    cu[3] = cu[2]  # the last sequence is empty
    for empty_at in (2, 0):
        cu_e = cu.copy()
        if empty_at == 0:  # empty first sequence: its nodes are dropped at the front
            n0 = int(case.cu_nodes[1])
            sub = make_case("tiny", batch=3)
            sub.logits, sub.tokens, sub.parents = case.logits[n0:], case.tokens[n0:], case.parents[n0:]
            cu_e = np.concatenate([[0], case.cu_nodes[1:] - n0]).astype(np.int32)
            src, Tn = sub, int(cu_e[-1])
        else:
            src, Tn = case, T
        ws = torch.zeros(binding.sv_greedy_accept_workspace_size(3, Tn), dtype=torch.uint8, device="cuda")
        res = _accept_call(src, cu_e, Tn, ws)
        assert res["err"] == binding.SV_DEVERR_BAD_TREE
        assert res["accept_len"][empty_at] == 0 and res["bonus"][empty_at] == -1
        assert (res["accepted_nodes"][empty_at] == -1).all()
        others = [b for b in range(3) if b != empty_at]
        sub_cu = np.concatenate([[0], np.cumsum([cu_e[b + 1] - cu_e[b] for b in others])]).astype(np.int32)
        ref = oracle.greedy_accept(src.logits[:Tn], src.tokens[:Tn], src.parents[:Tn], sub_cu)
        for i, b in enumerate(others):
            assert res["accept_len"][b] == ref["accept_len"][i]
            assert res["bonus"][b] == ref["bonus"][i]
            assert list(res["accepted_nodes"][b][: ref["accept_len"][i] + 1]) == ref["accepted_nodes"][i]
        assert int(ws[256:].count_nonzero()) == 0  # keys and tickets reset


def test_oversized_tree_resets_its_keys_and_gets_defined_outputs():
    """A tree of more than 128 nodes (device cu_nodes disagreeing with the
    host's max_nodes) is not walked: defined outputs, a bad-tree report, and
    its arg-max keys return to zero, so the next call on the same workspace
    is right."""
    rng = np.random.default_rng(5)
    T, V = 150, 4096
    bad = _Tiny()
    bad.vocab, bad.max_nodes, bad.max_depth = V, 128, 12
    bad.logits = rng.standard_normal((T, V)).astype(np.float32)
    bad.tokens = rng.integers(0, V, T).astype(np.int32)
    bad.parents = np.concatenate([[-1], np.arange(T - 1)]).astype(np.int32)  # a chain of 140 ...
    bad.parents[140:] = np.arange(-1, 9)  # ... then a chain of 10 (local ids) from index 140
    cu_bad = np.array([0, 140, 150], np.int32)
    ws = torch.zeros(binding.sv_greedy_accept_workspace_size(2, T), dtype=torch.uint8, device="cuda")
    res = _accept_call(bad, cu_bad, T, ws)
    assert res["err"] == binding.SV_DEVERR_BAD_TREE
    assert res["accept_len"][0] == 0 and res["bonus"][0] == -1 and (res["accepted_nodes"][0] == -1).all()
    ref = oracle.greedy_accept(bad.logits[140:], bad.tokens[140:], bad.parents[140:], np.array([0, 10], np.int32))
    assert res["accept_len"][1] == ref["accept_len"][0] and res["bonus"][1] == ref["bonus"][0]
    assert int(ws[256:].count_nonzero()) == 0
    # the same workspace, a valid call
    good = make_case("tiny", batch=2)
    Tg = int(good.cu_nodes[-1])
    assert Tg <= T
    res2 = _accept_call(good, good.cu_nodes, Tg, ws)
    _assert_accept_equal(res2, oracle.greedy_accept(good.logits, good.tokens, good.parents, good.cu_nodes), good)


def test_commit_depth_error_keeps_the_length():
    """accept_len beyond max_depth commits nothing for that sequence and
    leaves its new length at L (cache and length agree)."""
    case = make_case("tiny")
    dc = DeviceCase(case)
    T, Hkv, D = case.total_nodes, case.num_kv_heads, case.head_dim
    md = case.max_depth
    anodes = np.full((1, md + 1), -1, np.int32)
    anodes[0, :2] = [0, 1]
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    new_lens = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    before_k, before_v = dc.k_cache.clone(), dc.v_cache.clone()
    binding.sv_kv_commit(dc.tree_k, dc.tree_v, T * Hkv * D, dc.k_cache, dc.v_cache,
                         case.num_pages * Hkv * 16 * D, 1, case.num_pages, dc.block_table,
                         case.max_pages_per_seq, dc.ctx_lens, dc.cu_nodes, i32(anodes), i32([md + 1]), 1,
                         md, Hkv, D, 16, new_lens, ws)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == binding.SV_DEVERR_DEPTH
    assert int(new_lens.item()) == int(case.ctx_lens[0])
    assert torch.equal(before_k, dc.k_cache) and torch.equal(before_v, dc.v_cache)
