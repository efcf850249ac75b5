"""Pins for the attention oracle (CPU only).

Each check ties the oracle to something other than itself: torch's
scaled_dot_product_attention (a library routine) for chain trees (= causal
attention) and single-node trees (= decode attention), closed forms (constant
V, zero Q), invariants (full page list = full verification, relabelling the
tree, probability rows summing to one) and the SpecBlock Appendix A.2 mask
example.  A last test plants mistakes in the oracle and checks that these
pins catch them.
"""

import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attention as oatt
from synth import bf16_bits_from_f32, make_case, tree_random_depth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P = 16


def _f64(bits):
    # test-side decoding of bf16 bits, independent of the oracle's helper
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).astype(np.int16)).view(
        torch.bfloat16).to(torch.float64)


def _paged(rng, ctx_keys, extra_slots):
    """Scatter logical-order context K or V [L, Hkv, D] into a shuffled page
    pool; returns (cache [pages, Hkv, P, D], block_table row)."""
    L, Hkv, D = ctx_keys.shape
    npg = -(-(L + extra_slots) // P)
    perm = rng.permutation(npg + 3)
    cache = rng.integers(0, 1 << 16, size=(npg + 3, Hkv, P, D)).astype(np.uint16)
    cache &= np.uint16(0xBFFF)  # finite garbage in unused slots
    table = perm[:npg].astype(np.int32)
    for t in range(L):
        cache[table[t // P], :, t % P, :] = ctx_keys[t]
    return cache, table


def _rand_bf16(rng, shape):
    return bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32))


def _single_seq(rng, L, parents, Hq, Hkv, D):
    n = len(parents)
    kc = _rand_bf16(rng, (L, Hkv, D))
    vc = _rand_bf16(rng, (L, Hkv, D))
    kcache, table = _paged(rng, kc, n)
    # reuse the same permutation for V by writing V into a copy of the pool
    vcache = kcache.copy()
    for t in range(L):
        vcache[table[t // P], :, t % P, :] = vc[t]
    q = _rand_bf16(rng, (n, Hq, D))
    tk = _rand_bf16(rng, (n, Hkv, D))
    tv = _rand_bf16(rng, (n, Hkv, D))
    return dict(q=q, tree_k=tk, tree_v=tv, k_cache=kcache, v_cache=vcache,
                block_table=table[None, :], ctx_lens=np.array([L], np.int32),
                cu_nodes=np.array([0, n], np.int32), parents=np.asarray(parents, np.int32),
                kc=kc, vc=vc)


def _run_oracle(d, **kw):
    return oracle.tree_verify_attention(
        d["q"], d["tree_k"], d["tree_v"], d["k_cache"], d["v_cache"], d["block_table"],
        d["ctx_lens"], d["cu_nodes"], d["parents"], page_size=P, **kw)


def _sdpa(d, allowed, scale=None):
    """torch SDPA over the logical key sequence [context..., tree nodes...]."""
    n, Hq, D = d["q"].shape
    Hkv = d["tree_k"].shape[1]
    G = Hq // Hkv
    K = torch.cat([_f64(d["kc"]), _f64(d["tree_k"])])  # [L+n, Hkv, D]
    V = torch.cat([_f64(d["vc"]), _f64(d["tree_v"])])
    K = K.repeat_interleave(G, dim=1).permute(1, 0, 2)  # [Hq, L+n, D]
    V = V.repeat_interleave(G, dim=1).permute(1, 0, 2)
    Q = _f64(d["q"]).permute(1, 0, 2)  # [Hq, n, D]
    o = F.scaled_dot_product_attention(Q, K, V, attn_mask=torch.from_numpy(allowed), scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("L,n,Hq,Hkv,D", [(37, 9, 4, 2, 16), (64, 16, 8, 2, 64), (0, 12, 2, 1, 32), (5, 1, 4, 4, 8)])
def test_chain_tree_equals_causal_attention(L, n, Hq, Hkv, D):
    rng = np.random.default_rng(L * 1000 + n)
    d = _single_seq(rng, L, np.arange(-1, n - 1), Hq, Hkv, D)
    out, _ = _run_oracle(d)
    # bottom-right aligned causal mask: node i sits at position L + i
    allowed = np.arange(L + n)[None, :] <= (L + np.arange(n))[:, None]
    ref = _sdpa(d, allowed)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("L,Hq,Hkv,D", [(1, 8, 2, 64), (300, 32, 8, 128), (17, 4, 1, 16)])
def test_single_node_tree_equals_decode_attention(L, Hq, Hkv, D):
    rng = np.random.default_rng(L)
    d = _single_seq(rng, L, [-1], Hq, Hkv, D)
    out, _ = _run_oracle(d)
    ref = _sdpa(d, np.ones((1, L + 1), dtype=bool))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_custom_scale_matches_sdpa():
    rng = np.random.default_rng(7)
    d = _single_seq(rng, 40, [-1, 0, 0, 1, 2, 2], 4, 2, 32)
    out, _ = _run_oracle(d, sm_scale=0.05)
    allowed = np.ones((6, 46), dtype=bool)
    allowed[:, 40:] = False
    # explicit ancestor sets of this tree, written out by hand
    anc = {0: [0], 1: [0, 1], 2: [0, 2], 3: [0, 1, 3], 4: [0, 2, 4], 5: [0, 2, 5]}
    for i, js in anc.items():
        for j in js:
            allowed[i, 40 + j] = True
    ref = _sdpa(d, allowed, scale=0.05)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_random_tree_matches_sdpa_with_handwritten_mask():
    rng = np.random.default_rng(11)
    par = tree_random_depth(rng, 20, 5)
    d = _single_seq(rng, 33, par, 8, 4, 32)
    out, _ = _run_oracle(d)
    # ancestor sets by repeated parent lookup, written independently
    n = len(par)
    allowed = np.zeros((n, 33 + n), dtype=bool)
    allowed[:, :33] = True
    for i in range(n):
        chain = {i}
        frontier = i
        for _ in range(n):
            if frontier == 0:
                break
            frontier = int(par[frontier])
            chain.add(frontier)
        for j in chain:
            allowed[i, 33 + j] = True
    np.testing.assert_allclose(out, _sdpa(d, allowed), rtol=0, atol=1e-12)


def test_partial_with_every_page_equals_full():
    case = make_case("tiny", ctx=203, seed=5, with_logits=False)
    full, lse_f = oracle.tree_verify_attention(
        case.q[0], case.tree_k[0], case.tree_v[0], case.k_cache[0], case.v_cache[0],
        case.block_table, case.ctx_lens, case.cu_nodes, case.parents)
    pages = np.arange(-(-203 // P), dtype=np.int32)
    part, lse_p = oracle.tree_verify_attention(
        case.q[0], case.tree_k[0], case.tree_v[0], case.k_cache[0], case.v_cache[0],
        case.block_table, case.ctx_lens, case.cu_nodes, case.parents,
        kv_pages=pages, cu_kv_pages=np.array([0, len(pages)], np.int32))
    np.testing.assert_array_equal(full, part)
    np.testing.assert_array_equal(lse_f, lse_p)


def test_partial_list_equals_attention_over_listed_tokens():
    # a partial list is the same as full verification of a shorter context
    # holding exactly the listed tokens, in order (one continuous segment)
    rng = np.random.default_rng(3)
    L = 100  # last page (96..99) is partial
    pages = [0, 3, 6]
    d = _single_seq(rng, L, [-1, 0, 1, 0], 4, 2, 16)
    part, lse_p = _run_oracle(d, kv_pages=np.array(pages, np.int32), cu_kv_pages=np.array([0, 3], np.int32))
    keep = [t for p in pages for t in range(p * P, min(p * P + P, L))]
    assert len(keep) == 16 + 16 + 4
    d2 = _single_seq(np.random.default_rng(99), len(keep), [-1, 0, 1, 0], 4, 2, 16)
    d2.update(q=d["q"], tree_k=d["tree_k"], tree_v=d["tree_v"])
    d2["kc"], d2["vc"] = d["kc"][keep], d["vc"][keep]
    kcache, table = _paged(np.random.default_rng(5), d2["kc"], 4)
    vcache = kcache.copy()
    for t in range(len(keep)):
        vcache[table[t // P], :, t % P, :] = d2["vc"][t]
    d2.update(k_cache=kcache, v_cache=vcache, block_table=table[None, :])
    ref, lse_r = _run_oracle(d2)
    np.testing.assert_allclose(part, ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_p, lse_r, rtol=0, atol=1e-13)


def test_relabelling_tree_nodes_permutes_outputs():
    rng = np.random.default_rng(21)
    par = [-1, 0, 0, 1, 1, 2, 3, 3, 5]
    d = _single_seq(rng, 50, par, 4, 2, 32)
    out, lse = _run_oracle(d)
    # another topological numbering: depth first instead of breadth first
    children = {}
    for i in range(1, len(par)):
        children.setdefault(par[i], []).append(i)
    order = []

    def dfs(u):
        order.append(u)
        for c in children.get(u, []):
            dfs(c)
    dfs(0)
    new_of = {old: new for new, old in enumerate(order)}
    par2 = [-1 if old == 0 else new_of[par[old]] for old in order]
    d2 = dict(d)
    d2.update(parents=np.array(par2, np.int32), q=d["q"][order], tree_k=d["tree_k"][order],
              tree_v=d["tree_v"][order])
    out2, lse2 = _run_oracle(d2)
    np.testing.assert_allclose(out2, out[order], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse[order], rtol=0, atol=1e-13)


def test_constant_v_gives_constant_output():
    rng = np.random.default_rng(1)
    d = _single_seq(rng, 70, [-1, 0, 1, 1, 0], 4, 2, 16)
    c = bf16_bits_from_f32(np.array([0.375], np.float32))[0]
    d["tree_v"][:] = c
    d["v_cache"][:] = c
    out, _ = _run_oracle(d)
    np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-14)


def test_zero_q_gives_mean_of_visible_values_and_log_count_lse():
    rng = np.random.default_rng(2)
    par = [-1, 0, 1, 1, 0, 4]
    L = 45
    d = _single_seq(rng, L, par, 4, 2, 16)
    d["q"][:] = 0
    out, lse = _run_oracle(d)
    vc = _f64(d["vc"]).numpy()
    tv = _f64(d["tree_v"]).numpy()
    on_path = {0: [0], 1: [0, 1], 2: [0, 1, 2], 3: [0, 1, 3], 4: [0, 4], 5: [0, 4, 5]}
    for i, js in on_path.items():
        for h in range(4):
            g = h // 2
            vis = np.concatenate([vc[:, g, :], tv[js, g, :]])
            np.testing.assert_allclose(out[i, h], vis.mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[i, h] - math.log(L + len(js))) < 1e-13


def test_probability_rows_sum_to_one():
    rng = np.random.default_rng(4)
    par = tree_random_depth(rng, 12, 4)
    mask = oatt.visibility_mask(par, 30)
    q = rng.standard_normal((12, 16))
    k = rng.standard_normal((42, 16))
    p = oatt.attention_probabilities(q, k, mask, 0.25)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(p[~mask] == 0.0)


def _load_a2():
    parents, names, visible, masked = {}, {}, {}, {}
    with open(os.path.join(GOLDEN, "specblock_a2_mask.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "node":
                parents[int(t[1])] = int(t[3])
                names[int(t[1])] = t[2]
            elif t[0] == "visible":
                visible[int(t[1])] = [int(x) for x in t[2:]]
            elif t[0] == "masked":
                masked[int(t[1])] = [int(x) for x in t[2:]]
    return [parents[i] for i in range(len(parents))], visible, masked


def test_specblock_appendix_a2_mask_example():
    par, visible, masked = _load_a2()
    L = 5
    mask = oatt.visibility_mask(par, L)
    for row, cols in visible.items():
        assert mask[row, :L].all()
        for j in cols:
            assert mask[row, L + j]
        for j in masked[row]:
            assert not mask[row, L + j]
        assert sorted(cols + masked[row]) == list(range(len(par)))


def test_context_positions_partial_last_page():
    pos = oatt.context_positions(37, 16, [0, 2])
    assert list(pos) == list(range(0, 16)) + list(range(32, 37))
    assert len(oatt.context_positions(37, 16, [])) == 0
    assert len(oatt.context_positions(0, 16)) == 0


def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible oracle mistakes and check the pins above reject them."""
    rng = np.random.default_rng(8)
    d = _single_seq(rng, 20, np.arange(-1, 7), 4, 2, 16)
    allowed = np.arange(28)[None, :] <= (20 + np.arange(8))[:, None]
    ref = _sdpa(d, allowed)
    good = oracle.ancestor_or_self_mask

    def no_self(parents):
        m = good(parents)
        np.fill_diagonal(m, False)
        m[0, 0] = True
        return m

    def with_next_node(parents):
        m = good(parents)
        for i in range(len(parents) - 1):
            m[i, i + 1] = True
        return m

    for bad in (no_self, with_next_node):
        monkeypatch.setattr(oatt, "ancestor_or_self_mask", bad)
        out, _ = _run_oracle(d)
        assert np.abs(out - ref).max() > 1e-3
    monkeypatch.setattr(oatt, "ancestor_or_self_mask", good)
    out, _ = _run_oracle(d)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
