"""Pins of the SpecPV retrieval oracle (CPU): the summary score bounds every
key's dot product from above (brute force over the block's keys) and is
exact for one-token blocks; summaries cover valid tokens only; the three
reductions against explicit loops; the page list's structure; a planted
block is retrieved first; ties go to the lower page; retrieving every
candidate makes partial attention equal full attention."""

import numpy as np
import pytest

import oracle
from synth import bf16_bits_from_f32, make_case


def _bits(a):
    return bf16_bits_from_f32(np.asarray(a, dtype=np.float32))


def test_score_bounds_every_key_and_is_exact_for_one_key():
    rng = np.random.default_rng(0)
    for _ in range(200):
        d = 16
        keys = rng.standard_normal((int(rng.integers(1, 17)), d))
        q = rng.standard_normal(d)
        s = oracle.query_block_score(q, keys.max(axis=0), keys.min(axis=0))
        assert s >= max(float(q @ k) for k in keys) - 1e-12
        one = keys[:1]
        assert abs(oracle.query_block_score(q, one.max(axis=0), one.min(axis=0)) - float(q @ one[0])) < 1e-12


def test_score_is_the_max_over_the_box_corners():
    # brute force over every corner of the box [kmin, kmax] (d = 6)
    rng = np.random.default_rng(1)
    d = 6
    for _ in range(50):
        lo = rng.standard_normal(d)
        hi = lo + np.abs(rng.standard_normal(d))
        q = rng.standard_normal(d)
        corners = [np.where([(m >> j) & 1 for j in range(d)], hi, lo) for m in range(1 << d)]
        assert abs(oracle.query_block_score(q, hi, lo) - max(float(q @ c) for c in corners)) < 1e-12


def test_summaries_cover_valid_tokens_only():
    case = make_case("tiny", ctx=40, with_logits=False, seed=3)
    k = case.k_cache[0].copy()
    lp = 2  # logical page 2 holds tokens 32..39 (8 valid)
    phys = int(case.block_table[0, lp])
    k[phys, :, 8:, :] = _bits(np.full((k.shape[1], 8, k.shape[3]), 1e4))  # garbage past L
    summ, defined = oracle.page_summaries(k, case.block_table, case.ctx_lens)
    assert defined[phys]
    assert summ[phys, :, 0].max() < 100.0
    ref = oracle.bf16_to_f64(k[phys, :, :8, :])
    np.testing.assert_array_equal(summ[phys, :, 0], ref.max(axis=1))
    np.testing.assert_array_equal(summ[phys, :, 1], ref.min(axis=1))


@pytest.mark.parametrize("reduce", ["mean", "max", "last"])
def test_reductions_against_loops(reduce):
    rng = np.random.default_rng(7)
    n, hq, hkv, d, pages = 5, 8, 2, 16, 6
    q = rng.standard_normal((n, hq, d))
    summ = np.zeros((pages, hkv, 2, d))
    summ[:, :, 0] = np.abs(rng.standard_normal((pages, hkv, d)))
    summ[:, :, 1] = -np.abs(rng.standard_normal((pages, hkv, d)))
    got = oracle.block_importance(q, summ, list(range(pages)), hkv, reduce)
    g = hq // hkv
    for p in range(pages):
        per = np.array([[sum(max(q[i, h, j] * summ[p, h // g, 0, j], q[i, h, j] * summ[p, h // g, 1, j])
                             for j in range(d)) for h in range(hq)] for i in range(n)])
        want = {"mean": per.mean(), "max": per.max(), "last": per[-1].mean()}[reduce]
        assert abs(got[p] - want) < 1e-9


def test_last_reduction_ignores_other_nodes():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, 4, 8))
    summ = rng.standard_normal((3, 2, 2, 8))
    summ[:, :, 0], summ[:, :, 1] = np.maximum(summ[:, :, 0], summ[:, :, 1]), np.minimum(summ[:, :, 0], summ[:, :, 1])
    a = oracle.block_importance(q, summ, [0, 1, 2], 2, "last")
    q2 = q.copy()
    q2[:3] = rng.standard_normal((3, 4, 8))
    np.testing.assert_array_equal(a, oracle.block_importance(q2, summ, [0, 1, 2], 2, "last"))


def test_regions():
    assert oracle.page_regions(1000, 64, 256) == (63, 4, 46)
    assert oracle.page_regions(40, 64, 256) == (3, 3, 3)      # all sink
    assert oracle.page_regions(0, 64, 256) == (0, 0, 0)
    assert oracle.page_regions(1000, 0, 0) == (63, 0, 62)     # the last (partial) page is the window


@pytest.mark.parametrize("reduce", ["mean", "max", "last"])
def test_list_structure(reduce):
    case = make_case("serving_mix", batch=3, ctx=(300, 900), with_logits=False, seed=21, num_q_heads=8,
                     num_kv_heads=2, head_dim=64)
    kv, cu, scores = oracle.retrieve_pages(case.q[0], case.k_cache[0], case.block_table, case.ctx_lens,
                                           case.cu_nodes, sink_tokens=32, window_tokens=148, topk=6, reduce=reduce)
    for b, L in enumerate(case.ctx_lens):
        lst = kv[cu[b]:cu[b + 1]].tolist()
        n_pages, sink, fw = oracle.page_regions(int(L), 32, 148)
        assert lst == sorted(set(lst))
        assert set(range(sink)) <= set(lst) and set(range(fw, n_pages)) <= set(lst)
        assert len(lst) == sink + min(6, fw - sink) + (n_pages - fw)
        chosen = [p for p in lst if sink <= p < fw]
        thr = min(scores[b][p] for p in chosen)
        assert all(scores[b][p] <= thr for p in scores[b] if p not in chosen)


def test_planted_block_is_retrieved_first():
    case = make_case("tiny", ctx=600, with_logits=False, seed=5)
    k = case.k_cache[0].copy()
    qf = oracle.bf16_to_f64(case.q[0])
    lp = 17
    phys = int(case.block_table[0, lp])
    for g in range(k.shape[1]):
        mean_q = qf[:, 4 * g:4 * g + 4].mean(axis=(0, 1))  # G = 4
        k[phys, g] = _bits(np.tile(32.0 * np.sign(mean_q), (16, 1)))
    kv, cu, _ = oracle.retrieve_pages(case.q[0], k, case.block_table, case.ctx_lens, case.cu_nodes,
                                      sink_tokens=16, window_tokens=64, topk=1, reduce="mean")
    assert lp in kv.tolist()


def test_ties_go_to_the_lower_page():
    case = make_case("tiny", ctx=320, with_logits=False, seed=6)
    k = case.k_cache[0].copy()
    a, b2 = int(case.block_table[0, 5]), int(case.block_table[0, 9])
    k[a] = _bits(np.full(k.shape[1:], 3.0))
    k[b2] = _bits(np.full(k.shape[1:], 3.0))
    qpos = case.q.copy()
    qpos[0] = _bits(np.abs(oracle.bf16_to_f64(case.q[0])))
    kv, _, sc = oracle.retrieve_pages(qpos[0], k, case.block_table, case.ctx_lens, case.cu_nodes,
                                      sink_tokens=0, window_tokens=0, topk=1, reduce="mean")
    assert sc[0][5] == sc[0][9] and 5 in kv.tolist() and 9 not in kv.tolist()


def test_retrieving_every_candidate_gives_full_attention():
    case = make_case("tiny", batch=2, ctx=[203, 64], with_logits=False, seed=8)
    kv, cu, _ = oracle.retrieve_pages(case.q[0], case.k_cache[0], case.block_table, case.ctx_lens,
                                      case.cu_nodes, sink_tokens=16, window_tokens=32, topk=1000)
    part, _ = oracle.tree_verify_attention(case.q[0], case.tree_k[0], case.tree_v[0], case.k_cache[0],
                                           case.v_cache[0], case.block_table, case.ctx_lens, case.cu_nodes,
                                           case.parents, kv_pages=kv, cu_kv_pages=cu)
    full, _ = oracle.tree_verify_attention(case.q[0], case.tree_k[0], case.tree_v[0], case.k_cache[0],
                                           case.v_cache[0], case.block_table, case.ctx_lens, case.cu_nodes,
                                           case.parents)
    np.testing.assert_allclose(part, full, rtol=0, atol=1e-12)


def test_planted_mistake_is_caught():
    # a score without the max (plain q . kmax) breaks the upper bound
    rng = np.random.default_rng(11)
    broken = 0
    for _ in range(100):
        keys = rng.standard_normal((8, 8))
        q = rng.standard_normal(8)
        wrong = float(q @ keys.max(axis=0))
        if wrong < max(float(q @ k) for k in keys) - 1e-12:
            broken += 1
    assert broken > 0


def test_schedule_full_then_partial_until_the_buffer_overflows():
    # SpecPV Appendix C: the limit is one step's tokens plus 20
    step_tokens, limit = 8, 8 + 20
    kinds = oracle.specpv_schedule([5] * 12, step_tokens, limit, ctx_len0=1000)
    # after a full step the buffer grows by 5 per partial step; a partial
    # step needs buffered + 8 <= 28 (only exceeding the limit forces a full
    # step), so five partial steps (0, 5, 10, 15, 20 buffered) fit and the
    # next (25 + 8 > 28) is full again
    assert kinds == ["full"] + ["partial"] * 5 + ["full"] + ["partial"] * 5


def test_schedule_limit_below_one_step_is_always_full():
    assert oracle.specpv_schedule([3] * 5, 8, 7, 100) == ["full"] * 5


def test_extended_lists_append_the_buffer_pages():
    kv, cu = oracle.extend_partial_lists([0, 5, 9, 10, 1, 2], [0, 4, 6], [170, 40], [200, 40])
    # sequence 0: pages 0..10 at the refresh (last page 10), now 13 pages
    assert kv[cu[0]:cu[1]].tolist() == [0, 5, 9, 10, 11, 12]
    assert kv[cu[1]:cu[2]].tolist() == [1, 2]


# ------------------------------------------------------------ SpecPV full step
# SpecPV section 3.3: before a full verification, the partially verified
# tokens are prepended to the new candidates and the full KV cache is used.

def _rand_tree(rng, n):
    from synth import tree_random_depth
    return tree_random_depth(rng, n, min(4, n - 1)) if n > 1 else np.array([-1], np.int32)


def test_full_tree_without_buffer_is_the_candidate_tree():
    rng = np.random.default_rng(3)
    for n in (1, 2, 9, 16):
        par = _rand_tree(rng, n)
        tok = rng.integers(0, 1000, n).astype(np.int32)
        p2, t2 = oracle.specpv_full_tree(par, tok, [])
        np.testing.assert_array_equal(p2, par)
        np.testing.assert_array_equal(t2, tok)


def test_full_tree_layout_by_hand():
    # candidate tree 0 -> {1, 2}, 1 -> {3}; buffered tokens 11, 12, 13
    par, tok = oracle.specpv_full_tree([-1, 0, 0, 1], [5, 6, 7, 8], [11, 12, 13])
    assert par.tolist() == [-1, 0, 1, 2, 3, 3, 4]
    assert tok.tolist() == [11, 12, 13, 5, 6, 7, 8]
    par, tok, cu = oracle.specpv_full_step_trees([-1, 0, -1, 0, 0], [1, 2, 3, 4, 5], [0, 2, 5], [9, 8, 7], [0, 1, 3])
    assert cu.tolist() == [0, 3, 8]
    assert par.tolist() == [-1, 0, 1, -1, 0, 1, 2, 2]
    assert tok.tolist() == [9, 1, 2, 8, 7, 3, 4, 5]


@pytest.mark.parametrize("R,nb,n", [(40, 5, 9), (0, 3, 6), (17, 1, 1), (33, 12, 16)])
def test_full_step_attention_chain_is_causal_and_candidates_see_the_buffer(R, nb, n):
    """Rows of the chain (buffered tokens and the step's root) equal causal
    attention over the context and the chain (torch SDPA); a candidate row
    sees the context, the whole chain and its own ancestors."""
    from tests.test_oracle_attention import _sdpa, _single_seq
    rng = np.random.default_rng(R * 100 + nb * 10 + n)
    cand = _rand_tree(rng, n)
    par, _ = oracle.specpv_full_tree(cand, np.zeros(n, np.int32), np.zeros(nb, np.int32))
    d = _single_seq(rng, R, par, 8, 2, 32)
    out, _ = oracle.tree_verify_attention(d["q"], d["tree_k"], d["tree_v"], d["k_cache"], d["v_cache"],
                                          d["block_table"], d["ctx_lens"], d["cu_nodes"], d["parents"])
    m = nb + n
    allowed = np.zeros((m, R + m), dtype=bool)
    allowed[:, :R] = True
    for i in range(nb + 1):  # chain rows: causal, bottom-right aligned
        allowed[i, R: R + i + 1] = True
    for i in range(1, n):  # candidate rows: the chain, then their own ancestors
        row = nb + i
        allowed[row, R: R + nb + 1] = True
        j = i
        while j != 0:
            allowed[row, R + nb + j] = True
            j = int(cand[j])
    np.testing.assert_allclose(out, _sdpa(d, allowed), rtol=0, atol=1e-12)


@pytest.mark.parametrize("R,nb,n", [(48, 7, 12), (5, 2, 3), (64, 20, 30)])
def test_full_step_with_unchanged_buffer_kv_equals_full_verification(R, nb, n):
    """If the buffered tokens' K/V in the cache were already exact, re-verifying
    them changes nothing: the candidate rows of the combined step at context
    length R equal plain full verification of the candidate tree at L = R + nb
    over a cache holding the chain's K/V in slots R .. L-1."""
    from tests.test_oracle_attention import _paged, _rand_bf16
    rng = np.random.default_rng(R + nb + n)
    Hq, Hkv, D = 8, 2, 32
    cand = _rand_tree(rng, n)
    par, _ = oracle.specpv_full_tree(cand, np.zeros(n, np.int32), np.zeros(nb, np.int32))
    m = nb + n
    L = R + nb
    kc = _rand_bf16(rng, (L, Hkv, D))
    vc = _rand_bf16(rng, (L, Hkv, D))
    q = _rand_bf16(rng, (m, Hq, D))
    tk = _rand_bf16(rng, (m, Hkv, D))
    tv = _rand_bf16(rng, (m, Hkv, D))
    tk[:nb], tv[:nb] = kc[R:], vc[R:]  # the chain's K/V = what the cache holds there
    kcache, table = _paged(rng, kc, m + 2)
    vcache = kcache.copy()
    for t in range(L):
        vcache[table[t // 16], :, t % 16, :] = vc[t]
    bt = table[None, :]
    combined, _ = oracle.tree_verify_attention(q, tk, tv, kcache, vcache, bt, np.array([R], np.int32),
                                               np.array([0, m], np.int32), par)
    plain, _ = oracle.tree_verify_attention(q[nb:], tk[nb:], tv[nb:], kcache, vcache, bt, np.array([L], np.int32),
                                            np.array([0, n], np.int32), cand)
    np.testing.assert_allclose(combined[nb:], plain, rtol=0, atol=1e-12)


def _plant(logits, node, token):
    logits[node, :] = 0.0
    logits[node, token] = 5.0


def test_full_step_acceptance_rechecks_the_buffer():
    """Greedy acceptance over the combined tree: a buffer the target agrees
    with is accepted again and the walk continues into the candidates; a
    buffered token the target now rejects ends the path there, with the
    target's own token as the bonus."""
    rng = np.random.default_rng(8)
    V, nb = 64, 5
    cand = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    cand_tok = np.array([0, 10, 11, 12, 13, 14], np.int32)
    buf = np.array([40, 41, 42, 43, 44], np.int32)
    par, tok = oracle.specpv_full_tree(cand, cand_tok, buf)
    m = len(par)
    cu = np.array([0, m], np.int32)
    logits = rng.standard_normal((m, V))
    # chain agrees: am[j] = token of node j + 1 along the chain and into the
    # candidate root's child 1 (token 10), then child 3 (token 12)
    for j in range(nb - 1):
        _plant(logits, j, buf[j + 1])
    _plant(logits, nb - 1, cand_tok[0])  # the step's root token follows the buffer
    _plant(logits, nb, 10)
    _plant(logits, nb + 1, 12)
    _plant(logits, nb + 3, 63)  # no child carries 63: the walk stops at node nb + 3
    for i in (nb + 2, nb + 4, nb + 5):
        _plant(logits, i, 62)
    acc = oracle.greedy_accept(logits, tok, par, cu)
    assert acc["accept_len"][0] == nb + 2
    assert acc["accepted_nodes"][0] == list(range(nb + 1)) + [nb + 1, nb + 3]
    assert acc["bonus"][0] == 63
    # the target disagrees with buffered token 3 (node 3): the path ends at node 2
    _plant(logits, 2, 7)
    acc = oracle.greedy_accept(logits, tok, par, cu)
    assert acc["accept_len"][0] == 2 and acc["accepted_nodes"][0] == [0, 1, 2] and acc["bonus"][0] == 7


def test_full_step_commit_rewrites_the_buffered_slots():
    """The commit of the combined step at context length R writes slots
    R .. R + a: the buffered slots get this forward's K/V, the accepted
    candidates follow, and the new length is L + a_cand + 1 when the whole
    buffer is accepted again."""
    rng = np.random.default_rng(12)
    Hkv, D, R, nb = 2, 8, 30, 4
    L = R + nb
    cand = np.array([-1, 0, 1, 0], np.int32)
    par, _ = oracle.specpv_full_tree(cand, np.zeros(4, np.int32), np.zeros(nb, np.int32))
    m = len(par)
    pages = 4
    k_cache = rng.integers(0, 1 << 16, (1, pages, Hkv, 16, D)).astype(np.uint16)
    v_cache = rng.integers(0, 1 << 16, (1, pages, Hkv, 16, D)).astype(np.uint16)
    tk = rng.integers(0, 1 << 16, (1, m, Hkv, D)).astype(np.uint16)
    tv = rng.integers(0, 1 << 16, (1, m, Hkv, D)).astype(np.uint16)
    bt = np.array([[2, 0, 3, 1]], np.int32)
    path = list(range(nb + 1)) + [nb + 1, nb + 2]  # the buffer, the root, two candidates
    a = len(path) - 1
    k2, v2, lens = oracle.kv_commit(k_cache, v_cache, tk, tv, bt, np.array([R], np.int32),
                                    np.array([0, m], np.int32), [path], [a], 16)
    assert int(lens[0]) == L + 2 + 1
    for j, node in enumerate(path):
        s = R + j
        np.testing.assert_array_equal(k2[0, bt[0, s // 16], :, s % 16], tk[0, node])
        np.testing.assert_array_equal(v2[0, bt[0, s // 16], :, s % 16], tv[0, node])
    untouched = [s for s in range(pages * 16) if not R <= s <= R + a]
    for s in untouched:
        np.testing.assert_array_equal(k2[0, bt[0, s // 16], :, s % 16], k_cache[0, bt[0, s // 16], :, s % 16])
