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
