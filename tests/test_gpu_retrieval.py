"""Parity of the SpecPV retrieval kernels (CUDA, through the C ABI) with the
fp64 oracle: page summaries exactly (max and min of bf16 keys are bf16
values), incremental summaries after a commit equal a full rebuild, page
importance within fp32 accumulation error, and the partial lists equal the
oracle's except where two candidates' importances are too close for fp32 to
order (then the list must still be valid); the retrieved list drives
sv_tree_attention to the oracle's partial attention."""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_sv_gb300 import binding
from synth import make_case
from tests.gpu_support import ATOL_ATTN, DeviceCase, bf16, ensure_lib, i32, run_attention

pytestmark = pytest.mark.gpu

REDUCE = {"mean": binding.SV_REDUCE_MEAN, "max": binding.SV_REDUCE_MAX, "last": binding.SV_REDUCE_LAST}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _max_ctx_pages(case):
    return int(max(1, (int(np.max(case.ctx_lens)) + 15) // 16))


def _summaries(case, dc, li=0, first_page=None, ctx_lens=None, summ=None):
    c = case
    if summ is None:
        summ = torch.zeros((c.num_pages, c.num_kv_heads, 2, c.head_dim), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lens = dc.ctx_lens if ctx_lens is None else ctx_lens
    binding.sv_kv_page_summaries(dc.k_cache[li], c.num_pages, c.num_kv_heads, c.head_dim, dc.block_table,
                                 c.max_pages_per_seq, lens, first_page, c.batch, _max_ctx_pages(c), summ, ws)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 0
    return summ


def _retrieve(case, dc, summ, sink, window, topk, reduce, li=0):
    c = case
    mcp = _max_ctx_pages(c)
    cap = c.batch * binding.retrieve_list_bound(sink, window, topk)
    kv = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    cu = torch.full((c.batch + 1,), -1, dtype=torch.int32, device="cuda")
    scores = torch.empty((c.batch, mcp), dtype=torch.float32, device="cuda")
    ws = torch.zeros(binding.sv_retrieve_pages_workspace_size(c.batch, c.num_kv_heads, c.head_dim, mcp),
                     dtype=torch.uint8, device="cuda")
    p = binding.make_retrieve_params(
        q=dc.q[li], summaries=summ, block_table=dc.block_table, ctx_lens=dc.ctx_lens, cu_nodes=dc.cu_nodes,
        kv_pages=kv, cu_kv_pages=cu, batch=c.batch, num_q_heads=c.num_q_heads, num_kv_heads=c.num_kv_heads,
        head_dim=c.head_dim, num_pages=c.num_pages, total_nodes=c.total_nodes,
        max_pages_per_seq=c.max_pages_per_seq, max_ctx_pages=mcp, sink_tokens=sink, window_tokens=window,
        topk=topk, reduce=REDUCE[reduce], scores=scores, workspace=ws)
    binding.sv_retrieve_pages(p)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 0
    cu_h = cu.cpu().numpy()
    return kv.cpu().numpy()[:cu_h[-1]], cu_h, scores.cpu().numpy()


CASES = [
    ("tiny", dict(ctx=600, seed=31)),
    ("tiny", dict(batch=4, ctx=[0, 17, 300, 1000], seed=32)),
    ("serving_mix", dict(batch=3, ctx=(500, 1500), seed=33)),
    ("llama8b_eagle", dict(layers=1, ctx=4096, seed=34)),
]


@pytest.mark.parametrize("name,kw", CASES)
def test_page_summaries_exact(name, kw):
    case = make_case(name, with_logits=False, **kw)
    dc = DeviceCase(case, layers=[0])
    summ = _summaries(case, dc).float().cpu().numpy()
    ref, defined = oracle.page_summaries(case.k_cache[0], case.block_table, case.ctx_lens)
    assert defined.any()
    np.testing.assert_array_equal(summ[defined], ref[defined])


def test_summaries_after_a_commit_equal_a_rebuild():
    case = make_case("serving_mix", batch=3, ctx=(300, 700), with_logits=False, seed=35, extra_pages=4)
    dc = DeviceCase(case, layers=[0])
    summ = _summaries(case, dc)
    # append up to max_depth + 1 tokens per sequence (new keys in the cache), then refresh
    # only the pages from the old last page on
    rng = np.random.default_rng(1)
    old = case.ctx_lens.copy()
    add = rng.integers(1, case.max_depth + 2, size=case.batch)  # the slots the block table covers
    new = old + add
    k = case.k_cache[0].copy()
    for b in range(case.batch):
        for s in range(int(old[b]), int(new[b])):
            phys = int(case.block_table[b, s // 16])
            k[phys, :, s % 16, :] = rng.integers(0, 1 << 16, size=k.shape[1:2] + k.shape[3:], dtype=np.uint16) & 0x3FFF
    dc.k_cache = bf16(k[None])
    newd = i32(new)
    _summaries(case, dc, first_page=i32(old // 16), ctx_lens=newd, summ=summ)
    ref, defined = oracle.page_summaries(k, case.block_table, new)
    np.testing.assert_array_equal(summ.float().cpu().numpy()[defined], ref[defined])


def _check_lists(case, kv, cu, scores, sink, window, topk, reduce):
    ref_kv, ref_cu, ref_scores = oracle.retrieve_pages(case.q[0], case.k_cache[0], case.block_table, case.ctx_lens,
                                                       case.cu_nodes, sink, window, topk, reduce)
    np.testing.assert_array_equal(np.diff(cu), np.diff(ref_cu))
    for b in range(case.batch):
        got = kv[cu[b]:cu[b + 1]].tolist()
        want = ref_kv[ref_cu[b]:ref_cu[b + 1]].tolist()
        assert got == sorted(set(got))
        sc = ref_scores[b]
        for p_, s_ in sc.items():  # importance within fp32 accumulation error
            assert abs(scores[b, p_] - s_) <= 1e-3 + 1e-4 * abs(s_), (b, p_, scores[b, p_], s_)
        if got != want:
            # only candidates the fp32 scores cannot order may differ
            diff = set(got) ^ set(want)
            chosen = [p_ for p_ in want if p_ in sc]
            kth = min(sc[p_] for p_ in chosen)
            for p_ in diff:
                assert p_ in sc and abs(sc[p_] - kth) <= 2e-3 + 2e-4 * abs(kth), (b, p_)


@pytest.mark.parametrize("reduce", ["mean", "max", "last"])
@pytest.mark.parametrize("name,kw", CASES)
def test_retrieve_matches_oracle(name, kw, reduce):
    case = make_case(name, with_logits=False, **kw)
    dc = DeviceCase(case, layers=[0])
    summ = _summaries(case, dc)
    for sink, window, topk in [(64, 256, 8), (32, 148, 6), (0, 0, 3), (16, 64, 0), (64, 1024, 10000)]:
        kv, cu, scores = _retrieve(case, dc, summ, sink, window, topk, reduce)
        _check_lists(case, kv, cu, scores, sink, window, topk, reduce)


def test_long_context_retrieval_and_partial_attention():
    # the 60000-token workload: 64 sink tokens, 128 retrieved pages (the
    # budget of 32 blocks of 64 tokens), a 1024-token window
    case = make_case("long_partial", with_logits=False)
    dc = DeviceCase(case, layers=[0])
    summ = _summaries(case, dc)
    kv, cu, scores = _retrieve(case, dc, summ, 64, 1024, 128, "mean")
    _check_lists(case, kv, cu, scores, 64, 1024, 128, "mean")
    # the retrieved list drives the attention; compare with the oracle on
    # the same list, for two KV heads
    case.kv_pages, case.cu_kv_pages = kv.astype(np.int32), cu.astype(np.int32)
    dc2 = DeviceCase(case, layers=[0])
    out, _, _ = run_attention(dc2, 0, partial=True)
    ref, ref_lse = oracle.tree_verify_attention(case.q[0], case.tree_k[0], case.tree_v[0], case.k_cache[0],
                                                case.v_cache[0], case.block_table, case.ctx_lens, case.cu_nodes,
                                                case.parents, kv_pages=case.kv_pages, cu_kv_pages=case.cu_kv_pages,
                                                kv_heads=[1, 6])
    sel = ~np.isnan(ref_lse)
    assert np.abs(out - ref)[sel].max() <= ATOL_ATTN


def test_bad_page_is_reported():
    case = make_case("tiny", ctx=300, with_logits=False, seed=36)
    case.block_table = case.block_table.copy()
    case.block_table[0, 4] = case.num_pages + 7
    dc = DeviceCase(case, layers=[0])
    summ = torch.zeros((case.num_pages, case.num_kv_heads, 2, case.head_dim), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.sv_kv_page_summaries(dc.k_cache[0], case.num_pages, case.num_kv_heads, case.head_dim, dc.block_table,
                                 case.max_pages_per_seq, dc.ctx_lens, None, 1, _max_ctx_pages(case), summ, ws)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 3
