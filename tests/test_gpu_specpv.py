"""SpecPV partial verification on the GPU, driven by the library's schedule
(SpecPV section 3.3): a full verification refreshes the page summaries and
retrieves the partial lists; partial steps attend those lists extended by
the pages the buffer of partially verified tokens grows into; overflowing
the buffer (one step's tokens + 20) forces the next full verification.  Each
step's lists are checked against the oracle's and its attention against the
oracle's attention over the same lists."""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_sv_gb300 import binding
from synth import make_case
from tests.gpu_support import ATOL_ATTN, DeviceCase, ensure_lib, i32, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def test_list_extension_matches_oracle():
    rng = np.random.default_rng(4)
    B = 5
    ref_lens = rng.integers(0, 900, size=B).astype(np.int32)
    lists = [sorted(set(rng.integers(0, max(1, (int(L) + 15) // 16), size=7).tolist()) | (
        {(int(L) + 15) // 16 - 1} if L > 0 else set())) for L in ref_lens]
    ref_cu = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int32)
    ref_pages = np.array([p for x in lists for p in x] or [0], dtype=np.int32)
    now = ref_lens + rng.integers(0, 60, size=B).astype(np.int32)
    want_kv, want_cu = oracle.extend_partial_lists(ref_pages, ref_cu, ref_lens, now)
    kv = torch.full((len(want_kv) + 8,), -1, dtype=torch.int32, device="cuda")
    cu = torch.full((B + 1,), -1, dtype=torch.int32, device="cuda")
    binding.sv_partial_list_extend(i32(ref_pages), i32(ref_cu), i32(ref_lens), i32(now), B, kv, cu)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cu.cpu().numpy(), want_cu)
    np.testing.assert_array_equal(kv.cpu().numpy()[:want_cu[-1]], want_kv)


def test_specpv_loop():
    sink, window, topk = 32, 128, 8
    # contexts grow by the committed tokens; the generator's block table
    # covers the largest length, and the loop starts 160 tokens below it
    case = make_case("serving_mix", batch=2, ctx=[2600, 2600], num_q_heads=8, num_kv_heads=2, head_dim=64,
                     with_logits=False, seed=77)
    start = case.ctx_lens.copy() - 160
    step_tokens = case.max_depth + 1
    limit = step_tokens + 20
    rng = np.random.default_rng(5)
    commits = rng.integers(1, step_tokens + 1, size=14)
    want_kinds = oracle.specpv_schedule(commits, step_tokens, limit, ctx_len0=int(start[0]))
    dc = DeviceCase(case, layers=[0])
    c = case
    mcp = (int(case.ctx_lens.max()) + 15) // 16
    summ = torch.zeros((c.num_pages, c.num_kv_heads, 2, c.head_dim), dtype=torch.bfloat16, device="cuda")
    cap = c.batch * (binding.retrieve_list_bound(sink, window, topk) + 64)
    ref_kv = torch.empty(cap, dtype=torch.int32, device="cuda")
    ref_cu = torch.empty(c.batch + 1, dtype=torch.int32, device="cuda")
    kv = torch.empty(cap, dtype=torch.int32, device="cuda")
    cu = torch.empty(c.batch + 1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(binding.sv_retrieve_pages_workspace_size(c.batch, c.num_kv_heads, c.head_dim, mcp),
                     dtype=torch.uint8, device="cuda")
    seqs = [binding.sv_specpv_seq() for _ in range(c.batch)]
    lens = start.copy()
    ref_lens = None
    kinds = []
    for s, commit in enumerate(commits):
        kind = binding.sv_specpv_next(seqs[0], step_tokens, limit)
        assert all(binding.sv_specpv_next(q, step_tokens, limit) == kind for q in seqs)
        kinds.append("full" if kind == binding.SV_VERIFY_FULL else "partial")
        dlens = i32(lens)
        case.ctx_lens = lens.copy()
        if kind == binding.SV_VERIFY_FULL:
            # full attention, then refresh: summaries of every page, retrieval
            dc.ctx_lens = dlens
            out, _, _ = run_attention(dc, 0, partial=False)
            ref, _ = oracle.tree_verify_attention(c.q[0], c.tree_k[0], c.tree_v[0], c.k_cache[0], c.v_cache[0],
                                                  c.block_table, lens, c.cu_nodes, c.parents)
            assert np.abs(out - ref).max() <= ATOL_ATTN
            binding.sv_kv_page_summaries(dc.k_cache[0], c.num_pages, c.num_kv_heads, c.head_dim, dc.block_table,
                                         c.max_pages_per_seq, dlens, None, c.batch, mcp, summ, ws)
            p = binding.make_retrieve_params(
                q=dc.q[0], summaries=summ, block_table=dc.block_table, ctx_lens=dlens, cu_nodes=dc.cu_nodes,
                kv_pages=ref_kv, cu_kv_pages=ref_cu, batch=c.batch, num_q_heads=c.num_q_heads,
                num_kv_heads=c.num_kv_heads, head_dim=c.head_dim, num_pages=c.num_pages,
                total_nodes=c.total_nodes, max_pages_per_seq=c.max_pages_per_seq, max_ctx_pages=mcp,
                sink_tokens=sink, window_tokens=window, topk=topk, workspace=ws)
            binding.sv_retrieve_pages(p)
            torch.cuda.synchronize()
            ref_lens = lens.copy()
            want_kv, want_cu, sc = oracle.retrieve_pages(c.q[0], c.k_cache[0], c.block_table, lens, c.cu_nodes,
                                                         sink, window, topk)
            got_cu = ref_cu.cpu().numpy()
            np.testing.assert_array_equal(got_cu, want_cu)
        else:
            # partial attention over the refresh lists plus the buffer's pages
            binding.sv_partial_list_extend(ref_kv, ref_cu, i32(ref_lens), dlens, c.batch, kv, cu)
            torch.cuda.synchronize()
            got_cu = cu.cpu().numpy()
            got_kv = kv.cpu().numpy()[:got_cu[-1]]
            rk, rc = ref_kv.cpu().numpy(), ref_cu.cpu().numpy()
            want_kv, want_cu = oracle.extend_partial_lists(rk, rc, ref_lens, lens)
            np.testing.assert_array_equal(got_cu, want_cu)
            np.testing.assert_array_equal(got_kv, want_kv)
            case.kv_pages, case.cu_kv_pages = got_kv.astype(np.int32), got_cu.astype(np.int32)
            dc.ctx_lens, dc.kv_pages, dc.cu_kv_pages = dlens, i32(got_kv), i32(got_cu)
            out, _, _ = run_attention(dc, 0, partial=True)
            ref, _ = oracle.tree_verify_attention(c.q[0], c.tree_k[0], c.tree_v[0], c.k_cache[0], c.v_cache[0],
                                                  c.block_table, lens, c.cu_nodes, c.parents,
                                                  kv_pages=case.kv_pages, cu_kv_pages=case.cu_kv_pages)
            assert np.abs(out - ref).max() <= ATOL_ATTN
        lens = lens + int(commit)
        for q in seqs:
            binding.sv_specpv_after(q, kind, int(lens[0]))
    assert kinds == want_kinds
    assert "partial" in kinds and kinds.count("full") >= 2
