"""Parity of sv_tree_attention (CUDA, through the C ABI) with the fp64
oracle: |out - oracle| <= 2e-2 elementwise (bf16 inputs, fp32 accumulation),
log-sum-exp within 2e-3.  Covers the five workloads (sampled where the
oracle would take too long), several split counts, GQA groups 1..16, both
head sizes, ragged and empty contexts, root-only and 128-node chain trees,
partial page lists (empty, complete, SpecPV's small settings), batches on
both sides of the 64-sequence limit of longest-first dispatch, and the
device error word."""

import numpy as np
import pytest
import torch

import oracle
from synth import make_case, tree_chain
from speculative_decoding_tree_sv_gb300 import binding
from tests.gpu_support import ATOL_ATTN, ATOL_LSE, DeviceCase, ensure_lib, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _oracle(case, li=0, partial=False, seqs=None, kv_heads=None, sm_scale=None):
    return oracle.tree_verify_attention(
        case.q[li], case.tree_k[li], case.tree_v[li], case.k_cache[li], case.v_cache[li], case.block_table,
        case.ctx_lens, case.cu_nodes, case.parents, page_size=case.page_size,
        kv_pages=case.kv_pages if partial else None, cu_kv_pages=case.cu_kv_pages if partial else None,
        sm_scale=sm_scale, seqs=seqs, kv_heads=kv_heads)


def _compare(case, out, lse, ref, ref_lse, seqs=None, kv_heads=None):
    sel = ~np.isnan(ref_lse)
    if seqs is None and kv_heads is None:
        assert sel.all()
    assert sel.any()
    diff = np.abs(out - ref)[sel]
    assert np.isfinite(out[sel]).all()
    assert diff.max() <= ATOL_ATTN, f"max |diff| = {diff.max()}"
    if lse is not None:
        dl = np.abs(lse - ref_lse)[sel]
        assert dl.max() <= ATOL_LSE, f"max |lse diff| = {dl.max()}"


def _check(case, partial=False, num_splits=0, seqs=None, kv_heads=None, sm_scale=0.0, li=0, split_reduce=0,
           flags=0):
    dc = DeviceCase(case, layers=[li])
    out, lse, _ = run_attention(dc, 0, partial=partial, num_splits=num_splits, sm_scale=sm_scale,
                                split_reduce=split_reduce, flags=flags)
    ref, ref_lse = _oracle(case, li, partial, seqs, kv_heads, sm_scale=sm_scale if sm_scale > 0 else None)
    _compare(case, out, lse, ref, ref_lse, seqs, kv_heads)
    return out


# the library's choice, then each kernel forced
KERNELS = [0, binding.SV_ATTN_KERNEL_PAIRED, binding.SV_ATTN_KERNEL_WIDE, binding.SV_ATTN_KERNEL_DEALT]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits,mode", [(0, 0), (1, 0), (2, 2), (5, 2), (7, 2)])
def test_tiny(splits, mode, kernel):
    # more splits than tiles leaves some splits empty
    _check(make_case("tiny"), num_splits=splits, split_reduce=mode, flags=kernel)


@pytest.mark.parametrize("splits,mode", [(0, 0), (1, 0), (2, 2), (3, 2), (9, 2), (10, 2), (16, 2), (19, 2),
                                         (34, 2)])
@pytest.mark.parametrize("kernel", KERNELS)
def test_llama_eagle_layer(splits, mode, kernel):
    # 240 rows per KV head (a CTA pair sharing every K/V tile, or one
    # 256-row CTA); splits merge through workspace partials and a combine
    # kernel
    _check(make_case("llama8b_eagle", layers=1, with_logits=False), num_splits=splits, split_reduce=mode,
           flags=kernel)


@pytest.mark.parametrize("splits,mode", [(0, 0), (1, 0), (3, 2), (5, 2), (33, 2)])
@pytest.mark.parametrize("kernel", KERNELS)
def test_early_context_flag(splits, mode, kernel):
    # the context pages and index arrays are read before the wait on the
    # preceding grid; results are unchanged
    f = binding.SV_ATTN_EARLY_CONTEXT | kernel
    _check(make_case("llama8b_eagle", layers=1, with_logits=False), num_splits=splits, split_reduce=mode, flags=f)
    _check(make_case("tiny", batch=3, ctx=[0, 33, 200], with_logits=False, seed=5), num_splits=splits,
           split_reduce=mode, flags=f)


def test_early_context_back_to_back_layers():
    # consecutive launches on one stream overlap; every layer must still see
    # its own Q and write its own output
    case = make_case("llama8b_eagle", layers=4, with_logits=False)
    dc = DeviceCase(case)
    c = case
    outs = []
    ws = None
    params = []
    for li in range(4):
        out = torch.empty((c.total_nodes, c.num_q_heads, c.head_dim), dtype=torch.bfloat16, device="cuda")
        p = binding.make_attn_params(
            q=dc.q[li], tree_k=dc.tree_k[li], tree_v=dc.tree_v[li], k_cache=dc.k_cache[li],
            v_cache=dc.v_cache[li], block_table=dc.block_table, ctx_lens=dc.ctx_lens, cu_nodes=dc.cu_nodes,
            parents=dc.parents, out=out, total_nodes=c.total_nodes, max_nodes=c.max_nodes,
            flags=binding.SV_ATTN_EARLY_CONTEXT)
        if ws is None:
            ws = torch.zeros(binding.sv_tree_attention_workspace_size(p), dtype=torch.uint8, device="cuda")
        p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
        params.append(p)
        outs.append(out)
    for _ in range(3):
        for p in params:
            binding.sv_tree_attention(p)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 0
    for li in range(4):
        ref, _ = _oracle(case, li)
        diff = np.abs(outs[li].float().cpu().numpy() - ref).max()
        assert diff <= ATOL_ATTN, (li, diff)


@pytest.mark.parametrize("kernel", KERNELS)
def test_serving_mix_full_batch(kernel):
    _check(make_case("serving_mix", with_logits=False), flags=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_long_context_partial_and_full(kernel):
    case = make_case("long_partial", with_logits=False)
    _check(case, partial=True, flags=kernel)
    _check(case, partial=True, num_splits=12, split_reduce=2, flags=kernel)
    _check(case, partial=False, kv_heads=[0, 5], flags=kernel)
    _check(case, partial=False, kv_heads=[3], num_splits=16, split_reduce=2, flags=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_specblock_sampled(kernel):
    case = make_case("specblock", with_logits=False)
    _check(case, seqs=[0, 7, 15], kv_heads=[2, 6], flags=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_specblock_full_oracle_at_short_context(kernel):
    _check(make_case("specblock", ctx=300, with_logits=False), flags=kernel)


@pytest.mark.parametrize("ctx", [[0], [1], [15], [17], [127], [129], [1000], [0, 33, 16, 200]])
@pytest.mark.parametrize("kernel", KERNELS)
def test_ragged_and_empty_contexts(ctx, kernel):
    case = make_case("tiny", batch=len(ctx), ctx=ctx, seed=sum(ctx) + 7, with_logits=False)
    _check(case, num_splits=0, flags=kernel)
    _check(case, num_splits=3, flags=kernel)
    _check(case, num_splits=3, split_reduce=2, flags=kernel)


@pytest.mark.parametrize("batch", [64, 70])
@pytest.mark.parametrize("kernel", KERNELS)
def test_batch_order_limit_with_tied_lengths(batch, kernel):
    # up to 64 sequences are dispatched longest first (ties by index); more
    # are dispatched in index order; lengths repeat so the order has ties
    rng = np.random.default_rng(batch)
    ctx = [int(x) for x in rng.choice([0, 17, 128, 129, 300], size=batch)]
    case = make_case("tiny", batch=batch, ctx=ctx, seed=batch, with_logits=False)
    _check(case, flags=kernel)
    _check(case, num_splits=3, split_reduce=2, flags=kernel)


def test_root_only_tree_is_decode_attention():
    case = make_case("llama8b_eagle", layers=1, ctx=777, parents_list=[[-1]], with_logits=False)
    _check(case)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (8, 4, 64), (16, 8, 128), (64, 8, 128), (32, 2, 64)])
@pytest.mark.parametrize("kernel", KERNELS)
def test_group_sizes_and_head_dims(hq, hkv, d, kernel):
    case = make_case("serving_mix", batch=3, ctx=(40, 300), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                     with_logits=False, seed=hq * 100 + hkv)
    _check(case, flags=kernel)


def test_chain_of_128_nodes():
    case = make_case("tiny", num_q_heads=4, num_kv_heads=4, ctx=200, parents_list=[tree_chain(128)],
                     with_logits=False)
    _check(case)


@pytest.mark.parametrize("kernel", KERNELS)
def test_128_nodes_at_group_8_spans_four_row_groups(kernel):
    rng = np.random.default_rng(3)
    par = [-1] + [int(rng.integers(0, i)) for i in range(1, 128)]
    case = make_case("specblock", batch=2, ctx=[100, 40], parents_list=[par, par[:77]], with_logits=False)
    _check(case, flags=kernel)
    _check(case, num_splits=4, flags=kernel)
    _check(case, num_splits=4, split_reduce=2, flags=kernel)


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("kernel", KERNELS)
def test_partial_lists_small_settings(splits, kernel):
    # SpecPV Appendix D settings: 16-token blocks, 32 sink tokens, a 128-token
    # window plus a 20-token buffer (folded into the recent window).
    case = make_case("serving_mix", batch=4, ctx=(300, 900), with_logits=False,
                     partial=dict(sink=32, blocks=6, block_tokens=16, recent=148))
    _check(case, partial=True, num_splits=splits, flags=kernel)


def test_partial_all_pages_equals_full_and_empty_list():
    case = make_case("tiny", batch=3, ctx=[203, 0, 64], with_logits=False)
    lists = [np.arange(13), np.arange(0), np.arange(4)]
    case.kv_pages = np.concatenate(lists).astype(np.int32)
    case.cu_kv_pages = np.array([0, 13, 13, 17], np.int32)
    part = _check(case, partial=True)
    full = _check(case, partial=False)
    np.testing.assert_array_equal(part, full)
    # an empty list for every sequence: tree keys only
    case.kv_pages = np.zeros(1, np.int32)
    case.cu_kv_pages = np.zeros(4, np.int32)
    _check(case, partial=True)


def test_custom_scale():
    _check(make_case("tiny", seed=9, with_logits=False), sm_scale=0.05)


def test_bad_parent_is_reported_not_trapped():
    case = make_case("tiny", with_logits=False)
    case.parents = case.parents.copy()
    case.parents[5] = 9  # parent after the child
    dc = DeviceCase(case)
    _, _, err = run_attention(dc, 0, check_error=False)
    assert err == 2
    # the context stays usable
    good = make_case("tiny", with_logits=False)
    _check(good)


def test_bad_page_is_reported_not_trapped():
    case = make_case("tiny", with_logits=False)
    case.block_table = case.block_table.copy()
    case.block_table[0, 3] = case.num_pages + 100  # beyond the pool
    dc = DeviceCase(case)
    _, _, err = run_attention(dc, 0, check_error=False)
    assert err == 3
    torch.cuda.synchronize()


@pytest.mark.parametrize("nodes", [1, 2, 32])
@pytest.mark.parametrize("splits", [0, 1, 4])
@pytest.mark.parametrize("kernel", KERNELS)
def test_pair_with_an_empty_row_tile(nodes, splits, kernel):
    # the 60-node tree needs two 128-row tiles (a CTA pair sharing each K/V
    # tile); the small tree of the other sequence leaves the second CTA of
    # its pair without rows, and that CTA must still load and release its
    # half of every tile
    rng = np.random.default_rng(nodes)
    big = [-1] + [int(rng.integers(0, i)) for i in range(1, 60)]
    small = [-1] + list(range(nodes - 1))
    case = make_case("llama8b_eagle", layers=1, batch=2, ctx=[777, 300], parents_list=[big, small],
                     with_logits=False, seed=nodes + 11)
    for _ in range(2):
        _check(case, num_splits=splits, split_reduce=2 if splits > 1 else 0, flags=kernel)


@pytest.mark.parametrize("ctx", [[0], [17], [0, 0, 129], [5000]])
def test_dealt_ranges_narrower_than_a_tile(ctx):
    # a call whose total weight is below (or near) twice the CTA count: most
    # CTAs hold no tile or one 256-row tile (weight 2), some ranges fall
    # between two tile starts, and the combine must skip those CTAs
    case = make_case("llama8b_eagle", layers=1, batch=len(ctx), ctx=ctx, with_logits=False, seed=len(ctx) + 3)
    _check(case, flags=binding.SV_ATTN_KERNEL_DEALT)


def test_dealt_plan_reports_its_kernel():
    case = make_case("serving_mix", with_logits=False)
    dc = DeviceCase(case, layers=[0])
    c = case
    out = torch.empty((c.total_nodes, c.num_q_heads, c.head_dim), dtype=torch.bfloat16, device="cuda")
    p = binding.make_attn_params(q=dc.q[0], tree_k=dc.tree_k[0], tree_v=dc.tree_v[0], k_cache=dc.k_cache[0],
                                 v_cache=dc.v_cache[0], block_table=dc.block_table, ctx_lens=dc.ctx_lens,
                                 cu_nodes=dc.cu_nodes, parents=dc.parents, out=out, total_nodes=c.total_nodes,
                                 max_nodes=c.max_nodes, flags=binding.SV_ATTN_KERNEL_DEALT)
    splits, reduce, kernel = binding.sv_tree_attention_plan(p, with_kernel=True)
    assert (splits, reduce, kernel) == (1, 0, 2)


def test_dealt_workspace_left_ready_for_the_next_call():
    # cut units are merged by their last piece, which resets the unit's
    # counter: two calls on one workspace give the oracle's answer, and the
    # counters (the workspace's tail) are zero after each
    case = make_case("serving_mix", batch=5, ctx=(300, 2500), with_logits=False, seed=41)
    dc = DeviceCase(case, layers=[0])
    c = case
    ref, ref_lse = _oracle(case)
    out = torch.empty((c.total_nodes, c.num_q_heads, c.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.total_nodes, c.num_q_heads), dtype=torch.float32, device="cuda")
    p = binding.make_attn_params(q=dc.q[0], tree_k=dc.tree_k[0], tree_v=dc.tree_v[0], k_cache=dc.k_cache[0],
                                 v_cache=dc.v_cache[0], block_table=dc.block_table, ctx_lens=dc.ctx_lens,
                                 cu_nodes=dc.cu_nodes, parents=dc.parents, out=out, lse=lse,
                                 total_nodes=c.total_nodes, max_nodes=c.max_nodes, flags=binding.SV_ATTN_KERNEL_DEALT)
    n = binding.sv_tree_attention_workspace_size(p)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), n
    units = c.batch * c.num_kv_heads * ((c.max_nodes * (c.num_q_heads // c.num_kv_heads) + 255) // 256)
    for _ in range(2):
        out.fill_(float("nan"))
        binding.sv_tree_attention(p)
        torch.cuda.synchronize()
        assert binding.sv_get_device_error(ws) == 0
        _compare(case, out.float().cpu().numpy(), lse.cpu().numpy(), ref, ref_lse)
        tail = ws[n - ((units * 8 + 255) // 256) * 256:]
        assert int(tail.count_nonzero()) == 0
