"""SpecPV partial verification on the GPU, driven by the library's schedule
(SpecPV section 3.3), against the oracle at every step.

The loop: a full verification attends the full KV cache; when partial steps
came before it, the partially verified tokens are prepended to the new
candidates (sv_specpv_full_trees), the step is verified at the refresh's
context length, and its commit rewrites the buffered slots.  After it, the
page summaries are rebuilt and the partial lists retrieved (page ids compared
with the oracle's).  Partial steps attend the refresh lists extended by the
pages the buffer grows into (each side extends its own lists), accept, and
commit.  Every step's attention is compared with the oracle's within the
attention tolerance, and its acceptance and the whole KV cache after its
commit bit for bit."""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_sv_gb300 import binding
from synth import bf16_bits_from_f32, make_case, node_depths
from tests.gpu_support import ATOL_ATTN, bf16, ensure_lib, i32

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


def _full_trees_gpu(cand_par, cand_tok, cand_cu, buf_tok, buf_cu):
    B = len(cand_cu) - 1
    total = int(cand_cu[-1]) + int(buf_cu[-1])
    par = torch.full((total + 4,), -9, dtype=torch.int32, device="cuda")
    tok = torch.full((total + 4,), -9, dtype=torch.int32, device="cuda")
    cu = torch.full((B + 1,), -9, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    bt = i32(buf_tok) if len(buf_tok) else None
    binding.sv_specpv_full_trees(i32(cand_par), i32(cand_tok), i32(cand_cu), bt, i32(buf_cu), B, par, tok, cu, ws)
    torch.cuda.synchronize()
    err = binding.sv_get_device_error(ws)
    cu_h = cu.cpu().numpy()
    return par.cpu().numpy()[:cu_h[-1]], tok.cpu().numpy()[:cu_h[-1]], cu_h, err, par.cpu().numpy()[total:]


def test_full_trees_match_oracle():
    rng = np.random.default_rng(9)
    from synth import tree_random_depth
    for trial in range(20):
        B = int(rng.integers(1, 9))
        sizes = [int(rng.integers(2, 40)) for _ in range(B)]
        trees = [tree_random_depth(rng, n, min(4, n - 1)) for n in sizes]  # a depth the size allows
        nbs = [int(rng.integers(0, 30)) if trial % 4 else 0 for _ in range(B)]
        cand_par = np.concatenate(trees).astype(np.int32)
        cand_tok = rng.integers(0, 50000, len(cand_par)).astype(np.int32)
        cand_cu = np.concatenate([[0], np.cumsum([len(t) for t in trees])]).astype(np.int32)
        buf_cu = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
        buf_tok = rng.integers(0, 50000, int(buf_cu[-1])).astype(np.int32)
        want = oracle.specpv_full_step_trees(cand_par, cand_tok, cand_cu, buf_tok, buf_cu)
        par, tok, cu, err, tail = _full_trees_gpu(cand_par, cand_tok, cand_cu, buf_tok, buf_cu)
        assert err == 0
        np.testing.assert_array_equal(cu, want[2])
        np.testing.assert_array_equal(par, want[0])
        np.testing.assert_array_equal(tok, want[1])
        assert (tail == -9).all()  # nothing written past the combined nodes


def test_full_trees_report_oversized_and_bad_trees():
    par = np.array([-1, 0, -1, 5], np.int32)  # second tree: node 1's parent 5 is not before it
    tok = np.arange(4, dtype=np.int32)
    cand_cu = np.array([0, 2, 4], np.int32)
    # 127 buffered tokens + 2 candidate nodes exceed 128 nodes
    buf_cu = np.array([0, 127, 127], np.int32)
    buf_tok = np.zeros(127, np.int32)
    _, _, _, err, _ = _full_trees_gpu(par[:2], tok[:2], cand_cu[:2], buf_tok, buf_cu[:2])
    assert err == binding.SV_DEVERR_BAD_TREE
    _, _, _, err, _ = _full_trees_gpu(par, tok, cand_cu, np.zeros(0, np.int32), np.array([0, 0, 0], np.int32))
    assert err == binding.SV_DEVERR_BAD_PARENT


# ------------------------------------------------------------ the loop

class _Loop:
    """Host mirror of one layer's KV cache and the token history."""

    def __init__(self, case, rng):
        self.c = case
        self.rng = rng
        self.kh = case.k_cache[0].copy()
        self.vh = case.v_cache[0].copy()
        self.dk = bf16(self.kh)
        self.dv = bf16(self.vh)
        self.V = case.vocab
        B = case.batch
        self.hist = [list(rng.integers(0, self.V, int(case.ctx_lens.max()) + 200)) for _ in range(B)]
        self.bt = i32(case.block_table)

    def rand_bf16(self, shape):
        return bf16_bits_from_f32(self.rng.standard_normal(shape).astype(np.float32))

    def check_cache(self):
        got_k = self.dk.view(torch.int16).cpu().numpy().view(np.uint16)
        got_v = self.dv.view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(got_k, self.kh)
        np.testing.assert_array_equal(got_v, self.vh)


def _planted_logits(rng, parents, tokens, cu, paths, V):
    T = len(parents)
    logits = (rng.standard_normal((T, V)) * 0.5).astype(np.float32)
    for b in range(len(cu) - 1):
        n0, n1 = int(cu[b]), int(cu[b + 1])
        kids = {i: [] for i in range(n1 - n0)}
        for i in range(1, n1 - n0):
            kids[int(parents[n0 + i])].append(i)
        nxt = {u: v for u, v in zip(paths[b], paths[b][1:])}
        for u in range(n1 - n0):
            if u in nxt:
                t = int(tokens[n0 + nxt[u]])
            else:
                taken = {int(tokens[n0 + k]) for k in kids[u]}
                t = int(rng.integers(0, V))
                while t in taken:
                    t = int(rng.integers(0, V))
            logits[n0 + u, t] = 10.0
    return logits


def _step(loop, parents, tokens, cu, ctx_lens, paths, kv_pages=None, cu_kv_pages=None):
    """One verify step of layer 0 on both sides: attention (compared within
    the tolerance), greedy acceptance and the commit (bit-exact)."""
    c, rng = loop.c, loop.rng
    T, B = len(parents), c.batch
    Hq, Hkv, D = c.num_q_heads, c.num_kv_heads, c.head_dim
    md = int(max(node_depths(parents[cu[b]:cu[b + 1]]).max() for b in range(B)))
    N_max = int(np.diff(cu).max())
    q, tk, tv = loop.rand_bf16((T, Hq, D)), loop.rand_bf16((T, Hkv, D)), loop.rand_bf16((T, Hkv, D))
    dq, dtk, dtv = bf16(q), bf16(tk), bf16(tv)
    dpar, dtok, dcu, dlens = i32(parents), i32(tokens), i32(cu), i32(ctx_lens)
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    max_kv = int(np.diff(cu_kv_pages).max()) if kv_pages is not None else 0
    # the device lists stay referenced until the call has run
    dkv = i32(kv_pages) if kv_pages is not None else None
    dckv = i32(cu_kv_pages) if kv_pages is not None else None
    p = binding.make_attn_params(q=dq, tree_k=dtk, tree_v=dtv, k_cache=loop.dk, v_cache=loop.dv,
                                 block_table=loop.bt, ctx_lens=dlens, cu_nodes=dcu, parents=dpar, out=out,
                                 total_nodes=T, max_nodes=N_max, kv_pages=dkv, cu_kv_pages=dckv,
                                 max_kv_pages=max_kv)
    ws = torch.zeros(binding.sv_tree_attention_workspace_size(p), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    binding.sv_tree_attention(p)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 0
    ref, _ = oracle.tree_verify_attention(q, tk, tv, loop.kh, loop.vh, c.block_table, ctx_lens, cu, parents,
                                          kv_pages=kv_pages, cu_kv_pages=cu_kv_pages)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= ATOL_ATTN
    # acceptance along the planted paths
    logits = _planted_logits(rng, parents, tokens, cu, paths, loop.V)
    acc_ref = oracle.greedy_accept(logits, tokens, parents, cu)
    assert [list(x) for x in acc_ref["accepted_nodes"]] == [list(x) for x in paths]
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    alen = torch.empty(B, dtype=torch.int32, device="cuda")
    anodes = torch.empty((B, md + 1), dtype=torch.int32, device="cuda")
    bonus = torch.empty(B, dtype=torch.int32, device="cuda")
    wsa = torch.zeros(binding.sv_greedy_accept_workspace_size(B, T), dtype=torch.uint8, device="cuda")
    binding.sv_greedy_accept(torch.from_numpy(logits).cuda(), loop.V, dtok, dpar, dcu, B, T, N_max, md, am, alen,
                             anodes, bonus, wsa)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(wsa) == 0
    np.testing.assert_array_equal(alen.cpu().numpy(), acc_ref["accept_len"])
    np.testing.assert_array_equal(bonus.cpu().numpy(), acc_ref["bonus"])
    an = anodes.cpu().numpy()
    for b in range(B):
        assert list(an[b, : acc_ref["accept_len"][b] + 1]) == acc_ref["accepted_nodes"][b]
    # the commit at ctx_lens, both sides
    new_lens = torch.empty(B, dtype=torch.int32, device="cuda")
    binding.sv_kv_commit(dtk, dtv, T * Hkv * D, loop.dk, loop.dv, c.num_pages * Hkv * 16 * D, 1, c.num_pages,
                         loop.bt, c.max_pages_per_seq, dlens, dcu, anodes, alen, B, md, Hkv, D, 16, new_lens, ws)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 0
    k2, v2, lens_ref = oracle.kv_commit(loop.kh[None], loop.vh[None], tk[None], tv[None], c.block_table, ctx_lens,
                                        cu, acc_ref["accepted_nodes"], acc_ref["accept_len"], 16)
    loop.kh, loop.vh = k2[0], v2[0]
    np.testing.assert_array_equal(new_lens.cpu().numpy(), lens_ref)
    loop.check_cache()
    # the history: the committed tokens from ctx_lens on
    for b in range(B):
        for j, node in enumerate(acc_ref["accepted_nodes"][b]):
            loop.hist[b][int(ctx_lens[b]) + j] = int(tokens[cu[b] + node])
    return np.asarray(lens_ref, np.int32), acc_ref["bonus"], q, cu


def _candidate_paths(parents_list, commit, rng):
    """A root path of depth commit - 1 in every candidate tree."""
    paths = []
    for par in parents_list:
        dep = node_depths(par)
        ends = np.nonzero(dep == commit - 1)[0]
        node = int(rng.choice(ends))
        path = [node]
        while path[-1] != 0:
            path.append(int(par[path[-1]]))
        paths.append(path[::-1])
    return paths


def _retrieve(loop, q, cu, lens, sink, window, topk, mcp):
    c = loop.c
    dlens = i32(lens)
    summ = torch.zeros((c.num_pages, c.num_kv_heads, 2, c.head_dim), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(binding.sv_retrieve_pages_workspace_size(c.batch, c.num_kv_heads, c.head_dim, mcp),
                     dtype=torch.uint8, device="cuda")
    binding.sv_kv_page_summaries(loop.dk, c.num_pages, c.num_kv_heads, c.head_dim, loop.bt, c.max_pages_per_seq,
                                 dlens, None, c.batch, mcp, summ, ws)
    cap = c.batch * binding.retrieve_list_bound(sink, window, topk)
    kv = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    kcu = torch.full((c.batch + 1,), -1, dtype=torch.int32, device="cuda")
    scores = torch.empty((c.batch, mcp), dtype=torch.float32, device="cuda")
    dq, dcu = bf16(q), i32(cu)  # referenced until the call has run
    p = binding.make_retrieve_params(
        q=dq, summaries=summ, block_table=loop.bt, ctx_lens=dlens, cu_nodes=dcu, kv_pages=kv,
        cu_kv_pages=kcu, batch=c.batch, num_q_heads=c.num_q_heads, num_kv_heads=c.num_kv_heads,
        head_dim=c.head_dim, num_pages=c.num_pages, total_nodes=int(cu[-1]), max_pages_per_seq=c.max_pages_per_seq,
        max_ctx_pages=mcp, sink_tokens=sink, window_tokens=window, topk=topk, scores=scores, workspace=ws)
    binding.sv_retrieve_pages(p)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(ws) == 0
    kcu_h = kcu.cpu().numpy()
    got = kv.cpu().numpy()[:kcu_h[-1]]
    want_kv, want_cu, sc = oracle.retrieve_pages(q, loop.kh, c.block_table, lens, cu, sink, window, topk)
    np.testing.assert_array_equal(kcu_h, want_cu)
    sc_gpu = scores.cpu().numpy()
    for b in range(c.batch):
        g, w = got[kcu_h[b]:kcu_h[b + 1]].tolist(), want_kv[want_cu[b]:want_cu[b + 1]].tolist()
        if g != w:  # only candidates fp32 cannot order may differ
            chosen = [p_ for p_ in w if p_ in sc[b]]
            kth = min(sc[b][p_] for p_ in chosen)
            for p_ in set(g) ^ set(w):
                assert p_ in sc[b] and abs(sc[b][p_] - kth) <= 2e-3 + 2e-4 * abs(kth), (b, p_)
        for p_, s_ in sc[b].items():
            assert abs(sc_gpu[b, p_] - s_) <= 1e-3 + 1e-4 * abs(s_)
    return got, kcu_h, want_kv, want_cu


def test_specpv_loop():
    sink, window, topk = 32, 128, 8
    case = make_case("serving_mix", batch=2, ctx=[2600, 2600], num_q_heads=8, num_kv_heads=2, head_dim=64,
                     with_logits=False, seed=77)
    B = case.batch
    cand_list = [case.parents[case.cu_nodes[b]:case.cu_nodes[b + 1]] for b in range(B)]
    cand_par, cand_cu = case.parents, case.cu_nodes
    step_tokens = case.max_depth + 1
    limit = step_tokens + 20
    rng = np.random.default_rng(5)
    commits = rng.integers(1, step_tokens + 1, size=14)
    start = case.ctx_lens.copy() - 160
    want_kinds = oracle.specpv_schedule(commits, step_tokens, limit, ctx_len0=int(start[0]))
    loop = _Loop(case, np.random.default_rng(6))
    mcp = (int(case.ctx_lens.max()) + 15) // 16
    seqs = [binding.sv_specpv_seq() for _ in range(B)]
    lens = start.copy()
    bonus = np.array([loop.hist[b][int(lens[b])] for b in range(B)], np.int32)
    ref_lens = None
    gpu_lists = ora_lists = None
    kinds, full_with_buffer = [], 0
    for s, commit in enumerate(commits):
        kind = binding.sv_specpv_next(seqs[0], step_tokens, limit)
        assert all(binding.sv_specpv_next(q_, step_tokens, limit) == kind for q_ in seqs)
        kinds.append("full" if kind == binding.SV_VERIFY_FULL else "partial")
        cand_tok = case.tokens.copy()
        for b in range(B):
            cand_tok[cand_cu[b]] = bonus[b]  # the step's root is the last bonus token
        cpaths = _candidate_paths(cand_list, int(commit), rng)
        if kind == binding.SV_VERIFY_FULL:
            R = lens.copy() if ref_lens is None else ref_lens.copy()
            nbs = (lens - R).astype(np.int32)
            buf_cu = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
            buf_tok = np.array([t for b in range(B) for t in loop.hist[b][int(R[b]):int(lens[b])]], np.int32)
            par, tok, cu, err, _ = _full_trees_gpu(cand_par, cand_tok, cand_cu, buf_tok, buf_cu)
            assert err == 0
            want = oracle.specpv_full_step_trees(cand_par, cand_tok, cand_cu, buf_tok, buf_cu)
            np.testing.assert_array_equal(par, want[0])
            np.testing.assert_array_equal(tok, want[1])
            np.testing.assert_array_equal(cu, want[2])
            full_with_buffer += int(nbs.sum() > 0)
            # the whole buffer is accepted again, then the candidate path
            paths = [list(range(int(nbs[b]))) + [int(nbs[b]) + x for x in cpaths[b]] for b in range(B)]
            new_lens, bonus, q, cu_used = _step(loop, par, tok, cu, R, paths)
            np.testing.assert_array_equal(new_lens, lens + int(commit))
            # refresh: summaries of the committed context, retrieval with this step's queries
            g_kv, g_cu, o_kv, o_cu = _retrieve(loop, q, cu_used, new_lens, sink, window, topk, mcp)
            gpu_lists, ora_lists = (g_kv, g_cu), (o_kv, o_cu)
            ref_lens = new_lens.copy()
        else:
            kv = torch.empty(B * (binding.retrieve_list_bound(sink, window, topk) + 64), dtype=torch.int32,
                             device="cuda")
            kcu = torch.empty(B + 1, dtype=torch.int32, device="cuda")
            binding.sv_partial_list_extend(i32(gpu_lists[0]), i32(gpu_lists[1]), i32(ref_lens), i32(lens), B, kv, kcu)
            torch.cuda.synchronize()
            g_cu = kcu.cpu().numpy()
            g_kv = kv.cpu().numpy()[:g_cu[-1]]
            o_kv, o_cu = oracle.extend_partial_lists(ora_lists[0], ora_lists[1], ref_lens, lens)
            np.testing.assert_array_equal(g_cu, o_cu)
            if np.array_equal(gpu_lists[0], ora_lists[0]):
                np.testing.assert_array_equal(g_kv, o_kv)
            w_kv, w_cu = oracle.extend_partial_lists(gpu_lists[0], gpu_lists[1], ref_lens, lens)
            np.testing.assert_array_equal(g_kv, w_kv)  # the extension itself, on the GPU's refresh lists
            new_lens, bonus, _, _ = _step(loop, cand_par, cand_tok, cand_cu, lens, cpaths, kv_pages=g_kv,
                                          cu_kv_pages=g_cu)
            np.testing.assert_array_equal(new_lens, lens + int(commit))
        lens = new_lens
        for q_ in seqs:
            binding.sv_specpv_after(q_, kind, int(lens[0]))
    assert kinds == want_kinds
    assert "partial" in kinds and kinds.count("full") >= 2 and full_with_buffer >= 1


def test_full_step_rejects_a_buffered_token():
    """The target disagrees with a partially verified token: the full step's
    path ends before it, the bonus is the target's own token, the slots up to
    there are rewritten and the length rolls back."""
    case = make_case("serving_mix", batch=2, ctx=[700, 900], num_q_heads=8, num_kv_heads=2, head_dim=64,
                     with_logits=False, seed=78)
    B = case.batch
    loop = _Loop(case, np.random.default_rng(11))
    rng = np.random.default_rng(12)
    R = case.ctx_lens - 20
    lens = case.ctx_lens.copy()
    nbs = (lens - R).astype(np.int32)
    buf_cu = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    buf_tok = np.array([t for b in range(B) for t in loop.hist[b][int(R[b]):int(lens[b])]], np.int32)
    cand_tok = case.tokens.copy()
    par, tok, cu, err, _ = _full_trees_gpu(case.parents, cand_tok, case.cu_nodes, buf_tok, buf_cu)
    assert err == 0
    cand_list = [case.parents[case.cu_nodes[b]:case.cu_nodes[b + 1]] for b in range(B)]
    cpaths = _candidate_paths(cand_list, 3, rng)
    # sequence 0 keeps its whole buffer; sequence 1's target rejects buffered token 7
    paths = [list(range(int(nbs[0]))) + [int(nbs[0]) + x for x in cpaths[0]], list(range(7))]
    new_lens, bonus, _, _ = _step(loop, par, tok, cu, R, paths)
    assert int(new_lens[0]) == int(lens[0]) + 3
    assert int(new_lens[1]) == int(R[1]) + 7  # rolled back: tokens from position R + 7 on are discarded
