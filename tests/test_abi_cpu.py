"""The C-ABI library without a GPU: it builds, loads, exports every symbol
``include/sv.h`` declares, and rejects bad host arguments synchronously
(no CUDA call is made on these paths)."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from speculative_decoding_tree_sv_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "sv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:sv_status|int|const char\s*\*)\s+(sv_\w+)\s*\(", text, re.M)))


def test_header_declares_the_three_entry_points():
    names = _declared()
    for n in ("sv_tree_attention", "sv_greedy_accept", "sv_kv_commit"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        assert hasattr(lib, n)


def test_version_and_status_strings(lib):
    assert binding.sv_abi_version() == 2
    for code in range(7):
        s = binding.sv_status_string(code)
        assert s.startswith(binding.STATUS_NAMES[code])


def _fake_params(**over):
    # 16-byte aligned fake device addresses: host validation fails before use
    a = 1 << 20
    kw = dict(q=a, tree_k=a, tree_v=a, k_cache=a, v_cache=a, block_table=a, ctx_lens=a, cu_nodes=a,
              parents=a, out=a, workspace=a, workspace_bytes=1 << 30, total_nodes=60, max_nodes=60,
              batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, num_pages=300,
              max_pages_per_seq=300, num_splits=4)
    kw.update(over)
    return binding.make_attn_params(**kw)


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=96), 2),
    (dict(num_q_heads=24, num_kv_heads=8), 2),       # G = 3
    (dict(num_q_heads=30, num_kv_heads=8), 1),       # not divisible
    (dict(max_nodes=129), 2),
    (dict(q=None), 1),
    (dict(out=(1 << 20) + 8), 1),                    # misaligned
    (dict(page_size=32), 2),
    (dict(num_splits=65), 2),
    (dict(workspace_bytes=16), 4),
    (dict(kv_pages=1 << 20), 1),                     # list without prefix sums
    (dict(batch=0), 1),
    (dict(split_reduce=1), 1),                       # only 0 (auto) and 2 (partials) exist
    (dict(flags=16), 1),                             # unknown option bit
    (dict(flags=6), 1),                              # two kernels forced
    (dict(flags=10), 1),
    (dict(flags=12), 1),
])
def test_attention_host_validation(lib, over, status):
    p = _fake_params(**over)
    assert lib.sv_tree_attention(ctypes.byref(p), None) == status


def test_attention_workspace_size_with_explicit_splits(lib):
    p = _fake_params(num_splits=4)
    n = binding.sv_tree_attention_workspace_size(p)
    rows = 60 * 32
    assert n >= 256 + 4 * rows * 128 * 2 + 4 * rows * 4  # four splits' partials (bf16 O, fp32 lse)
    p2 = _fake_params(num_splits=4, split_reduce=2)
    assert binding.sv_tree_attention_workspace_size(p2) >= 256 + 4 * rows * 128 * 2 + 4 * rows * 4
    p1 = _fake_params(num_splits=1)
    assert binding.sv_tree_attention_workspace_size(p1) == 256


def test_attention_workspace_size_of_the_dealt_kernel(lib):
    # one CTA per SM (152 on GB300 when no device answers), two partial
    # pieces of 256 rows each: bf16 O / l and fp32 log2-sum-exp; a counter
    # per (sequence, KV head, 256-row group) and M tile, padded to 256 bytes
    p = _fake_params(num_splits=4, flags=binding.SV_ATTN_KERNEL_DEALT)
    rows = 152 * 2 * 256
    assert binding.sv_tree_attention_workspace_size(p) == 256 + rows * 128 * 2 + rows * 4 + 256


def test_attention_null_params(lib):
    assert lib.sv_tree_attention(None, None) == 1
    n = ctypes.c_size_t(0)
    assert lib.sv_tree_attention_workspace_size(None, ctypes.byref(n)) == 1


def test_accept_host_validation(lib):
    a = 1 << 20
    need = binding.sv_greedy_accept_workspace_size(4, 100)
    assert need >= 256 + 100 * 8 + 4 * 4
    f = lib.sv_greedy_accept
    assert f(None, 10, a, a, a, 1, 4, 4, 3, None, a, a, a, a, need, None) == 1
    assert f(a, 10, a, a, a, 1, 4, 129, 3, None, a, a, a, a, need, None) == 2
    assert f(a, 10, a, a, a, 4, 100, 4, 3, None, a, a, a, a, 16, None) == 4
    assert f(a, 0, a, a, a, 1, 4, 4, 3, None, a, a, a, a, need, None) == 1


def test_sample_accept_host_validation(lib):
    a = 1 << 20
    need = binding.sv_sample_accept_workspace_size(4, 100)
    assert need >= 256 + 100 * 4 * 2 + 100 * 129 * 4
    f = lib.sv_sample_accept

    def call(**kw):
        args = dict(logits=a, q=a, vocab=1000, temp=1.0, tokens=a, parents=a, cu=a, batch=4, total=100,
                    max_nodes=60, max_depth=8, ua=a, ub=a, acc=None, alen=a, anodes=a, bonus=a, ws=a,
                    ws_bytes=need)
        args.update(kw)
        return f(*args.values(), None)

    assert call(logits=None) == 1
    assert call(q=None) == 1
    assert call(ua=None) == 1
    assert call(temp=0.0) == 1                        # temperature must be positive
    assert call(temp=-1.0) == 1
    assert call(temp=float("inf")) == 1
    assert call(temp=float("nan")) == 1
    assert call(vocab=4) == 1                         # below one entry per CTA of a cluster
    assert call(max_nodes=129) == 2
    assert call(vocab=(1 << 18) + 1) == 2                 # eight 2^15-entry slices at most
    assert call(vocab=(1 << 24) + 1) == 2
    assert call(ws_bytes=need - 1) == 4
    assert call(total=0) == 0                         # nothing to do, nothing launched


def test_selftest_host_validation(lib):
    f = lib.sv_selftest_bounded_wait
    assert f(None, 0, None) == 1
    assert f(1 << 20, -1, None) == 1
    assert f(1 << 20, 2_000_000_000, None) == 1       # must abort before the wait's own limit


def test_commit_host_validation(lib):
    a = 1 << 20
    f = lib.sv_kv_commit
    base = [a, a, 1024, a, a, 4096, 2, 10, a, 4, a, a, a, a, 1, 3, 2, 64, 16]
    # new_ctx_lens aliasing ctx_lens is rejected
    args = base[:]
    assert f(*args, a, None, 0, None) == 1
    args = base[:]
    args[2] = 1001  # stride not a multiple of 8
    assert f(*args, None, None, 0, None) == 1
    args = base[:]
    args[17] = 60  # head_dim not a multiple of 8
    assert f(*args, None, None, 0, None) == 2
    args = base[:]
    assert f(*args, None, a, 8, None) == 4  # workspace too small


def test_retrieval_host_validation(lib):
    a = 1 << 20
    n = binding.sv_retrieve_pages_workspace_size(2, 8, 128, 100)
    assert n >= 256 + 2 * 8 * 2 * 128 * 4 + 2 * 100 * 4
    base = dict(q=a, summaries=a, block_table=a, ctx_lens=a, cu_nodes=a, kv_pages=a, cu_kv_pages=a, batch=2,
                num_q_heads=32, num_kv_heads=8, head_dim=128, num_pages=500, total_nodes=100,
                max_pages_per_seq=200, max_ctx_pages=100, sink_tokens=64, window_tokens=256, topk=8,
                kv_pages_capacity=2 * binding.retrieve_list_bound(64, 256, 8), workspace=a, workspace_bytes=n)

    def call(**over):
        kw = dict(base)
        kw.update(over)
        p = binding.make_retrieve_params(**kw)
        return lib.sv_retrieve_pages(ctypes.byref(p), None)

    assert call(head_dim=96) == 2
    assert call(page_size=32) == 2
    assert call(max_ctx_pages=20000, max_pages_per_seq=20000) == 2
    assert call(kv_pages_capacity=10) == 1
    assert call(workspace_bytes=16) == 4
    assert call(reduce=3) == 1
    assert call(q=None) == 1
    assert call(num_q_heads=30) == 1
    f = lib.sv_kv_page_summaries
    assert f(None, 10, 8, 128, 16, a, 4, a, None, 1, 4, a, None, 0, None) == 1
    assert f(a, 10, 8, 96, 16, a, 4, a, None, 1, 4, a, None, 0, None) == 2
    assert f(a, 10, 8, 128, 16, a, 4, a, None, 1, 4, a, a, 8, None) == 4


def test_host_tensors_are_refused_before_any_call(lib):
    import torch
    logits = torch.zeros(4, 8)                        # host memory
    with pytest.raises(ValueError):
        binding.sv_greedy_accept(logits, 8, 1 << 20, 1 << 20, 1 << 20, 1, 4, 4, 3, None, 1 << 20, 1 << 20,
                                 1 << 20, 1 << 20, workspace_bytes=4096)
    with pytest.raises(ValueError):
        binding.make_attn_params(q=torch.zeros(4, 8, 64, dtype=torch.bfloat16), tree_k=1 << 20, tree_v=1 << 20,
                                 k_cache=1 << 20, v_cache=1 << 20, block_table=1 << 20, ctx_lens=1 << 20,
                                 cu_nodes=1 << 20, parents=1 << 20, out=1 << 20, total_nodes=4, max_nodes=4,
                                 batch=1, num_q_heads=8, num_kv_heads=2, head_dim=64, num_pages=10,
                                 max_pages_per_seq=10)


def test_partial_list_extend_host_validation(lib):
    a = 1 << 20
    f = lib.sv_partial_list_extend
    assert f(None, a, a, a, 2, a, a, None, 0, None) == 1      # no refresh list
    assert f(a, a, a, a, 0, a, a, None, 0, None) == 1         # empty batch
    assert f(a, a, a, a, 2, None, a, None, 0, None) == 1      # no output list
    assert f(a, a, a, a, 2, a, a, a, 16, None) == 4           # workspace below its header


def test_specpv_full_trees_host_validation(lib):
    a = 1 << 20
    f = lib.sv_specpv_full_trees
    assert f(None, a, a, a, a, 2, a, a, a, None, 0, None) == 1   # no candidate parents
    assert f(a, a, a, a, None, 2, a, a, a, None, 0, None) == 1   # no buffer offsets
    assert f(a, a, a, a, a, 0, a, a, a, None, 0, None) == 1      # empty batch
    assert f(a, a, a, a, a, 2, a, a, None, None, 0, None) == 1   # no output offsets
    assert f(a, a, a, a, a, 2, a, a, a, a, 16, None) == 4        # workspace below its header
    assert f(a, a, a, a, a, 70000, a, a, a, None, 0, None) == 2  # batch beyond one grid dimension


def test_specpv_schedule_matches_the_oracle(lib):
    import oracle
    rng = np.random.default_rng(0)
    for trial in range(50):
        step_tokens = int(rng.integers(1, 10))
        limit = step_tokens + int(rng.integers(0, 30))
        commits = rng.integers(1, step_tokens + 1, size=20)
        want = oracle.specpv_schedule(commits, step_tokens, limit, ctx_len0=500)
        seq = binding.sv_specpv_seq()
        ctx, got = 500, []
        for c in commits:
            kind = binding.sv_specpv_next(seq, step_tokens, limit)
            got.append("full" if kind == binding.SV_VERIFY_FULL else "partial")
            ctx += int(c)
            binding.sv_specpv_after(seq, kind, ctx)
        assert got == want, trial
    seq = binding.sv_specpv_seq()
    with pytest.raises(binding.SvError):
        binding.sv_specpv_after(seq, binding.SV_VERIFY_PARTIAL, 10)  # no partial cache yet
