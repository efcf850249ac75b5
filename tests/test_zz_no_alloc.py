"""The workspace-free greedy acceptance (sv_greedy_accept_noalloc) against the
regular entry point, through the C ABI.

Callers that cannot allocate device memory while they verify (an engine that
gave its free memory to the KV pool, a plugin without an allocator, a decode
loop that forbids allocation after warm-up) use this variant; its scratch is
a fixed array inside the library.  Results must be identical to
sv_greedy_accept (acceptance is bit-exact), on two calls in a row, since the
array keeps the previous call's contents.  This file is collected last so a
run that stops at the first failure has already run every other test."""

import numpy as np
import pytest
import torch

from speculative_decoding_tree_sv_gb300 import binding
from synth import make_case
from tests.gpu_support import ensure_lib, i32

pytestmark = pytest.mark.gpu


def _outputs(case, dev="cuda"):
    T, B = case.total_nodes, case.batch
    return dict(am=torch.full((T,), -7, dtype=torch.int32, device=dev),
                alen=torch.full((B,), -7, dtype=torch.int32, device=dev),
                anodes=torch.full((B, case.max_depth + 1), -7, dtype=torch.int32, device=dev),
                bonus=torch.full((B,), -7, dtype=torch.int32, device=dev))


def _inputs(case):
    return (torch.from_numpy(case.logits).cuda(), i32(case.tokens), i32(case.parents), i32(case.cu_nodes))


def _regular(case):
    logits, tok, par, cu = _inputs(case)
    o = _outputs(case)
    ws = torch.zeros(binding.sv_greedy_accept_workspace_size(case.batch, case.total_nodes), dtype=torch.uint8,
                     device="cuda")
    binding.sv_greedy_accept(logits, case.vocab, tok, par, cu, case.batch, case.total_nodes, case.max_nodes,
                             case.max_depth, o["am"], o["alen"], o["anodes"], o["bonus"], ws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


def _no_alloc(case):
    logits, tok, par, cu = _inputs(case)
    o = _outputs(case)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    binding.sv_greedy_accept_noalloc(logits, case.vocab, tok, par, cu, case.batch, case.total_nodes,
                                     case.max_nodes, case.max_depth, o["am"], o["alen"], o["anodes"], o["bonus"],
                                     err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return {k: v.cpu().numpy() for k, v in o.items()}


def _same(a, b):
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_no_alloc_matches_regular_entry_point_on_consecutive_calls():
    ensure_lib()
    first = make_case("serving_mix", batch=6, ctx=16, vocab=20000, seed=77)
    second = make_case("specblock", batch=5, ctx=16, vocab=9000, seed=78)
    # two calls in a row on different trees: the shared array must not leak
    # one call's keys or tickets into the next
    for case in (first, second, first):
        _same(_no_alloc(case), _regular(case))
        np.testing.assert_array_equal(_no_alloc(case)["alen"], case.planted_len)


def test_no_alloc_rejects_sizes_beyond_its_array():
    lib = ensure_lib()
    a = 1 << 20
    # more than 8192 tree nodes or 1024 sequences: refused before any launch
    assert lib.sv_greedy_accept_noalloc(a, 10, a, a, a, 1, 8193, 4, 3, None, a, a, a, None, None) == 2
    assert lib.sv_greedy_accept_noalloc(a, 10, a, a, a, 1025, 4, 4, 3, None, a, a, a, None, None) == 2
