"""Failure detection without a GPU fault: the bounded mbarrier wait that every
kernel of the library uses is made to run out (a barrier nothing completes),
both by its time limit and by the abort flag another role raises.  The error
word must read SV_DEVERR_TIMEOUT, the host call must report it as a timeout,
and the context must stay usable: a normal call right after gives the
oracle's answer."""

import time

import numpy as np
import pytest
import torch

import oracle
from synth import make_case
from tests.gpu_support import ensure_lib, run_accept

from speculative_decoding_tree_sv_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _context_still_usable():
    case = make_case("tiny", batch=3)
    ref = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    res = run_accept(case)
    assert res["err"] == 0
    np.testing.assert_array_equal(res["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(res["bonus"], ref["bonus"])


def test_wait_runs_out_at_its_time_limit():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    binding.sv_selftest_bounded_wait(ws)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert binding.sv_get_device_error(ws) == binding.SV_DEVERR_TIMEOUT
    assert 1.5 <= elapsed <= 30.0, elapsed   # the 2 s limit, give or take the launch
    assert binding.sv_get_device_error(ws) == 0  # the read cleared it
    _context_still_usable()


@pytest.mark.parametrize("abort_ms", [1, 50])
def test_wait_gives_up_when_another_role_aborts(abort_ms):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    binding.sv_selftest_bounded_wait(ws, abort_after_ns=abort_ms * 1_000_000)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert binding.sv_get_device_error(ws) == binding.SV_DEVERR_TIMEOUT
    assert elapsed < 1.5, elapsed             # well before the time limit
    _context_still_usable()


def test_timeout_code_maps_to_the_timeout_status():
    import ctypes
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.sv_selftest_bounded_wait(ws, abort_after_ns=1_000_000)
    code = ctypes.c_int(0)
    st = binding.load().sv_get_device_error(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(code), None)
    assert st == 6 and code.value == binding.SV_DEVERR_TIMEOUT   # SV_ERR_TIMEOUT
