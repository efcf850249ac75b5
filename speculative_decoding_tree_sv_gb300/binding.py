"""ctypes binding of ``libsv.so`` (argument marshalling only).

The functions carry the names of the C entry points declared in
``include/sv.h``.  Tensor arguments may be torch tensors (their
``data_ptr()`` is passed) or raw integer device addresses; ``stream``
defaults to torch's current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels: if the library is not built, loading
fails with an error instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int, c_longlong, c_size_t, c_void_p
from typing import Optional

from . import build as _build

SV_OK = 0
STATUS_NAMES = {0: "SV_OK", 1: "SV_ERR_INVALID_ARG", 2: "SV_ERR_UNSUPPORTED", 3: "SV_ERR_CUDA",
                4: "SV_ERR_WORKSPACE", 5: "SV_ERR_DEVICE", 6: "SV_ERR_TIMEOUT"}
# device error codes (sv_deverr in include/sv.h)
SV_DEVERR_NONE, SV_DEVERR_TIMEOUT, SV_DEVERR_BAD_PARENT, SV_DEVERR_BAD_PAGE = 0, 1, 2, 3
SV_DEVERR_BAD_PATH, SV_DEVERR_DEPTH, SV_DEVERR_BAD_TREE = 4, 5, 6
SV_ATTN_EARLY_CONTEXT = 1
SV_ATTN_KERNEL_PAIRED = 2
SV_ATTN_KERNEL_WIDE = 4
SV_ATTN_KERNEL_DEALT = 8
DEVICE_ERRORS = {0: "none", 1: "timeout", 2: "bad parent", 3: "bad page", 4: "bad path", 5: "depth",
                 6: "bad tree"}


class SvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class sv_attn_params(ctypes.Structure):
    _fields_ = [
        ("batch", c_int), ("num_q_heads", c_int), ("num_kv_heads", c_int), ("head_dim", c_int),
        ("page_size", c_int), ("num_pages", c_int), ("total_nodes", c_int), ("max_nodes", c_int),
        ("max_pages_per_seq", c_int), ("max_kv_pages", c_int), ("num_splits", c_int),
        ("split_reduce", c_int), ("sm_scale", c_float), ("flags", c_int),
        ("q", c_void_p), ("tree_k", c_void_p), ("tree_v", c_void_p), ("k_cache", c_void_p),
        ("v_cache", c_void_p), ("block_table", c_void_p), ("ctx_lens", c_void_p),
        ("cu_nodes", c_void_p), ("parents", c_void_p), ("kv_pages", c_void_p),
        ("cu_kv_pages", c_void_p), ("out", c_void_p), ("lse", c_void_p), ("workspace", c_void_p),
        ("workspace_bytes", c_size_t),
    ]


class sv_retrieve_params(ctypes.Structure):
    _fields_ = [
        ("batch", c_int), ("num_q_heads", c_int), ("num_kv_heads", c_int), ("head_dim", c_int),
        ("page_size", c_int), ("num_pages", c_int), ("total_nodes", c_int), ("max_pages_per_seq", c_int),
        ("max_ctx_pages", c_int), ("sink_tokens", c_int), ("window_tokens", c_int), ("topk", c_int),
        ("reduce", c_int),
        ("q", c_void_p), ("summaries", c_void_p), ("block_table", c_void_p), ("ctx_lens", c_void_p),
        ("cu_nodes", c_void_p), ("kv_pages", c_void_p), ("cu_kv_pages", c_void_p), ("scores", c_void_p),
        ("kv_pages_capacity", c_size_t), ("workspace", c_void_p), ("workspace_bytes", c_size_t),
    ]


SV_REDUCE_MEAN, SV_REDUCE_MAX, SV_REDUCE_LAST = 0, 1, 2
SV_VERIFY_PARTIAL, SV_VERIFY_FULL = 0, 1


class sv_specpv_seq(ctypes.Structure):
    _fields_ = [("has_partial_cache", c_int), ("refresh_ctx_len", c_int), ("buffer_tokens", c_int)]

_LIB = None


def load(path: Optional[str] = None):
    """Load the built library (raises if it is missing)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libsv.so is not built ({path}); run __graft_entry__.build() or "
                           "python -m speculative_decoding_tree_sv_gb300.build")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.sv_abi_version.restype = c_int
    lib.sv_abi_version.argtypes = []
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_status_string.argtypes = [c_int]
    lib.sv_tree_attention_workspace_size.restype = c_int
    lib.sv_tree_attention_workspace_size.argtypes = [P(sv_attn_params), P(c_size_t)]
    lib.sv_tree_attention_plan.restype = c_int
    lib.sv_tree_attention_plan.argtypes = [P(sv_attn_params), P(c_int), P(c_int), P(c_int)]
    lib.sv_tree_attention.restype = c_int
    lib.sv_tree_attention.argtypes = [P(sv_attn_params), c_void_p]
    lib.sv_greedy_accept_workspace_size.restype = c_int
    lib.sv_greedy_accept_workspace_size.argtypes = [c_int, c_int, P(c_size_t)]
    lib.sv_greedy_accept.restype = c_int
    lib.sv_greedy_accept.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.sv_greedy_accept_noalloc.restype = c_int
    lib.sv_greedy_accept_noalloc.argtypes = [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                             c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.sv_sample_accept_workspace_size.restype = c_int
    lib.sv_sample_accept_workspace_size.argtypes = [c_int, c_int, P(c_size_t)]
    lib.sv_sample_accept.restype = c_int
    lib.sv_sample_accept.argtypes = [c_void_p, c_void_p, c_int, ctypes.c_float, c_void_p, c_void_p, c_void_p,
                                     c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.sv_selftest_bounded_wait.restype = c_int
    lib.sv_selftest_bounded_wait.argtypes = [c_void_p, c_longlong, c_void_p]
    lib.sv_kv_commit.restype = c_int
    lib.sv_kv_commit.argtypes = [c_void_p, c_void_p, c_longlong, c_void_p, c_void_p, c_longlong, c_int, c_int,
                                 c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                 c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.sv_kv_page_summaries.restype = c_int
    lib.sv_kv_page_summaries.argtypes = [c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_int, c_void_p, c_void_p,
                                         c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.sv_retrieve_pages_workspace_size.restype = c_int
    lib.sv_retrieve_pages_workspace_size.argtypes = [c_int, c_int, c_int, c_int, P(c_size_t)]
    lib.sv_retrieve_pages.restype = c_int
    lib.sv_retrieve_pages.argtypes = [P(sv_retrieve_params), c_void_p]
    lib.sv_partial_list_extend.restype = c_int
    lib.sv_partial_list_extend.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                           c_void_p, c_size_t, c_void_p]
    lib.sv_specpv_full_trees.restype = c_int
    lib.sv_specpv_full_trees.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.sv_specpv_next.restype = c_int
    lib.sv_specpv_next.argtypes = [P(sv_specpv_seq), c_int, c_int]
    lib.sv_specpv_after.restype = c_int
    lib.sv_specpv_after.argtypes = [P(sv_specpv_seq), c_int, c_int]
    lib.sv_set_trace_buffer.restype = c_int
    lib.sv_set_trace_buffer.argtypes = [c_void_p, c_size_t]
    lib.sv_get_device_error.restype = c_int
    lib.sv_get_device_error.argtypes = [c_void_p, P(c_int), c_void_p]
    if path == _build.library_path():
        _LIB = lib
    return lib


def _ptr(x) -> Optional[int]:
    """Address of a device buffer: None, a raw device address, or a CUDA
    tensor.  A tensor in host memory is refused here, before the library
    could hand its address to a kernel."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if getattr(x, "is_cuda", True) is False:
        raise ValueError(f"the library takes device memory; got a tensor on {x.device}")
    return int(x.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, where: str):
    if status != SV_OK:
        raise SvError(status, where)


def sv_abi_version() -> int:
    return load().sv_abi_version()


def sv_status_string(status: int) -> str:
    return load().sv_status_string(status).decode()


def make_attn_params(*, q, tree_k, tree_v, k_cache, v_cache, block_table, ctx_lens, cu_nodes, parents,
                     out, total_nodes: int, max_nodes: int, workspace=None, workspace_bytes: int = 0,
                     kv_pages=None, cu_kv_pages=None, max_kv_pages: int = 0, lse=None,
                     sm_scale: float = 0.0, num_splits: int = 0, split_reduce: int = 0, flags: int = 0,
                     page_size: int = 16, batch=None,
                     num_q_heads=None, num_kv_heads=None, head_dim=None, num_pages=None,
                     max_pages_per_seq=None) -> sv_attn_params:
    """Fill an ``sv_attn_params``; shapes come from torch tensors unless given."""
    p = sv_attn_params()
    p.batch = batch if batch is not None else int(block_table.shape[0])
    p.num_q_heads = num_q_heads if num_q_heads is not None else int(q.shape[1])
    p.num_kv_heads = num_kv_heads if num_kv_heads is not None else int(tree_k.shape[1])
    p.head_dim = head_dim if head_dim is not None else int(q.shape[2])
    p.page_size = page_size
    p.num_pages = num_pages if num_pages is not None else int(k_cache.shape[0])
    p.total_nodes = int(total_nodes)
    p.max_nodes = int(max_nodes)
    p.max_pages_per_seq = max_pages_per_seq if max_pages_per_seq is not None else int(block_table.shape[1])
    p.max_kv_pages = int(max_kv_pages)
    p.num_splits = int(num_splits)
    p.split_reduce = int(split_reduce)
    p.sm_scale = float(sm_scale)
    p.flags = int(flags)
    p.q, p.tree_k, p.tree_v = _ptr(q), _ptr(tree_k), _ptr(tree_v)
    p.k_cache, p.v_cache = _ptr(k_cache), _ptr(v_cache)
    p.block_table, p.ctx_lens, p.cu_nodes, p.parents = _ptr(block_table), _ptr(ctx_lens), _ptr(cu_nodes), _ptr(parents)
    p.kv_pages, p.cu_kv_pages = _ptr(kv_pages), _ptr(cu_kv_pages)
    p.out, p.lse = _ptr(out), _ptr(lse)
    p.workspace = _ptr(workspace)
    p.workspace_bytes = int(workspace_bytes if workspace_bytes else
                            (workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0))
    return p


def sv_tree_attention_workspace_size(params: sv_attn_params) -> int:
    n = c_size_t(0)
    _check(load().sv_tree_attention_workspace_size(ctypes.byref(params), ctypes.byref(n)),
           "sv_tree_attention_workspace_size")
    return int(n.value)


def sv_tree_attention_plan(params: sv_attn_params, with_kernel: bool = False):
    """(num_splits, split_reduce) the library would launch with, plus the
    kernel (0 = paired, 1 = wide, 2 = dealt) when with_kernel is set."""
    s, m, k = c_int(0), c_int(0), c_int(0)
    _check(load().sv_tree_attention_plan(ctypes.byref(params), ctypes.byref(s), ctypes.byref(m), ctypes.byref(k)),
           "sv_tree_attention_plan")
    if with_kernel:
        return int(s.value), int(m.value), int(k.value)
    return int(s.value), int(m.value)


def sv_tree_attention(params: sv_attn_params, stream=None) -> None:
    _check(load().sv_tree_attention(ctypes.byref(params), _stream(stream)), "sv_tree_attention")


def sv_greedy_accept_workspace_size(batch: int, total_nodes: int) -> int:
    n = c_size_t(0)
    _check(load().sv_greedy_accept_workspace_size(batch, total_nodes, ctypes.byref(n)),
           "sv_greedy_accept_workspace_size")
    return int(n.value)


def sv_greedy_accept(logits, vocab: int, tokens, parents, cu_nodes, batch: int, total_nodes: int,
                     max_nodes: int, max_depth: int, argmax_out, accept_len, accepted_nodes, bonus_token,
                     workspace, workspace_bytes: Optional[int] = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().sv_greedy_accept(_ptr(logits), vocab, _ptr(tokens), _ptr(parents), _ptr(cu_nodes), batch,
                                   total_nodes, max_nodes, max_depth, _ptr(argmax_out), _ptr(accept_len),
                                   _ptr(accepted_nodes), _ptr(bonus_token), _ptr(workspace), workspace_bytes,
                                   _stream(stream)), "sv_greedy_accept")


def sv_greedy_accept_noalloc(logits, vocab: int, tokens, parents, cu_nodes, batch: int, total_nodes: int,
                             max_nodes: int, max_depth: int, argmax_out, accept_len, accepted_nodes, bonus_token,
                             device_error=None, stream=None) -> None:
    """Greedy acceptance without a workspace, for callers that cannot
    allocate device memory; its scratch is a fixed array in the library (see
    include/sv.h for its limits and for why overlapping calls race)."""
    _check(load().sv_greedy_accept_noalloc(_ptr(logits), vocab, _ptr(tokens), _ptr(parents), _ptr(cu_nodes),
                                           batch, total_nodes, max_nodes, max_depth, _ptr(argmax_out),
                                           _ptr(accept_len), _ptr(accepted_nodes), _ptr(bonus_token),
                                           _ptr(device_error), _stream(stream)), "sv_greedy_accept_noalloc")


def sv_selftest_bounded_wait(workspace, abort_after_ns: int = 0, stream=None) -> None:
    """Launches a kernel whose bounded mbarrier wait must give up (see
    include/sv.h); read the outcome with sv_get_device_error."""
    _check(load().sv_selftest_bounded_wait(_ptr(workspace), int(abort_after_ns), _stream(stream)),
           "sv_selftest_bounded_wait")


def sv_sample_accept_workspace_size(batch: int, total_nodes: int) -> int:
    n = c_size_t(0)
    _check(load().sv_sample_accept_workspace_size(batch, total_nodes, ctypes.byref(n)),
           "sv_sample_accept_workspace_size")
    return int(n.value)


def sv_sample_accept(logits, draft_probs, vocab: int, temperature: float, tokens, parents, cu_nodes, batch: int,
                     total_nodes: int, max_nodes: int, max_depth: int, u_accept, u_bonus, accepted_child,
                     accept_len, accepted_nodes, bonus_token, workspace, workspace_bytes: Optional[int] = None,
                     stream=None) -> None:
    """Stochastic (temperature > 0) acceptance: speculative sampling node by
    node over the tree (see include/sv.h for the rule and the layouts)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().sv_sample_accept(_ptr(logits), _ptr(draft_probs), vocab, float(temperature), _ptr(tokens),
                                   _ptr(parents), _ptr(cu_nodes), batch, total_nodes, max_nodes, max_depth,
                                   _ptr(u_accept), _ptr(u_bonus), _ptr(accepted_child), _ptr(accept_len),
                                   _ptr(accepted_nodes), _ptr(bonus_token), _ptr(workspace), workspace_bytes,
                                   _stream(stream)), "sv_sample_accept")


def sv_kv_commit(tree_k, tree_v, tree_layer_stride: int, k_cache, v_cache, cache_layer_stride: int,
                 num_layers: int, num_pages: int, block_table, max_pages_per_seq: int, ctx_lens, cu_nodes,
                 accepted_nodes, accept_len, batch: int, max_depth: int, num_kv_heads: int, head_dim: int,
                 page_size: int = 16, new_ctx_lens=None, workspace=None, workspace_bytes: int = 0,
                 stream=None) -> None:
    if workspace is not None and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().sv_kv_commit(_ptr(tree_k), _ptr(tree_v), tree_layer_stride, _ptr(k_cache), _ptr(v_cache),
                               cache_layer_stride, num_layers, num_pages, _ptr(block_table), max_pages_per_seq,
                               _ptr(ctx_lens), _ptr(cu_nodes), _ptr(accepted_nodes), _ptr(accept_len), batch,
                               max_depth, num_kv_heads, head_dim, page_size, _ptr(new_ctx_lens),
                               _ptr(workspace), workspace_bytes, _stream(stream)), "sv_kv_commit")


def sv_kv_page_summaries(k_cache, num_pages: int, num_kv_heads: int, head_dim: int, block_table,
                         max_pages_per_seq: int, ctx_lens, first_page, batch: int, max_ctx_pages: int, summaries,
                         workspace=None, workspace_bytes: int = 0, page_size: int = 16, stream=None) -> None:
    if workspace is not None and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().sv_kv_page_summaries(_ptr(k_cache), num_pages, num_kv_heads, head_dim, page_size,
                                       _ptr(block_table), max_pages_per_seq, _ptr(ctx_lens), _ptr(first_page),
                                       batch, max_ctx_pages, _ptr(summaries), _ptr(workspace), workspace_bytes,
                                       _stream(stream)), "sv_kv_page_summaries")


def retrieve_list_bound(sink_tokens: int, window_tokens: int, topk: int, page_size: int = 16) -> int:
    """Longest partial list sv_retrieve_pages writes for one sequence."""
    return -(-sink_tokens // page_size) + topk + -(-window_tokens // page_size) + 1


def sv_retrieve_pages_workspace_size(batch: int, num_kv_heads: int, head_dim: int, max_ctx_pages: int) -> int:
    n = c_size_t(0)
    _check(load().sv_retrieve_pages_workspace_size(batch, num_kv_heads, head_dim, max_ctx_pages, ctypes.byref(n)),
           "sv_retrieve_pages_workspace_size")
    return int(n.value)


def make_retrieve_params(*, q, summaries, block_table, ctx_lens, cu_nodes, kv_pages, cu_kv_pages, batch: int,
                         num_q_heads: int, num_kv_heads: int, head_dim: int, num_pages: int, total_nodes: int,
                         max_pages_per_seq: int, max_ctx_pages: int, sink_tokens: int, window_tokens: int,
                         topk: int, reduce: int = SV_REDUCE_MEAN, scores=None, kv_pages_capacity=None,
                         workspace=None, workspace_bytes: int = 0, page_size: int = 16) -> sv_retrieve_params:
    r = sv_retrieve_params()
    r.batch, r.num_q_heads, r.num_kv_heads, r.head_dim = batch, num_q_heads, num_kv_heads, head_dim
    r.page_size, r.num_pages, r.total_nodes, r.max_pages_per_seq = page_size, num_pages, total_nodes, max_pages_per_seq
    r.max_ctx_pages, r.sink_tokens, r.window_tokens, r.topk, r.reduce = (max_ctx_pages, sink_tokens, window_tokens,
                                                                         topk, reduce)
    r.q, r.summaries, r.block_table, r.ctx_lens, r.cu_nodes = (_ptr(q), _ptr(summaries), _ptr(block_table),
                                                              _ptr(ctx_lens), _ptr(cu_nodes))
    r.kv_pages, r.cu_kv_pages, r.scores = _ptr(kv_pages), _ptr(cu_kv_pages), _ptr(scores)
    if kv_pages_capacity is None:
        kv_pages_capacity = kv_pages.numel() if hasattr(kv_pages, "numel") else 0
    r.kv_pages_capacity = int(kv_pages_capacity)
    r.workspace = _ptr(workspace)
    r.workspace_bytes = int(workspace_bytes if workspace_bytes else
                            (workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0))
    return r


def sv_retrieve_pages(params: sv_retrieve_params, stream=None) -> None:
    _check(load().sv_retrieve_pages(ctypes.byref(params), _stream(stream)), "sv_retrieve_pages")


def sv_partial_list_extend(ref_pages, ref_cu, ref_ctx_lens, ctx_lens, batch: int, kv_pages, cu_kv_pages,
                           workspace=None, workspace_bytes: int = 0, stream=None) -> None:
    if workspace is not None and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().sv_partial_list_extend(_ptr(ref_pages), _ptr(ref_cu), _ptr(ref_ctx_lens), _ptr(ctx_lens), batch,
                                         _ptr(kv_pages), _ptr(cu_kv_pages), _ptr(workspace), workspace_bytes,
                                         _stream(stream)), "sv_partial_list_extend")


def sv_specpv_full_trees(cand_parents, cand_tokens, cand_cu, buffer_tokens, buffer_cu, batch: int, parents,
                         tokens, cu_nodes, workspace=None, workspace_bytes: int = 0, stream=None) -> None:
    if workspace is not None and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().sv_specpv_full_trees(_ptr(cand_parents), _ptr(cand_tokens), _ptr(cand_cu), _ptr(buffer_tokens),
                                       _ptr(buffer_cu), batch, _ptr(parents), _ptr(tokens), _ptr(cu_nodes),
                                       _ptr(workspace), workspace_bytes, _stream(stream)), "sv_specpv_full_trees")


def sv_specpv_next(seq: sv_specpv_seq, step_tokens: int, buffer_limit: int) -> int:
    return int(load().sv_specpv_next(ctypes.byref(seq), step_tokens, buffer_limit))


def sv_specpv_after(seq: sv_specpv_seq, kind: int, ctx_len_after: int) -> None:
    _check(load().sv_specpv_after(ctypes.byref(seq), kind, ctx_len_after), "sv_specpv_after")


TRACE_SLOTS = 16
TRACE_EVENTS = ["start_ns", "prologue", "inputs", "first_ids", "first_mma", "first_s", "loop_end", "o_ready",
                "epilogue", "merge_ready", "merge_done", "exit", "tree_mask"]


def sv_set_trace_buffer(buffer, nbytes: int = 0) -> None:
    """Install (or with None remove) the per-CTA phase trace buffer."""
    if buffer is not None and not nbytes:
        nbytes = buffer.numel() * buffer.element_size()
    _check(load().sv_set_trace_buffer(_ptr(buffer), nbytes), "sv_set_trace_buffer")


def sv_get_device_error(workspace, stream=None) -> int:
    """Returns the workspace's device error code (0 = none) and clears it."""
    code = c_int(0)
    st = load().sv_get_device_error(_ptr(workspace), ctypes.byref(code), _stream(stream))
    if st not in (SV_OK, 5, 6):
        _check(st, "sv_get_device_error")
    return int(code.value)
