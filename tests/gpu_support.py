"""Shared helpers of the GPU tests: move a generated case to the device and
call the library through its C ABI (ctypes binding)."""

from __future__ import annotations

import numpy as np
import torch

from speculative_decoding_tree_sv_gb300 import binding, build

ATOL_ATTN = 2e-2   # bf16 inputs, fp32 accumulation, bf16 output
ATOL_LSE = 2e-3


def ensure_lib():
    build.build()
    return binding.load()


def bf16(arr_u16: np.ndarray, dev="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(arr_u16).view(np.int16)).view(torch.bfloat16)
    return t.to(dev)


def i32(arr, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(arr, dtype=np.int32))).to(dev)


class DeviceCase:
    """Device copies of one layer (or all layers) of a VerifyCase."""

    def __init__(self, case, layers=None):
        self.case = case
        layers = list(range(case.num_layers)) if layers is None else list(layers)
        self.layers = layers
        self.q = [bf16(case.q[l]) for l in layers]
        self.tree_k = bf16(case.tree_k[layers])
        self.tree_v = bf16(case.tree_v[layers])
        self.k_cache = bf16(case.k_cache[layers])
        self.v_cache = bf16(case.v_cache[layers])
        self.block_table = i32(case.block_table)
        self.ctx_lens = i32(case.ctx_lens)
        self.cu_nodes = i32(case.cu_nodes)
        self.parents = i32(case.parents)
        self.tokens = i32(case.tokens)
        self.kv_pages = i32(case.kv_pages) if case.kv_pages is not None else None
        self.cu_kv_pages = i32(case.cu_kv_pages) if case.cu_kv_pages is not None else None


def run_attention(dc: DeviceCase, li: int = 0, partial: bool = False, num_splits: int = 0,
                  with_lse: bool = True, sm_scale: float = 0.0, check_error: bool = True,
                  split_reduce: int = 0, flags: int = 0):
    c = dc.case
    T, Hq, D = c.total_nodes, c.num_q_heads, c.head_dim
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    kvp = dc.kv_pages if partial else None
    ckvp = dc.cu_kv_pages if partial else None
    max_kv = int(np.diff(c.cu_kv_pages).max()) if partial else 0
    p = binding.make_attn_params(
        q=dc.q[li], tree_k=dc.tree_k[li], tree_v=dc.tree_v[li], k_cache=dc.k_cache[li],
        v_cache=dc.v_cache[li], block_table=dc.block_table, ctx_lens=dc.ctx_lens, cu_nodes=dc.cu_nodes,
        parents=dc.parents, out=out, lse=lse, total_nodes=T, max_nodes=c.max_nodes,
        kv_pages=kvp, cu_kv_pages=ckvp, max_kv_pages=max_kv, num_splits=num_splits, sm_scale=sm_scale,
        split_reduce=split_reduce, flags=flags)
    ws_bytes = binding.sv_tree_attention_workspace_size(p)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    p.workspace = ws.data_ptr()
    p.workspace_bytes = ws_bytes
    binding.sv_tree_attention(p)
    torch.cuda.synchronize()
    err = binding.sv_get_device_error(ws)
    if check_error:
        assert err == 0, f"device error {binding.DEVICE_ERRORS.get(err, err)}"
    return out.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None), err


def run_accept(case, logits_dev=None, max_depth=None):
    dev = "cuda"
    T, V, B = case.total_nodes, case.vocab, case.batch
    max_depth = case.max_depth if max_depth is None else max_depth
    logits = logits_dev if logits_dev is not None else torch.from_numpy(case.logits).to(dev)
    tokens, parents, cu = i32(case.tokens), i32(case.parents), i32(case.cu_nodes)
    am = torch.full((T,), -7, dtype=torch.int32, device=dev)
    alen = torch.full((B,), -7, dtype=torch.int32, device=dev)
    anodes = torch.full((B, max_depth + 1), -7, dtype=torch.int32, device=dev)
    bonus = torch.full((B,), -7, dtype=torch.int32, device=dev)
    ws = torch.zeros(binding.sv_greedy_accept_workspace_size(B, T), dtype=torch.uint8, device=dev)
    binding.sv_greedy_accept(logits, V, tokens, parents, cu, B, T, case.max_nodes, max_depth, am, alen, anodes,
                             bonus, ws)
    torch.cuda.synchronize()
    err = binding.sv_get_device_error(ws)
    return dict(argmax=am.cpu().numpy(), accept_len=alen.cpu().numpy(), accepted_nodes=anodes.cpu().numpy(),
                bonus=bonus.cpu().numpy(), err=err, ws=ws)
