"""Benchmark of one tree-verification step on GB300 (one GPU).

A step is the whole hot path over one synthetic verify step of the
Llama-3.1-8B shaped workload (batch 1, 32 layers of 32 query / 8 KV heads of
128, 4096 context tokens in shuffled 16-token pages, a 60-node EAGLE-3 style
tree, 128256-entry fp32 logits with a planted accepted path of length 4):

  32 x sv_tree_attention (one per layer) + sv_greedy_accept + sv_kv_commit

The step is captured once in a CUDA graph and replayed.  The metric is tree
nodes verified per second per layer (nodes x layers / step time).  The
attention kernel is also timed alone (a graph of the 32 attention launches)
to give its achieved HBM bandwidth against the measured GB300 copy peak.

``per_config`` times one attention layer of each other workload (tiny, the
serving mix, the 60K context with full and with SpecPV partial KV, SpecBlock
trees), the layer's buffers repeated on the device until the bytes the
replayed calls read exceed twice the L2, next to the oracle on the host cores.

``--impl reference`` times the CPU oracle (NumPy float64, the machine's host
cores) over whole steps of the same workload.

The library is for one GPU: its paired attention kernel shares K/V tiles
between the two CTAs of a cluster with TMA multicast, which is kept to
single-GPU jobs, so the GPU arm refuses a multi-GPU launch before loading it.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tree-verify nodes/s per layer; attention HBM GB/s as % of GB300 peak (1 GPU)"
UNIT = "nodes/s/layer"
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0  # TFLOP/s, one earlier GB300 measurement
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
WORKLOADS = {
    "llama8b_eagle": "Llama-3.1-8B shaped verify step: batch 1, 32 layers x (32 q / 8 kv heads, head_dim 128), "
                     "context 4096 in shuffled 16-token pages, 60-node EAGLE-3 static tree (depth 7), "
                     "fp32 logits 60x128256 with a planted accepted path of length 4",
    "tiny": "Tiny single-layer verify: batch 1, 8 q / 2 kv heads, head_dim 64, context 512, 16-node tree of depth 4, "
            "fp32 logits 16x32000 with a planted path of 3",
    "serving_mix": "Batched serving mix: 32 sequences, context U[1000,1600], 60-node trees, Llama-3.1-8B attention",
    "long_partial": "60000-token context, 48-node tree, full KV",
    "long_partial_pv": "60000-token context, 48-node tree, SpecPV partial list (64 sink + 32x64 retrieved + last 1024)",
    "specblock": "SpecBlock trees (<=128 nodes, depth <=12), batch 16, 64 q / 8 kv heads, context 16384",
}
KERNEL_NAMES = ["paired 128-row CTAs", "256-row CTAs", "256-row CTAs, work dealt evenly over one CTA per SM"]
# one attention layer of each of these is timed next to the headline step
PER_CONFIG = ("tiny", "serving_mix", "long_partial", "long_partial_pv", "specblock")
# (sequence, KV head) units of the SpecBlock layer the oracle times; the
# layer's time is scaled from them (a fp64 layer is about a teraFLOP)
SPECBLOCK_ORACLE_UNITS = ((0, 0), (5, 3), (11, 6))


# ---------------------------------------------------------------------------- helpers

def refuse_multi_gpu(args) -> None:
    """The GPU arm runs on one GPU only: exit before the library is loaded."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != 1 or world != 1:
        sys.stderr.write("bench.py: the sv library runs on one GPU only (its paired attention kernel uses TMA "
                         f"multicast inside a two-CTA cluster); got --gpus {args.gpus}, WORLD_SIZE {world}\n")
        sys.exit(2)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Sustained dense bf16 TFLOP/s (the attention is timed in a seconds-long
    loop of launches), and whether it was measured here."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def measured_traffic(config: str):
    """DRAM bytes per attention launch from the committed ncu record, or None
    when the kernel source changed since those counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    csrc = os.path.join(ROOT, "speculative_decoding_tree_sv_gb300", "csrc")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(config)
    if not rec:
        return None
    h = hashlib.sha256()
    for name in ("tree_attention.cu", "tree_attention_wide.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return rec["dram_bytes_per_launch"] if h.hexdigest()[:16] == rec.get("kernel_source_sha256_16") else None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    def __init__(self, device_index: int, out_dir: str):
        self.proc = None
        self.path = os.path.join(out_dir, f"clocks_rank{device_index}.csv")
        self.dev = device_index

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
                 "clocks_event_reasons.gpu_idle",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        """Median SM clock over the samples taken while the GPU was busy (the
        idle reason not active), the maximum clock, and every throttle
        reason seen in them."""
        return summarize_clocks(open(self.path).read().splitlines()
                                if self.proc is not None and os.path.exists(self.path) else [])


def summarize_clocks(lines):
    sm, smax, reasons, total = [], [], set(), 0
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            mhz, mx = float(parts[0]), float(parts[1])
        except ValueError:
            continue
        total += 1
        if parts[8].lower() == "active":  # idle between timed regions
            continue
        sm.append(mhz)
        smax.append(mx)
        for name, v in zip(names, parts[4:8]):
            if v.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                "samples_total": total}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm), "samples_total": total}


# ---------------------------------------------------------------------------- workload

def _workload_seed(name: str) -> int:
    from synth import CONFIGS
    base = {"long_partial_pv": "long_partial"}.get(name, name)
    return int(CONFIGS[base]["seed"])


def build_case(name: str, with_logits: bool = True):
    """The synthetic case of workload ``name`` and whether its attention
    takes the SpecPV partial list."""
    from synth import make_case
    if name in ("long_partial", "long_partial_pv"):
        return make_case("long_partial", with_partial=True, with_logits=with_logits), name == "long_partial_pv"
    if name in WORKLOADS:
        return make_case(name, with_logits=with_logits), False
    raise ValueError(name)


def workload_config(name: str, case) -> dict:
    """The ``config`` object both arms print: the workload, nothing about how
    it is computed."""
    kv_bytes = sum(int(x) for x in case.ctx_lens) * 4 * case.num_kv_heads * case.head_dim * case.num_layers
    return {"workload": WORKLOADS[name], "layers": case.num_layers, "batch": case.batch,
            "total_nodes": case.total_nodes, "seed": _workload_seed(name),
            "l2": "inputs larger than L2 (distinct KV per layer, %.0f MB per step)" % (kv_bytes / 1e6),
            "parallelism": "single GPU"}


class GpuStep:
    """Device-resident inputs and the library calls of one verify step."""

    def __init__(self, case, partial: bool, dev: str, flags: int = 0):
        import torch

        from speculative_decoding_tree_sv_gb300 import binding
        self.torch, self.binding, self.case, self.partial = torch, binding, case, partial
        c = case
        self.dev = dev

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

        self.T, self.Hq, self.Hkv, self.D = c.total_nodes, c.num_q_heads, c.num_kv_heads, c.head_dim
        self.layers = c.num_layers
        # each layer's Q, tree K and tree V sit side by side in one arena row,
        # so one host-to-device copy moves a layer's (or a run of layers')
        # per-step inputs
        nq, nk = int(np.prod(c.q.shape[1:])), int(np.prod(c.tree_k.shape[1:]))
        self.layer_arena = torch.empty((c.num_layers, nq + 2 * nk), dtype=torch.bfloat16, device=dev)
        self.q = self.layer_arena[:, :nq].view(c.q.shape)
        self.tree_k = self.layer_arena[:, nq:nq + nk].view(c.tree_k.shape)
        self.tree_v = self.layer_arena[:, nq + nk:].view(c.tree_v.shape)
        self.q.copy_(bf(c.q))
        self.tree_k.copy_(bf(c.tree_k))
        self.tree_v.copy_(bf(c.tree_v))
        self.k_cache = bf(c.k_cache)
        self.v_cache = bf(c.v_cache)
        self.block_table = i32(c.block_table)
        self.ctx_lens = i32(c.ctx_lens)
        self.cu_nodes = i32(c.cu_nodes)
        self.parents = i32(c.parents)
        self.tokens = i32(c.tokens)
        self.logits = torch.from_numpy(c.logits).to(dev)
        self.kv_pages = i32(c.kv_pages) if partial else None
        self.cu_kv_pages = i32(c.cu_kv_pages) if partial else None
        self.max_kv_pages = int(np.diff(c.cu_kv_pages).max()) if partial else 0
        self.out = torch.empty((self.layers, self.T, self.Hq, self.D), dtype=torch.bfloat16, device=dev)
        self.params = []
        ws_bytes = 0
        for l in range(self.layers):
            p = binding.make_attn_params(
                q=self.q[l], tree_k=self.tree_k[l], tree_v=self.tree_v[l], k_cache=self.k_cache[l],
                v_cache=self.v_cache[l], block_table=self.block_table, ctx_lens=self.ctx_lens,
                cu_nodes=self.cu_nodes, parents=self.parents, out=self.out[l], total_nodes=self.T,
                max_nodes=c.max_nodes, kv_pages=self.kv_pages, cu_kv_pages=self.cu_kv_pages,
                max_kv_pages=self.max_kv_pages, flags=flags)
            ws_bytes = max(ws_bytes, binding.sv_tree_attention_workspace_size(p))
            self.params.append(p)
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        for p in self.params:
            p.workspace, p.workspace_bytes = self.ws.data_ptr(), ws_bytes
        self.splits, self.split_reduce, self.kernel = binding.sv_tree_attention_plan(self.params[0], with_kernel=True)
        B = c.batch
        self.am = torch.empty(self.T, dtype=torch.int32, device=dev)
        self.alen = torch.empty(B, dtype=torch.int32, device=dev)
        self.anodes = torch.empty((B, c.max_depth + 1), dtype=torch.int32, device=dev)
        self.bonus = torch.empty(B, dtype=torch.int32, device=dev)
        self.ws_acc = torch.zeros(binding.sv_greedy_accept_workspace_size(B, self.T), dtype=torch.uint8,
                                  device=dev)
        self.new_lens = torch.empty(B, dtype=torch.int32, device=dev)

    def launches_per_step(self):
        per_attn = 2 if (self.split_reduce == 2 or self.kernel == 2) else 1  # + the split or dealt combine
        return self.layers * per_attn + 2

    def attention_all_layers(self):
        for p in self.params:
            self.binding.sv_tree_attention(p)

    def accept_and_commit(self):
        c, b = self.case, self.binding
        b.sv_greedy_accept(self.logits, c.vocab, self.tokens, self.parents, self.cu_nodes, c.batch, self.T,
                           c.max_nodes, c.max_depth, self.am, self.alen, self.anodes, self.bonus, self.ws_acc)
        b.sv_kv_commit(self.tree_k, self.tree_v, self.tree_k.stride(0), self.k_cache, self.v_cache,
                       c.num_pages * self.Hkv * c.page_size * self.D, self.layers, c.num_pages,
                       self.block_table, c.max_pages_per_seq, self.ctx_lens, self.cu_nodes, self.anodes,
                       self.alen, c.batch, c.max_depth, self.Hkv, self.D, c.page_size, self.new_lens, self.ws)

    def step(self):
        self.attention_all_layers()
        self.accept_and_commit()


def _time_graph(torch, fn, steps: int, warmup: int):
    """Capture fn in a CUDA graph, warm up, time `steps` replays (events on the
    capturing stream's side of the current stream, synchronize on both
    sides)."""
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        fn()  # eager warm-up outside the graph
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(steps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), g


# ---------------------------------------------------------------------------- CPU oracle leg

CPU_BASELINE_SECONDS = 10.0
REFERENCE_BUDGET_SECONDS = 200.0


def copy_runs(layers: int, growth: int = 4):
    """Half-open layer ranges [a, b) of 1, growth, growth^2, ... layers that
    cover 0 .. layers - 1 in order: the host-to-device copies of the
    end-to-end step, one per range."""
    runs, a, n = [], 0, 1
    while a < layers:
        runs.append((a, min(layers, a + n)))
        a, n = runs[-1][1], growth * n
    return runs


def oracle_attention_layer(case, partial: bool, layer: int = 0, seqs=None, kv_heads=None):
    import oracle
    return oracle.tree_verify_attention(
        case.q[layer], case.tree_k[layer], case.tree_v[layer], case.k_cache[layer], case.v_cache[layer],
        case.block_table, case.ctx_lens, case.cu_nodes, case.parents, page_size=case.page_size,
        kv_pages=case.kv_pages if partial else None, cu_kv_pages=case.cu_kv_pages if partial else None,
        seqs=seqs, kv_heads=kv_heads)


def oracle_step_seconds(case, partial: bool, attn_layers: int = 1):
    """Times the oracle on `attn_layers` layers of attention plus one
    acceptance and one full commit; returns (seconds per full step, detail)."""
    import oracle
    t0 = time.perf_counter()
    for l in range(attn_layers):
        oracle_attention_layer(case, partial, l)
    t_attn = (time.perf_counter() - t0) / attn_layers
    t1 = time.perf_counter()
    acc = oracle.greedy_accept(case.logits, case.tokens, case.parents, case.cu_nodes)
    t_acc = time.perf_counter() - t1
    t2 = time.perf_counter()
    oracle.kv_commit(case.k_cache, case.v_cache, case.tree_k, case.tree_v, case.block_table, case.ctx_lens,
                     case.cu_nodes, acc["accepted_nodes"], acc["accept_len"], case.page_size)
    t_commit = time.perf_counter() - t2
    step = t_attn * case.num_layers + t_acc + t_commit
    return step, dict(attn_layer_s=t_attn, accept_s=t_acc, commit_s=t_commit)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def reference_plan(steps: int, warmup: int, step_s: float, budget_s: float = REFERENCE_BUDGET_SECONDS):
    """How many whole oracle steps the reference arm times: all `steps` when
    they fit the budget, else as many as fit (at least one)."""
    fit = int(budget_s // max(step_s, 1e-9))
    return max(1, min(steps, fit))


def run_reference(args):
    """The oracle timed over whole steps of the workload (every layer's
    attention, the acceptance over all logits, the commit of every layer).
    Warm-up steps are one attention layer each; when K whole steps would not
    end within the time budget, the arm times as many as fit and says so."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    case, partial = build_case(args.config)
    for _ in range(args.warmup):
        oracle_attention_layer(case, partial, 0)
    first, _ = oracle_step_seconds(case, partial, attn_layers=case.num_layers)
    n = reference_plan(args.steps, args.warmup, first, args.reference_budget_s)
    times = []
    t_start = time.perf_counter()
    for _ in range(n):
        s, _detail = oracle_step_seconds(case, partial, attn_layers=case.num_layers)
        times.append(s)
    wall = time.perf_counter() - t_start
    nodes = case.total_nodes * case.num_layers
    step_s = wall / n
    value = nodes / step_s
    sample = (f"{n} whole oracle steps timed ({case.num_layers} layers of attention, acceptance over all "
              f"{case.total_nodes}x{case.vocab} logits, the commit of all layers), {wall:.1f} s; warm-up: "
              f"{args.warmup} single attention layers and one untimed whole step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": n, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.config, case),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if n < args.steps:
        line["steps_requested"] = args.steps
        line["note"] = (f"{args.steps} whole oracle steps would take about {args.steps * first:.0f} s; "
                        f"{n} were timed, within the {args.reference_budget_s:.0f} s budget")
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU leg

def retrieval_timing(torch, st, args):
    """SpecPV retrieval on the partial-KV workload (layer 0): the page
    summaries of the whole context (built once per full verification) and one
    retrieval (mean reduction, the workload's 64 sink tokens, 128 retrieved
    pages = 32 blocks of 64 tokens, 1024-token window), each timed alone in a
    CUDA graph."""
    from speculative_decoding_tree_sv_gb300 import binding
    c = st.case
    mcp = int(max(1, (int(np.max(c.ctx_lens)) + 15) // 16))
    summ = torch.zeros((c.num_pages, c.num_kv_heads, 2, c.head_dim), dtype=torch.bfloat16, device=st.dev)
    sink, window, topk = 64, 1024, 128
    cap = c.batch * binding.retrieve_list_bound(sink, window, topk)
    kv = torch.empty(cap, dtype=torch.int32, device=st.dev)
    cu = torch.empty(c.batch + 1, dtype=torch.int32, device=st.dev)
    ws = torch.zeros(binding.sv_retrieve_pages_workspace_size(c.batch, c.num_kv_heads, c.head_dim, mcp),
                     dtype=torch.uint8, device=st.dev)

    def summaries():
        binding.sv_kv_page_summaries(st.k_cache[0], c.num_pages, c.num_kv_heads, c.head_dim, st.block_table,
                                     c.max_pages_per_seq, st.ctx_lens, None, c.batch, mcp, summ, ws)

    params = binding.make_retrieve_params(
        q=st.q[0], summaries=summ, block_table=st.block_table, ctx_lens=st.ctx_lens, cu_nodes=st.cu_nodes,
        kv_pages=kv, cu_kv_pages=cu, batch=c.batch, num_q_heads=c.num_q_heads, num_kv_heads=c.num_kv_heads,
        head_dim=c.head_dim, num_pages=c.num_pages, total_nodes=c.total_nodes,
        max_pages_per_seq=c.max_pages_per_seq, max_ctx_pages=mcp, sink_tokens=sink, window_tokens=window,
        topk=topk, workspace=ws)

    def retrieve():
        binding.sv_retrieve_pages(params)

    ms_s, _ = _time_graph(torch, summaries, args.steps, args.warmup)
    ms_r, _ = _time_graph(torch, retrieve, args.steps, args.warmup)
    tokens = int(np.sum(c.ctx_lens))
    pages = int(np.sum((c.ctx_lens + 15) // 16))
    row = c.num_kv_heads * c.head_dim * 2                     # one token's K (bf16)
    sum_bytes = tokens * row + pages * 2 * row                 # keys read, max/min written
    cand = pages - c.batch * (sink // 16 + window // 16)
    ret_bytes = cand * 2 * row + c.total_nodes * c.num_q_heads * c.head_dim * 2 + pages * 8
    us_s, us_r = ms_s * 1e3 / args.steps, ms_r * 1e3 / args.steps
    return {"summaries_us": us_s, "summaries_gbs": sum_bytes / (us_s * 1e-6) / 1e9,
            "retrieve_us": us_r, "retrieve_gbs": ret_bytes / (us_r * 1e-6) / 1e9,
            "reduce": "mean", "sink_tokens": sink, "window_tokens": window, "topk_pages": topk}


def accept_commit_timing(torch, st, args, peak):
    """sv_greedy_accept, sv_kv_commit and sv_sample_accept (temperature 1)
    each timed alone in a CUDA graph.  The acceptances rotate copies of the
    logits (and of the drafts) so that together they exceed L2: each call
    reads its inputs from HBM, as in the step."""
    c, b = st.case, st.binding
    logits_bytes = st.logits.numel() * 4
    copies = int(min(8, max(1, -(-200_000_000 // logits_bytes))))
    bufs = [st.logits] + [st.logits.clone() for _ in range(copies - 1)]

    def accept_only():
        for lg in bufs:
            b.sv_greedy_accept(lg, c.vocab, st.tokens, st.parents, st.cu_nodes, c.batch, st.T, c.max_nodes,
                               c.max_depth, st.am, st.alen, st.anodes, st.bonus, st.ws_acc)

    def commit_only():
        b.sv_kv_commit(st.tree_k, st.tree_v, st.tree_k.stride(0), st.k_cache, st.v_cache,
                       c.num_pages * st.Hkv * c.page_size * st.D, st.layers, c.num_pages, st.block_table,
                       c.max_pages_per_seq, st.ctx_lens, st.cu_nodes, st.anodes, st.alen, c.batch, c.max_depth,
                       st.Hkv, st.D, c.page_size, st.new_lens, st.ws)

    # stochastic acceptance at temperature 1 (drafts near the target), on
    # the same logits copies and one draft array per copy
    from synth import make_sampling_inputs
    q_np, tok_np, ua_np, ub_np = make_sampling_inputs(c, seed=1)
    qs = [torch.from_numpy(q_np).to(st.dev)] + [None] * (copies - 1)
    for i in range(1, copies):
        qs[i] = qs[0].clone()
    s_tok = torch.from_numpy(tok_np).to(st.dev)
    s_ua, s_ub = torch.from_numpy(ua_np).to(st.dev), torch.from_numpy(ub_np).to(st.dev)
    s_ws = torch.zeros(b.sv_sample_accept_workspace_size(c.batch, st.T), dtype=torch.uint8, device=st.dev)

    def sample_only():
        for lg, qq in zip(bufs, qs):
            b.sv_sample_accept(lg, qq, c.vocab, 1.0, s_tok, st.parents, st.cu_nodes, c.batch, st.T, c.max_nodes,
                               c.max_depth, s_ua, s_ub, None, st.alen, st.anodes, st.bonus, s_ws)

    ms_a, _ = _time_graph(torch, accept_only, args.steps, args.warmup)
    ms_c, _ = _time_graph(torch, commit_only, args.steps, args.warmup)
    ms_s, _ = _time_graph(torch, sample_only, args.steps, args.warmup)
    us_a = ms_a * 1e3 / (args.steps * copies)
    us_c = ms_c * 1e3 / args.steps
    us_s = ms_s * 1e3 / (args.steps * copies)
    slots = int(np.sum(np.asarray(c.planted_len) + 1))                      # root + accepted nodes
    commit_bytes = 2 * slots * 2 * st.Hkv * st.D * 2 * st.layers            # K and V, read + written
    gbs_a = logits_bytes / (us_a * 1e-6) / 1e9
    return {"accept_us": us_a, "accept_gbs": gbs_a, "accept_frac": gbs_a / peak,
            "accept_bytes": logits_bytes, "accept_logits_copies": copies,
            "commit_us": us_c, "commit_gbs": commit_bytes / (us_c * 1e-6) / 1e9, "commit_bytes": commit_bytes,
            "sample_accept_us": us_s, "sample_accept_gbs": 2 * logits_bytes / (us_s * 1e-6) / 1e9,
            "sample_accept_bytes": 2 * logits_bytes, "sample_temperature": 1.0}


def attention_roofline(case, partial, us_per_call, peak, peak_kind, tpeak, tpeak_kind, traffic):
    """Roofline object of one attention call (attention + split combine):
    algorithmic bytes (or FLOPs past the ridge) per call / the call time."""
    from synth import node_depths

    from speculative_decoding_tree_sv_gb300 import cost
    c = case
    if partial:
        ctx_keys = [cost.context_keys(int(c.ctx_lens[b]), c.page_size,
                                      c.kv_pages[c.cu_kv_pages[b]:c.cu_kv_pages[b + 1]]) for b in range(c.batch)]
    else:
        ctx_keys = [int(x) for x in c.ctx_lens]
    ns = np.diff(c.cu_nodes)
    bytes_launch = cost.attention_bytes(ctx_keys, ns, c.num_q_heads, c.num_kv_heads, c.head_dim)
    depths = [node_depths(c.parents[c.cu_nodes[b]:c.cu_nodes[b + 1]]) for b in range(c.batch)]
    flops_launch = cost.attention_flops(ctx_keys, depths, c.num_q_heads, c.head_dim)
    t = us_per_call * 1e-6
    achieved = bytes_launch / t / 1e9
    # past the ridge (large trees at large GQA) the tensor pipe is the bound
    if flops_launch / bytes_launch > tpeak * 1e12 / (peak * 1e9):
        tf = flops_launch / t / 1e12
        return {"bound": "tensor", "achieved": tf, "peak": tpeak, "unit": "TFLOP/s", "frac": tf / tpeak,
                "traffic": traffic, "peak_kind": tpeak_kind + " (sustained bf16)",
                "flops_per_launch": flops_launch, "bytes_per_launch": bytes_launch, "hbm_gbs": achieved,
                "hbm_frac": achieved / peak, "launch_us": us_per_call}
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "peak_kind": peak_kind, "bytes_per_launch": bytes_launch,
            "flops_per_launch": flops_launch, "launch_us": us_per_call}


class AttentionLeg:
    """One attention layer of a workload, its device buffers repeated
    `replicas` times (distinct addresses) so the calls of one replay read
    more than twice the L2 from HBM."""

    def __init__(self, torch, case, partial, dev, bytes_per_call, flags: int = 0, num_splits: int = 0):
        from speculative_decoding_tree_sv_gb300 import binding
        self.torch, self.binding, self.case, self.partial = torch, binding, case, partial
        c = case

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

        per_replica = (c.k_cache[0].nbytes + c.v_cache[0].nbytes + c.q[0].nbytes + c.tree_k[0].nbytes +
                       c.tree_v[0].nbytes + c.q[0].nbytes)
        want = -(-2 * L2_BYTES // max(1, bytes_per_call))
        self.replicas = int(max(1, min(want, 24_000_000_000 // per_replica, 2048)))
        R = self.replicas
        k1, v1 = bf(c.k_cache[0]), bf(c.v_cache[0])
        q1, tk1, tv1 = bf(c.q[0]), bf(c.tree_k[0]), bf(c.tree_v[0])
        self.k_cache = k1.unsqueeze(0).repeat(R, *([1] * k1.dim()))
        self.v_cache = v1.unsqueeze(0).repeat(R, *([1] * v1.dim()))
        self.q = q1.unsqueeze(0).repeat(R, 1, 1, 1)
        self.tree_k = tk1.unsqueeze(0).repeat(R, 1, 1, 1)
        self.tree_v = tv1.unsqueeze(0).repeat(R, 1, 1, 1)
        self.out = torch.empty((R,) + tuple(q1.shape), dtype=torch.bfloat16, device=dev)
        del k1, v1
        self.block_table, self.ctx_lens = i32(c.block_table), i32(c.ctx_lens)
        self.cu_nodes, self.parents = i32(c.cu_nodes), i32(c.parents)
        self.kv_pages = i32(c.kv_pages) if partial else None
        self.cu_kv_pages = i32(c.cu_kv_pages) if partial else None
        max_kv = int(np.diff(c.cu_kv_pages).max()) if partial else 0
        self.params = []
        ws_bytes = 0
        for r in range(R):
            p = binding.make_attn_params(
                q=self.q[r], tree_k=self.tree_k[r], tree_v=self.tree_v[r], k_cache=self.k_cache[r],
                v_cache=self.v_cache[r], block_table=self.block_table, ctx_lens=self.ctx_lens,
                cu_nodes=self.cu_nodes, parents=self.parents, out=self.out[r], total_nodes=c.total_nodes,
                max_nodes=c.max_nodes, kv_pages=self.kv_pages, cu_kv_pages=self.cu_kv_pages,
                max_kv_pages=max_kv, flags=flags, num_splits=num_splits)
            ws_bytes = max(ws_bytes, binding.sv_tree_attention_workspace_size(p))
            self.params.append(p)
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        for p in self.params:
            p.workspace, p.workspace_bytes = self.ws.data_ptr(), ws_bytes
        self.splits, self.split_reduce, self.kernel = binding.sv_tree_attention_plan(self.params[0], with_kernel=True)

    def calls(self):
        for p in self.params:
            self.binding.sv_tree_attention(p)

    def launches(self):
        return self.replicas * (2 if (self.split_reduce == 2 or self.kernel == 2) else 1)


def per_config_leg(torch, name, args, dev, peaks):
    """One attention layer of workload `name`: time per call on the GPU and
    the oracle's time for the same layer on the host cores."""
    peak, peak_kind, tpeak, tpeak_kind = peaks
    case, partial = build_case(name, with_logits=False)
    probe = attention_roofline(case, partial, 1.0, peak, peak_kind, tpeak, tpeak_kind, None)
    leg = AttentionLeg(torch, case, partial, dev, probe["bytes_per_launch"])
    ms, _g = _time_graph(torch, leg.calls, args.steps, args.warmup)
    us = ms * 1e3 / (args.steps * leg.replicas)
    err = leg.binding.sv_get_device_error(leg.ws)
    if err != 0:
        raise RuntimeError(f"{name}: device error {err}")
    roof = attention_roofline(case, partial, us, peak, peak_kind, tpeak, tpeak_kind, measured_traffic(name))
    nodes = case.total_nodes
    out = {"workload": WORKLOADS[name], "us_per_call": us, "nodes_per_s_per_layer": nodes / (us * 1e-6),
           "roofline": roof, "kernel": KERNEL_NAMES[leg.kernel],
           "kv_splits": leg.splits, "layer_copies": leg.replicas,
           "gpu_launches": leg.launches() * args.steps}
    if not args.no_cpu_baseline:
        if name == "specblock":
            units = SPECBLOCK_ORACLE_UNITS
            t0 = time.perf_counter()
            for b, h in units:
                oracle_attention_layer(case, partial, 0, seqs=[b], kv_heads=[h])
            per_unit = (time.perf_counter() - t0) / len(units)
            # units differ in their tree's size: scale by each sequence's
            # nodes relative to the sampled ones
            ns = np.diff(case.cu_nodes)
            sampled_nodes = np.mean([ns[b] for b, _ in units])
            layer_s = per_unit * float(ns.sum()) / sampled_nodes * case.num_kv_heads
            sample = (f"{len(units)} (sequence, KV head) units of the layer timed, scaled by tree nodes to all "
                      f"{case.batch} x {case.num_kv_heads} units (extrapolated)")
        else:
            t0 = time.perf_counter()
            oracle_attention_layer(case, partial, 0)
            layer_s = time.perf_counter() - t0
            sample = "one whole attention layer"
        out["oracle"] = {"seconds_per_layer": layer_s, "nodes_per_s_per_layer": nodes / layer_s,
                         "cores": host_cores(), "sample": sample}
    if partial:
        out["retrieval"] = retrieval_timing(torch, leg_as_step(leg), args)
    del leg
    torch.cuda.empty_cache()
    return out


def leg_as_step(leg):
    """The fields retrieval_timing reads, from an attention leg."""
    class _S:
        pass
    s = _S()
    s.case, s.dev = leg.case, leg.q.device
    s.k_cache, s.q = leg.k_cache, leg.q
    s.block_table, s.ctx_lens, s.cu_nodes = leg.block_table, leg.ctx_lens, leg.cu_nodes
    return s


def run_gpu(args):
    refuse_multi_gpu(args)
    import torch

    from speculative_decoding_tree_sv_gb300 import build as _build

    torch.cuda.set_device(0)
    dev = "cuda:0"
    _build.build()
    case, partial = build_case(args.config)
    flags = 0
    if args.early_context:
        from speculative_decoding_tree_sv_gb300 import binding
        flags = binding.SV_ATTN_EARLY_CONTEXT
    st = GpuStep(case, partial, dev, flags=flags)
    c = case
    nodes_per_step = c.total_nodes * c.num_layers
    peak, peak_kind = measured_peaks()
    tpeak, tpeak_kind = measured_tensor_peak()

    # Clocks are sampled over every timed region of the run.
    clk = ClockSampler(0, args.clocks_dir).__enter__()
    try:
        # whole step, graph-replayed
        ms, _g = _time_graph(torch, st.step, args.steps, args.warmup)
        # attention alone (the dominant kernel) for the roofline
        ms_attn, _ga = _time_graph(torch, st.attention_all_layers, args.steps, args.warmup)
        # the same attention calls without the graph (eager launches, events
        # on the current stream), for comparison
        for _ in range(args.warmup):
            st.attention_all_layers()
        torch.cuda.synchronize()
        eager_steps = max(1, min(args.steps, 200))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(eager_steps):
            st.attention_all_layers()
        e1.record()
        torch.cuda.synchronize()
        attn_eager_us = e0.elapsed_time(e1) * 1e3 / (eager_steps * c.num_layers)
        ms_step = ms / args.steps
        value = nodes_per_step / (ms_step * 1e-3)
        attn_us = ms_attn * 1e3 / (args.steps * c.num_layers)
        roofline = attention_roofline(c, partial, attn_us, peak, peak_kind, tpeak, tpeak_kind,
                                      measured_traffic(args.config))
        roofline["kernel"] = "sv_tree_attention (attention + split combine)"
        roofline["launch_us_without_graph"] = attn_eager_us

        # end to end through the public API with host buffers: pinned H2D of
        # the step's inputs, the step, D2H of the results; captured like the
        # step.
        pin = {}
        h2d = 0
        for name in ("layer_arena", "logits", "parents", "tokens", "cu_nodes", "ctx_lens"):
            t = getattr(st, name)
            pin[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
            h2d += t.numel() * t.element_size()
        res_host = {n: torch.empty(getattr(st, n).shape, dtype=torch.int32, pin_memory=True)
                    for n in ("alen", "anodes", "bonus")}
        d2h = sum(v.numel() * 4 for v in res_host.values())

        # The copies run on a second stream in the order the step consumes
        # them: the index arrays, then the layers' Q / tree K / tree V in runs
        # of 1, 4, 16, ... layers (a layer's inputs copy about four times
        # faster than its attention runs, so each run lands while the runs
        # before it are being computed), then the logits and tokens.  The
        # first call of each run waits for that run; a cross-stream wait costs
        # a few microseconds in the replayed graph, so there is one per run,
        # not one per layer.
        copy_stream = torch.cuda.Stream()
        first = ("parents", "cu_nodes", "ctx_lens")
        last = ("logits", "tokens")
        assert set(first + last + ("layer_arena",)) == set(pin)
        runs = copy_runs(st.layers)

        def e2e_step():
            cur = torch.cuda.current_stream()
            copy_stream.wait_stream(cur)
            run_ready = {}
            with torch.cuda.stream(copy_stream):
                for name in first:
                    getattr(st, name).copy_(pin[name], non_blocking=True)
                for a, b in runs:
                    st.layer_arena[a:b].copy_(pin["layer_arena"][a:b], non_blocking=True)
                    run_ready[a] = torch.cuda.Event()
                    run_ready[a].record(copy_stream)
                for name in last:
                    getattr(st, name).copy_(pin[name], non_blocking=True)
            for li, p in enumerate(st.params):
                if li in run_ready:
                    cur.wait_event(run_ready[li])
                st.binding.sv_tree_attention(p)
            cur.wait_stream(copy_stream)
            st.accept_and_commit()
            for name, h in res_host.items():
                h.copy_(getattr(st, name), non_blocking=True)

        ms_e2e, _ge = _time_graph(torch, e2e_step, args.steps, args.warmup)
        # the synthetic logits plant each sequence's accepted path: the
        # lengths read back through the timed path must be those
        if not np.array_equal(res_host["alen"].numpy(), np.asarray(c.planted_len)):
            raise RuntimeError("accepted lengths read back differ from the planted paths")
        e2e_value = nodes_per_step / (ms_e2e * 1e-3 / args.steps)

        retrieval = retrieval_timing(torch, st, args) if partial else None
        acc_commit = accept_commit_timing(torch, st, args, peak)
        err = st.binding.sv_get_device_error(st.ws)
        if err != 0:
            raise RuntimeError(f"device error {err} in the step")

        per_config = {}
        if not args.no_per_config:
            peaks = (peak, peak_kind, tpeak, tpeak_kind)
            for name in PER_CONFIG:
                if name != args.config:
                    per_config[name] = per_config_leg(torch, name, args, dev, peaks)
    finally:
        clk.__exit__(None, None, None)
    clocks = clk.summary()

    cpu = None
    if not args.no_cpu_baseline:
        # whole steps (every layer's attention, the acceptance, the commit),
        # repeated until about ten seconds of host work have been timed
        t_start, n_steps, details = time.perf_counter(), 0, []
        while n_steps == 0 or time.perf_counter() - t_start < CPU_BASELINE_SECONDS:
            details.append(oracle_step_seconds(case, partial, attn_layers=c.num_layers)[1])
            n_steps += 1
        s = (time.perf_counter() - t_start) / n_steps
        mean = {k: statistics.mean(d[k] for d in details) for k in details[0]}
        cpu = {"value": nodes_per_step / s, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"oracle (NumPy fp64): {n_steps} whole steps of the workload ({c.num_layers} layers of "
                         f"attention, acceptance over all {c.total_nodes}x{c.vocab} logits, the commit of all "
                         f"layers) in {s * n_steps:.1f} s; per step "
                         + ", ".join(f"{k} {v:.3f}" for k, v in mean.items())}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args.config, c),
        "plan": {"kv_splits": st.splits, "split_merge": "combine kernel" if (st.split_reduce == 2 or st.kernel == 2) else "none",
                 "attention_kernel": KERNEL_NAMES[st.kernel], "cuda_graph": True,
                 "early_context": bool(flags)},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": st.launches_per_step() * args.steps,
        "clocks": clocks,
        "accept_commit": acc_commit,
        **({"retrieval": retrieval} if retrieval else {}),
        **({"per_config": per_config} if per_config else {}),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["sv", "reference"], default="sv")
    ap.add_argument("--config", choices=sorted(WORKLOADS), default="llama8b_eagle")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline step (not one layer of each other workload)")
    ap.add_argument("--reference-budget-s", type=float, default=REFERENCE_BUDGET_SECONDS,
                    help="time budget of the reference arm's timed whole steps")
    ap.add_argument("--clocks-dir", default=os.path.join(ROOT, "bench_out"),
                    help="where the nvidia-smi clock samples of the timed regions are written")
    ap.add_argument("--early-context", action="store_true",
                    help="launch attention with SV_ATTN_EARLY_CONTEXT")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
