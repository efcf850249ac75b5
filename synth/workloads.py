"""Seeded generators for the five verification workloads.

Shapes follow the workloads described on the speculative-decoding pages:
EAGLE-3 style static trees ("Dynamic Speculative Decoding", benchmark table:
config = [num_steps, topk, num_draft_tokens]), SpecBlock block-iterative trees
with rank-bucket branching (SpecBlock, section 3 "Bucket-driven branching" and
Appendix B), the serving mix of ~1000-token prompts with ~600 generated tokens
("Dynamic Speculative Decoding", Problem Context) and SpecPV's long-context
partial-KV lists (SpecPV section 3.2 and Appendix D).

Value recipe: Q/K/V ~ N(0, 1) rounded to bf16 (round to nearest even), logits
~ N(0, 1) fp32, tokens uniform in [0, V) with distinct tokens among siblings.
Every row of the logits gets a planted, unique maximum so that the greedy
acceptance result is fixed by construction: along a chosen root path of
length ``a`` the planted maximum is the next path node's token, everywhere
else it is a token that none of the row's children carries.

bf16 tensors are returned as ``uint16`` bit patterns; numpy has no bf16 type.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

PAGE_SIZE = 16

# Workload definitions.  ``layers`` is the number of distinct attention layers
# a verify step covers; parity tests use one layer of the multi-layer cases.
CONFIGS = {
    # Tiny single-layer verify, oracle runs in well under a second.
    "tiny": dict(
        batch=1, num_q_heads=8, num_kv_heads=2, head_dim=64, layers=1,
        ctx=512, tree=("random_depth", 16, 4), vocab=32000, plant=3, seed=1001,
    ),
    # Llama-3.1-8B shaped verify step with an EAGLE-3 static tree
    # (steps 7, top-k 10, 60 draft tokens incl. the root).
    "llama8b_eagle": dict(
        batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, layers=32,
        ctx=4096, tree=("eagle", 60, 7, 10), vocab=128256, plant=4, seed=2002,
    ),
    # Batched serving mix: 32 sequences, context uniform in [1000, 1600].
    "serving_mix": dict(
        batch=32, num_q_heads=32, num_kv_heads=8, head_dim=128, layers=1,
        ctx=(1000, 1600), tree=("eagle", 60, 7, 10), vocab=128256,
        plant=(1, 7), seed=3003,
    ),
    # 60K context, 48-node tree, full KV plus a SpecPV partial page list of
    # 64 sink tokens + 32 retrieved 64-token blocks + the last 1024 tokens.
    "long_partial": dict(
        batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, layers=1,
        ctx=60000, tree=("eagle", 48, 7, 10), vocab=128256, plant=4,
        partial=dict(sink=64, blocks=32, block_tokens=64, recent=1024),
        seed=4004,
    ),
    # SpecBlock trees (K = 4, up to 3 blocks, <= 128 nodes, depth <= 12) at
    # 64 q heads / 8 kv heads, 16 sequences of 16384 context tokens.
    "specblock": dict(
        batch=16, num_q_heads=64, num_kv_heads=8, head_dim=128, layers=1,
        ctx=16384, tree=("specblock", 128, 12, 4), vocab=151936,
        plant="deepest", seed=5005,
    ),
}

BUCKET_PROBS = (0.6, 0.25, 0.1, 0.05)
BUCKET_BRANCHING = (2, 4, 10, 0)


# ----------------------------------------------------------------------------
# value helpers


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _bf16_normal(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) values rounded to bf16, generated in chunks to bound host memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = bf16_bits_from_f32(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# tree shapes (parent arrays, root = node 0 with parent -1, parent[i] < i)


def node_depths(parents) -> np.ndarray:
    d = np.zeros(len(parents), dtype=np.int64)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def tree_chain(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def tree_random_depth(rng: np.random.Generator, n: int, depth: int) -> np.ndarray:
    """parent[i] uniform over earlier nodes of depth < ``depth``; redrawn until
    the tree reaches exactly that depth (at most n - 1)."""
    if not 0 <= depth <= n - 1:
        raise ValueError(f"a tree of {n} nodes cannot have depth {depth}")
    while True:
        par = [-1]
        dep = [0]
        for i in range(1, n):
            cand = [j for j in range(i) if dep[j] < depth]
            p = cand[int(rng.integers(len(cand)))]
            par.append(p)
            dep.append(dep[p] + 1)
        if max(dep) == depth:
            return np.asarray(par, dtype=np.int32)


def tree_eagle_static(rng: np.random.Generator, num_draft: int, num_steps: int,
                      topk: int, sharpness: float = 2.5) -> np.ndarray:
    """EAGLE-3 style static tree.

    Level by level, the ``topk`` best frontier nodes (by cumulative draft
    log-probability) each get ``topk`` children whose draft log-probabilities
    come from a softmax over random logits; after ``num_steps`` levels the
    ``num_draft - 1`` best nodes overall plus the root are kept.  Scores fall
    strictly along a path, so the kept set is closed under taking parents.
    Nodes are renumbered breadth first, so parent[i] < i.  Redrawn until the
    tree reaches depth ``num_steps``.
    """
    while True:
        score = [0.0]
        par = [-1]
        dep = [0]
        frontier = [0]
        for _step in range(num_steps):
            new = []
            for f in frontier:
                z = np.sort(rng.standard_normal(topk))[::-1] * sharpness
                logp = z - np.log(np.exp(z - z.max()).sum()) - z.max()
                for k in range(topk):
                    score.append(score[f] + float(logp[k]))
                    par.append(f)
                    dep.append(dep[f] + 1)
                    new.append(len(score) - 1)
            new.sort(key=lambda i: -score[i])
            frontier = new[:topk]
        order = sorted(range(1, len(score)), key=lambda i: -score[i])[: num_draft - 1]
        keep = [0] + sorted(order, key=lambda i: (dep[i], -score[i]))
        if max(dep[i] for i in keep) != num_steps:
            continue
        remap = {old: new for new, old in enumerate(keep)}
        out = np.empty(len(keep), dtype=np.int32)
        for new_i, old in enumerate(keep):
            out[new_i] = -1 if old == 0 else remap[par[old]]
        return out


def tree_specblock(rng: np.random.Generator, max_nodes: int, max_depth: int,
                   block: int = 4) -> np.ndarray:
    """SpecBlock style tree from blocks of ``block`` dependent positions.

    Block 1 is a chain of ``block`` positions from the root.  At each position
    a rank bucket b0..b3 is drawn with probabilities (0.6, 0.25, 0.1, 0.05);
    it attaches (2, 4, 10, 0) sibling candidates, the first of which continues
    the chain (0 ends it).  Each candidate at the last position of a block
    starts a chain of the next block.  Blocks continue until ``max_depth``;
    the tree is truncated breadth first to ``max_nodes`` (closure holds since
    parents precede children in breadth-first order).
    """
    par = [-1]
    dep = [0]
    starts = [0]
    while starts and dep[starts[0]] + block <= max_depth:
        next_starts = []
        for s in starts:
            cur = s
            for pos in range(block):
                b = int(rng.choice(4, p=BUCKET_PROBS))
                nb = BUCKET_BRANCHING[b]
                if nb == 0:
                    break
                first = None
                for c in range(nb):
                    par.append(cur)
                    dep.append(dep[cur] + 1)
                    if c == 0:
                        first = len(par) - 1
                    if pos == block - 1:
                        next_starts.append(len(par) - 1)
                cur = first
        starts = next_starts
    # breadth-first renumbering and truncation
    order = sorted(range(len(par)), key=lambda i: (dep[i], i))[:max_nodes]
    remap = {old: new for new, old in enumerate(order)}
    out = np.empty(len(order), dtype=np.int32)
    for new_i, old in enumerate(order):
        out[new_i] = -1 if old == 0 else remap[par[old]]
    return out


def _sibling_distinct_tokens(rng, parents, vocab) -> np.ndarray:
    n = len(parents)
    tok = rng.integers(0, vocab, size=n).astype(np.int32)
    children = {}
    for i in range(1, n):
        children.setdefault(int(parents[i]), []).append(i)
    for kids in children.values():
        seen = set()
        for c in kids:
            while int(tok[c]) in seen:
                tok[c] = int(rng.integers(0, vocab))
            seen.add(int(tok[c]))
    return tok


# ----------------------------------------------------------------------------
# the case container


@dataclass
class VerifyCase:
    """All inputs of one verify step (one or more layers)."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_layers: int
    vocab: int
    # tree (concatenated over sequences; parents/ids are sequence-local)
    cu_nodes: np.ndarray          # int32 [B+1]
    parents: np.ndarray           # int32 [T]
    tokens: np.ndarray            # int32 [T]
    ctx_lens: np.ndarray          # int32 [B]
    # paged pool (per layer), bf16 bits
    num_pages: int
    block_table: np.ndarray       # int32 [B, max_pages_per_seq]
    k_cache: np.ndarray           # uint16 [layers, num_pages, Hkv, P, D]
    v_cache: np.ndarray
    q: np.ndarray                 # uint16 [layers, T, Hq, D]
    tree_k: np.ndarray            # uint16 [layers, T, Hkv, D]
    tree_v: np.ndarray
    logits: Optional[np.ndarray] = None   # float32 [T, V]
    planted_len: Optional[np.ndarray] = None   # int32 [B]
    planted_path: list = field(default_factory=list)  # per seq: local ids
    planted_bonus: Optional[np.ndarray] = None  # int32 [B]
    kv_pages: Optional[np.ndarray] = None  # int32 [sum], logical page ids
    cu_kv_pages: Optional[np.ndarray] = None  # int32 [B+1]
    max_depth: int = 0

    @property
    def total_nodes(self) -> int:
        return int(self.cu_nodes[-1])

    @property
    def max_nodes(self) -> int:
        return int(np.diff(self.cu_nodes).max())

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def nodes_of(self, b: int) -> slice:
        return slice(int(self.cu_nodes[b]), int(self.cu_nodes[b + 1]))


def _partial_pages(rng, L, page, sink, blocks, block_tokens, recent) -> np.ndarray:
    """Logical page ids (ascending, unique) covering the sink tokens, ``blocks``
    retrieved blocks of ``block_tokens`` tokens drawn from between the sink and
    the recent window, and the last ``recent`` tokens."""
    pages = set(range(0, -(-min(sink, L) // page)))
    lo = max(0, L - recent)
    pages.update(range(lo // page, -(-L // page)))
    per = block_tokens // page
    first_blk = -(-sink // block_tokens)
    last_blk = lo // block_tokens  # exclusive: block k covers [k*bt, (k+1)*bt)
    cand = np.arange(first_blk, last_blk)
    if blocks > 0 and len(cand) > 0:
        chosen = rng.choice(cand, size=min(blocks, len(cand)), replace=False)
        for k in chosen:
            pages.update(range(int(k) * per, int(k) * per + per))
    return np.asarray(sorted(p for p in pages if p * page < L), dtype=np.int32)


def make_case(name: str, *, layers: Optional[int] = None, batch: Optional[int] = None,
              ctx=None, seed: Optional[int] = None, with_logits: bool = True,
              with_partial: Optional[bool] = None, parents_list=None,
              num_q_heads=None, num_kv_heads=None, head_dim=None, vocab=None,
              plant=None, partial=None, tree=None, extra_pages: int = 0) -> VerifyCase:
    """Build one verify step of workload ``name`` (keys of ``CONFIGS``).

    Keyword overrides shrink or reshape a workload for tests; ``parents_list``
    supplies explicit trees (one parent array per sequence).
    """
    cfg = dict(CONFIGS[name])
    if layers is not None:
        cfg["layers"] = layers
    if batch is not None:
        cfg["batch"] = batch
    if ctx is not None:
        cfg["ctx"] = ctx
    if seed is not None:
        cfg["seed"] = seed
    for k, v in (("num_q_heads", num_q_heads), ("num_kv_heads", num_kv_heads),
                 ("head_dim", head_dim), ("vocab", vocab), ("plant", plant),
                 ("partial", partial), ("tree", tree)):
        if v is not None:
            cfg[k] = v
    B = cfg["batch"]
    Hq, Hkv, D = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    layers_n = cfg["layers"]
    V = cfg["vocab"]
    P = PAGE_SIZE
    ss = np.random.SeedSequence(cfg["seed"])
    r_tree, r_ctx, r_tok, r_q, r_kv, r_cache, r_logit, r_pool, r_part, r_plant = [
        np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(10)]

    # trees
    if parents_list is None:
        parents_list = []
        kind = cfg["tree"][0]
        for _ in range(B):
            if kind == "random_depth":
                parents_list.append(tree_random_depth(r_tree, cfg["tree"][1], cfg["tree"][2]))
            elif kind == "eagle":
                parents_list.append(tree_eagle_static(r_tree, cfg["tree"][1], cfg["tree"][2], cfg["tree"][3]))
            elif kind == "specblock":
                parents_list.append(tree_specblock(r_tree, cfg["tree"][1], cfg["tree"][2], cfg["tree"][3]))
            elif kind == "chain":
                parents_list.append(tree_chain(cfg["tree"][1]))
            else:
                raise ValueError(kind)
    parents_list = [np.asarray(p, dtype=np.int32) for p in parents_list]
    assert len(parents_list) == B
    ns = [len(p) for p in parents_list]
    cu_nodes = np.zeros(B + 1, dtype=np.int32)
    cu_nodes[1:] = np.cumsum(ns)
    T = int(cu_nodes[-1])
    parents = np.concatenate(parents_list).astype(np.int32)
    depths = [node_depths(p) for p in parents_list]
    max_depth = int(max(int(d.max()) for d in depths))

    # context lengths
    c = cfg["ctx"]
    if isinstance(c, tuple):
        ctx_lens = r_ctx.integers(c[0], c[1] + 1, size=B).astype(np.int32)
    elif isinstance(c, (list, np.ndarray)):
        ctx_lens = np.asarray(c, dtype=np.int32)
    else:
        ctx_lens = np.full(B, int(c), dtype=np.int32)

    # tokens (siblings distinct)
    tokens = np.concatenate([_sibling_distinct_tokens(r_tok, p, V) for p in parents_list]).astype(np.int32)

    # paged pool: every sequence owns pages for its context plus the commit
    # slots L .. L + max_depth; physical ids are a random permutation.
    need = [-(-(int(L) + max_depth + 1) // P) for L in ctx_lens]
    num_pages = int(sum(need)) + int(extra_pages)
    perm = r_pool.permutation(num_pages).astype(np.int32)
    mpps = max(need)
    block_table = np.full((B, mpps), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        block_table[b, : need[b]] = perm[o: o + need[b]]
        o += need[b]

    k_cache = _bf16_normal(r_cache, (layers_n, num_pages, Hkv, P, D))
    v_cache = _bf16_normal(r_cache, (layers_n, num_pages, Hkv, P, D))
    q = _bf16_normal(r_q, (layers_n, T, Hq, D))
    tree_k = _bf16_normal(r_kv, (layers_n, T, Hkv, D))
    tree_v = _bf16_normal(r_kv, (layers_n, T, Hkv, D))

    case = VerifyCase(
        name=name, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
        num_layers=layers_n, vocab=V, cu_nodes=cu_nodes, parents=parents, tokens=tokens,
        ctx_lens=ctx_lens, num_pages=num_pages, block_table=block_table,
        k_cache=k_cache, v_cache=v_cache, q=q, tree_k=tree_k, tree_v=tree_v,
        max_depth=max_depth)

    # partial page lists
    part = cfg.get("partial") if with_partial is not False else None
    if with_partial and part is None:
        part = dict(sink=64, blocks=32, block_tokens=64, recent=1024)
    if part is not None:
        lists = [_partial_pages(r_part, int(ctx_lens[b]), P, **part) for b in range(B)]
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum([len(x) for x in lists])
        case.kv_pages = (np.concatenate(lists) if lists else np.zeros(0)).astype(np.int32)
        case.cu_kv_pages = cu

    if with_logits:
        _plant_logits(case, r_logit, r_plant, cfg["plant"], depths, parents_list)
    return case


def _plant_logits(case: VerifyCase, r_logit, r_plant, plant, depths, parents_list):
    T, V = case.total_nodes, case.vocab
    logits = np.empty((T, V), dtype=np.float32)
    chunk = max(1, (1 << 24) // V)
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        logits[s:e] = r_logit.standard_normal((e - s, V), dtype=np.float32)
    plens = np.zeros(case.batch, dtype=np.int32)
    bonus = np.zeros(case.batch, dtype=np.int32)
    paths = []
    for b in range(case.batch):
        par = parents_list[b]
        dep = depths[b]
        base = int(case.cu_nodes[b])
        n = len(par)
        if isinstance(plant, tuple):
            a = int(r_plant.integers(plant[0], plant[1] + 1))
        elif plant == "deepest":
            a = int(r_plant.integers(1, int(dep.max()) + 1)) if dep.max() > 0 else 0
        else:
            a = int(plant)
        a = min(a, int(dep.max()))
        ends = np.nonzero(dep == a)[0]
        end = int(ends[int(r_plant.integers(len(ends)))])
        path = [end]
        while path[-1] != 0:
            path.append(int(par[path[-1]]))
        path = path[::-1]
        children = {}
        for i in range(1, n):
            children.setdefault(int(par[i]), []).append(i)
        on_path = {path[j]: path[j + 1] for j in range(a)}
        for node in range(n):
            row = logits[base + node]
            if node in on_path:
                tgt = int(case.tokens[base + on_path[node]])
            else:
                banned = {int(case.tokens[base + c]) for c in children.get(node, [])}
                tgt = int(r_plant.integers(0, V))
                while tgt in banned:
                    tgt = int(r_plant.integers(0, V))
            row[tgt] = row.max() + np.float32(1.0)
            if node == path[-1]:
                bonus[b] = tgt
        plens[b] = a
        paths.append(path)
    case.logits = logits
    case.planted_len = plens
    case.planted_path = paths
    case.planted_bonus = bonus


def make_sampling_inputs(case: VerifyCase, *, seed: int = 0, sharpness: float = 1.0, closeness: float = 0.5,
                         draft: str = "near"):
    """Inputs of stochastic acceptance for a case that has logits: per node a
    draft probability vector (float32 [T, V], each row sums to 1), children
    tokens redrawn independently from their parent's draft row, and two
    uniforms per node in [0, 1).

    draft "near": rows proportional to exp(sharpness * (logits + noise)), the
    noise N(0, closeness) so that drafts resemble the target; "flat": uniform
    rows.  The case's tokens are replaced (int32 [T]); the root's stays 0."""
    assert case.logits is not None
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x5A3]))
    T, V = case.logits.shape
    if draft == "flat":
        q = np.full((T, V), 1.0 / V, dtype=np.float64)
    else:
        z = sharpness * (case.logits.astype(np.float64) + rng.normal(0.0, closeness, size=(T, V)))
        z -= z.max(axis=1, keepdims=True)
        q = np.exp(z)
        q /= q.sum(axis=1, keepdims=True)
    q32 = q.astype(np.float32)
    q32 /= q32.sum(axis=1, keepdims=True, dtype=np.float64).astype(np.float32)
    tokens = np.zeros(T, dtype=np.int32)
    cdf = None
    for b in range(case.batch):
        n0, n1 = int(case.cu_nodes[b]), int(case.cu_nodes[b + 1])
        for c in range(n0 + 1, n1):
            par = n0 + int(case.parents[c])
            cdf = np.cumsum(q[par])
            tokens[c] = min(V - 1, int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right")))
    u_accept = rng.random(T).astype(np.float32)
    u_bonus = rng.random(T).astype(np.float32)
    return q32, tokens, u_accept, u_bonus
