"""Seeded synthetic workloads for one tree-verification step.

This module only *makes inputs*: token-tree shapes, drafted tokens, target
logits, drafter distributions, uniforms and the Q/K/V of one attention layer,
with the shapes and value distributions of the LLaMA/OPT serving workloads that
SpecInfer (arXiv 2305.09781, sec. 6) measures. It performs no step of the
verification method itself (no linearisation, no attention, no acceptance test):
both the CUDA library and the test-only oracle consume the very same arrays.

Randomness: numpy ``default_rng(seed)`` (PCG64). Generation order per request:
topology -> target logits -> drafter logits -> drafted tokens -> uniforms ->
Q -> K/V of the new nodes -> K/V of the prefix. bfloat16 values are the
round-to-nearest-even of float32 draws and are carried as uint16 bit patterns.

Array conventions (every per-node array is in *input node order*):
  parent  [B][n_max] int32   -1 for the root, -1 padding beyond n_nodes[b]
  tokens  [B][n_max] int32   token of each node (the root's is the committed one)
  q, k_new, v_new [B][n_max][H][d]  (token-major, as a QKV projection writes it)
  k_cache, v_cache [B][H][L_max][d]  rows 0..prefix_len[b]-1 filled, rest zero
  logits  [B][NP][V] float32; node v reads row p_row[b][v] (identity if None)
  ssm     [B][NQ][V] float32 drafter probabilities; child v tests row q_row[b][v]
  uniforms [B][2][n_max] float32 in [0,1): [0][v] accept test of child v,
           [1][u] the final sample drawn at node u
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CONFIG_NAMES = ("tiny", "llama7b", "merge", "long65b", "opt30b")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    """Drafter probabilities from drafter logits (input synthesis only)."""
    z = z.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


@dataclass
class Workload:
    name: str
    B: int
    H: int
    d: int
    dtype: str                 # "f32" or "bf16"
    V: int
    n_max: int
    L_max: int
    verify: str                # "greedy", "mss" or "both"
    temperature: float
    prefix_len: np.ndarray
    tree_mode: str             # "widths", "parent" or "chains"
    n_nodes: np.ndarray | None = None
    parent: np.ndarray | None = None
    tokens: np.ndarray | None = None
    widths: tuple | None = None
    chains: np.ndarray | None = None       # [B][C][len]
    root_token: np.ndarray | None = None   # [B]
    logits: np.ndarray | None = None
    p_row: np.ndarray | None = None
    ssm: np.ndarray | None = None
    q_row: np.ndarray | None = None
    uniforms: np.ndarray | None = None
    q: np.ndarray | None = None
    k_new: np.ndarray | None = None
    v_new: np.ndarray | None = None
    k_cache: np.ndarray | None = None
    v_cache: np.ndarray | None = None
    meta: dict = field(default_factory=dict)

    @property
    def total_nodes(self) -> int:
        return int(np.sum(self.n_nodes)) if self.n_nodes is not None else -1


def _expansion_parent(widths) -> np.ndarray:
    """Level-order shape of an expansion drafter's tree: each node of depth i-1
    gets widths[i-1] children, numbered consecutively (drafter rank order)."""
    par = [-1]
    level = [0]
    for k in widths:
        nxt = []
        for u in level:
            for _ in range(k):
                par.append(u)
                nxt.append(len(par) - 1)
        level = nxt
    return np.array(par, np.int32)


def _pad(a: np.ndarray, n_max: int, fill) -> np.ndarray:
    out = np.full(n_max, fill, a.dtype)
    out[: len(a)] = a
    return out


def _qkv(rng, B, n_max, H, d, L_max, prefix_len, dtype, scale=1.0):
    """Q, K_new, V_new for the tree nodes and the K/V prefix cache, N(0, scale^2).
    The prefix K/V of request b comes from its own child generator
    (rng.spawn(B)[b]: K, then V), so the requests are drawn on several threads
    with a result that does not depend on the thread count."""
    def draw(g, shape):
        x = g.standard_normal(shape, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        return f32_to_bf16_bits(x) if dtype == "bf16" else x

    q = draw(rng, (B, n_max, H, d))
    k_new = draw(rng, (B, n_max, H, d))
    v_new = draw(rng, (B, n_max, H, d))
    cdt = np.uint16 if dtype == "bf16" else np.float32
    k_cache = np.zeros((B, H, L_max, d), cdt)
    v_cache = np.zeros((B, H, L_max, d), cdt)
    children = rng.spawn(B)

    def fill(b):
        P = int(prefix_len[b])
        k_cache[b, :, :P] = draw(children[b], (H, P, d))
        v_cache[b, :, :P] = draw(children[b], (H, P, d))

    with ThreadPoolExecutor(max_workers=min(B, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(B)))
    return q, k_new, v_new, k_cache, v_cache


def _topk_stable(row: np.ndarray, k: int) -> np.ndarray:
    """The k largest entries of row, best first, ties to the lower index: the
    first k of a stable argsort of -row, without sorting the whole row."""
    if k >= row.size:
        return np.argsort(-row, kind="stable")[:k]
    thr = np.partition(row, row.size - k)[row.size - k]     # the k-th largest value
    cand = np.nonzero(row >= thr)[0]                         # increasing index
    order = np.lexsort((cand, -row[cand]))                   # by value desc, then index asc
    return cand[order][:k]


def _round_up(x, m):
    return (x + m - 1) // m * m


def make(name: str, seed: int | None = None, *, attention: bool = True, scale_down: int = 1,
         batch: int | None = None) -> Workload:
    """Build one of the five workloads.

    name       : tiny | llama7b | merge | long65b | opt30b
    seed       : defaults to the workload's own seed (0..4)
    attention  : False skips Q/K/V (verification-only callers)
    scale_down : divides batch (and the long prefix) for reduced-size parity runs
    batch      : the LLaMA-7B-shaped layer at another batch size (the other
                 workloads keep theirs)
    """
    seeds = dict(tiny=0, llama7b=1, merge=2, long65b=3, opt30b=4)
    if name not in seeds:
        raise ValueError(f"unknown workload {name!r}; choose from {CONFIG_NAMES}")
    rng = np.random.default_rng(seeds[name] if seed is None else seed)
    if batch is not None:
        if name != "llama7b":
            raise ValueError("batch overrides only the llama7b workload")
        return _make_llama7b(rng, attention, 1, batch=int(batch))
    return globals()["_make_" + name](rng, attention, max(1, int(scale_down)))


# ----------------------------------------------------------------------------
def _expansion_workload(rng, *, name, B, H, d, dtype, P, widths, V, sigma_t, sigma_noise,
                        independent_ssm, plant, verify, attention):
    par1 = _expansion_parent(widths)
    n = len(par1)
    n_max = n
    n_internal = int(np.max(par1)) + 1          # level order: internal nodes come first
    parent = np.tile(par1, (B, 1))
    n_nodes = np.full(B, n, np.int32)
    prefix_len = np.full(B, P, np.int32)
    L_max = _round_up(P + n_max, 64)

    # target logits per node (the distribution of the token that follows it)
    logits = (rng.standard_normal((B, n, V), dtype=np.float32) * np.float32(sigma_t))
    ssm = None
    q_row = None
    if verify in ("mss", "both") or plant == "topk":
        if independent_ssm:
            z = rng.standard_normal((B, n_internal, V), dtype=np.float32) * np.float32(sigma_t)
        else:
            z = logits[:, :n_internal] + rng.standard_normal((B, n_internal, V), dtype=np.float32) * np.float32(sigma_noise)
        ssm = _softmax_rows(z)
        q_row = np.where(parent >= 0, parent, 0).astype(np.int32)

    tokens = np.zeros((B, n_max), np.int32)
    tokens[:, 0] = rng.integers(0, V, B)
    for b in range(B):
        for u in range(n_internal):
            kids = np.nonzero(par1 == u)[0]
            k = len(kids)
            if plant == "topk":
                # the drafter's top-k tokens at u, best first
                order = _topk_stable(ssm[b, u], k)
                tokens[b, kids] = order
            else:
                # first child = target argmax with probability `plant`, the other
                # children random distinct tokens
                am = int(np.argmax(logits[b, u]))
                used = {am}
                if rng.random() < plant:
                    first = am
                else:
                    first = am
                    while first in used:
                        first = int(rng.integers(0, V))
                used.add(first)
                tokens[b, kids[0]] = first
                for c in kids[1:]:
                    t = int(rng.integers(0, V))
                    while t in used:
                        t = int(rng.integers(0, V))
                    used.add(t)
                    tokens[b, c] = t
    uniforms = rng.random((B, 2, n_max), dtype=np.float32)
    w = Workload(name=name, B=B, H=H, d=d, dtype=dtype, V=V, n_max=n_max, L_max=L_max, verify=verify,
                 temperature=1.0, prefix_len=prefix_len, tree_mode="widths", n_nodes=n_nodes, parent=parent,
                 tokens=tokens, widths=tuple(widths), logits=logits, ssm=ssm, q_row=q_row, uniforms=uniforms)
    if attention:
        w.q, w.k_new, w.v_new, w.k_cache, w.v_cache = _qkv(rng, B, n_max, H, d, L_max, prefix_len, dtype)
    return w


def _make_tiny(rng, attention, sd):
    """1 request, prefix 64, widths (2,2,1), 4 heads x 64, fp32, vocab 256;
    target logits N(0, 2^2); drafter = softmax of independent N(0, 2^2) logits;
    children = drafter top-k."""
    return _expansion_workload(rng, name="tiny", B=1, H=4, d=64, dtype="f32", P=64, widths=(2, 2, 1), V=256,
                               sigma_t=2.0, sigma_noise=0.0, independent_ssm=True, plant="topk",
                               verify="both", attention=attention)


def _make_llama7b(rng, attention, sd, batch=None):
    """LLaMA-7B-shaped layer: batch 8, 32 heads x 128, bf16, prefix 2048,
    widths (1,1,3,1,1,1,1,1) -> 21 nodes; greedy, vocab 32000, logits N(0, 3^2);
    first child planted as the target argmax with probability 0.68."""
    return _expansion_workload(rng, name="llama7b", B=batch or max(1, 8 // sd), H=32, d=128, dtype="bf16", P=2048,
                               widths=(1, 1, 3, 1, 1, 1, 1, 1), V=32000, sigma_t=3.0, sigma_noise=0.0,
                               independent_ssm=False, plant=0.68, verify="greedy", attention=attention)


def _make_opt30b(rng, attention, sd):
    """OPT-30B-shaped high batch: batch 64, 56 heads x 128, bf16, prefix 1024,
    widths (2,2,2,2,1) -> 47 nodes; MSS over vocab 50272, target N(0, 3^2),
    drafter logits = target + N(0, 1.5^2); children = drafter top-k."""
    return _expansion_workload(rng, name="opt30b", B=max(1, 64 // sd), H=56, d=128, dtype="bf16", P=1024,
                               widths=(2, 2, 2, 2, 1), V=50272, sigma_t=3.0, sigma_noise=1.5,
                               independent_ssm=False, plant="topk", verify="mss", attention=attention)


def _make_long65b(rng, attention, sd):
    """Long-context LLaMA-65B-shaped layer: batch 4, 64 heads x 128, bf16,
    prefix 16384, random topology of 128 nodes (parent uniform over earlier
    nodes of depth < 12); tokens drawn i.i.d. from the drafter at the parent;
    greedy + MSS over vocab 32000, target N(0, 3^2), drafter = target + N(0, 1)."""
    B, H, d, V, n, P = max(1, 4 // sd), 64, 128, 32000, 128, 16384 // sd
    parent = np.full((B, n), -1, np.int32)
    for b in range(B):
        depth = np.zeros(n, np.int32)
        for v in range(1, n):
            allowed = np.nonzero(depth[:v] < 12)[0]
            u = int(allowed[rng.integers(0, len(allowed))])
            parent[b, v] = u
            depth[v] = depth[u] + 1
    n_nodes = np.full(B, n, np.int32)
    prefix_len = np.full(B, P, np.int32)
    L_max = _round_up(P + n, 64)
    logits = rng.standard_normal((B, n, V), dtype=np.float32) * np.float32(3.0)
    ssm = _softmax_rows(logits + rng.standard_normal((B, n, V), dtype=np.float32))
    q_row = np.where(parent >= 0, parent, 0).astype(np.int32)
    tokens = np.zeros((B, n), np.int32)
    tokens[:, 0] = rng.integers(0, V, B)
    for b in range(B):
        cdf = np.cumsum(ssm[b].astype(np.float64), axis=-1)
        for v in range(1, n):
            u = parent[b, v]
            x = int(np.searchsorted(cdf[u], rng.random() * cdf[u, -1], side="right"))
            tokens[b, v] = min(x, V - 1)
    uniforms = rng.random((B, 2, n), dtype=np.float32)
    w = Workload(name="long65b", B=B, H=H, d=d, dtype="bf16", V=V, n_max=n, L_max=L_max, verify="both",
                 temperature=1.0, prefix_len=prefix_len, tree_mode="parent", n_nodes=n_nodes, parent=parent,
                 tokens=tokens, logits=logits, ssm=ssm, q_row=q_row, uniforms=uniforms)
    if attention:
        w.q, w.k_new, w.v_new, w.k_cache, w.v_cache = _qkv(rng, B, n, H, d, L_max, prefix_len, "bf16")
    return w


def _make_merge(rng, attention, sd):
    """Merge-based trees: batch 16, 32 heads x 128, bf16, prefixes U[512, 4096];
    3 drafter chains of 8 tokens; chain j >= 1 copies a uniformly chosen earlier
    chain position by position while a Bernoulli(0.6) succeeds (at most 7
    shared), then continues with fresh tokens, the first of which differs from
    the copied chain's. MSS, vocab 32000, T = 1, target N(0, 3^2), drafter logits
    = target at the parent + N(0, 1) per (chain, position).

    Row layout (the merge itself is left to tree_build's chains mode):
      logits [B][1 + C*len][V]: row 0 = after the root, row 1 + c*len + p =
             after chain c's p-th token;
      ssm    [B][C*len][V]: row c*len + p = chain c's drafter before its p-th token.
    """
    B, H, d, V, Cn, ln = max(1, 16 // sd), 32, 128, 32000, 3, 8
    prefix_len = rng.integers(512, 4097, B).astype(np.int32)
    n_max = 1 + Cn * ln
    L_max = _round_up(int(prefix_len.max()) + n_max, 64)
    chains = np.zeros((B, Cn, ln), np.int32)
    root_token = rng.integers(0, V, B).astype(np.int32)
    logits = np.zeros((B, 1 + Cn * ln, V), np.float32)
    ssm = np.zeros((B, Cn * ln, V), np.float32)
    share = np.zeros((B, Cn), np.int32)
    src_chain = np.zeros((B, Cn), np.int32)
    for b in range(B):
        logits[b, 0] = rng.standard_normal(V, dtype=np.float32) * np.float32(3.0)
        for c in range(Cn):
            s, i = 0, 0
            if c > 0:
                i = int(rng.integers(0, c))
                while s < ln - 1 and rng.random() < 0.6:
                    s += 1
            share[b, c], src_chain[b, c] = s, i
            for p in range(ln):
                parent_row = 0 if p == 0 else 1 + c * ln + p - 1
                if p < s:
                    chains[b, c, p] = chains[b, i, p]
                    logits[b, 1 + c * ln + p] = logits[b, 1 + i * ln + p]
                    ssm[b, c * ln + p] = ssm[b, i * ln + p]
                    continue
                z = logits[b, parent_row] + rng.standard_normal(V, dtype=np.float32)
                qd = _softmax_rows(z[None])[0]
                ssm[b, c * ln + p] = qd
                cdf = np.cumsum(qd.astype(np.float64))
                while True:
                    t = min(int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right")), V - 1)
                    if not (c > 0 and p == s and t == chains[b, i, p]):
                        break
                chains[b, c, p] = t
                logits[b, 1 + c * ln + p] = rng.standard_normal(V, dtype=np.float32) * np.float32(3.0)
    uniforms = rng.random((B, 2, n_max), dtype=np.float32)
    w = Workload(name="merge", B=B, H=H, d=d, dtype="bf16", V=V, n_max=n_max, L_max=L_max, verify="mss",
                 temperature=1.0, prefix_len=prefix_len, tree_mode="chains", chains=chains,
                 root_token=root_token, logits=logits, ssm=ssm, uniforms=uniforms,
                 meta=dict(share=share, src_chain=src_chain))
    if attention:
        w.q, w.k_new, w.v_new, w.k_cache, w.v_cache = _qkv(rng, B, n_max, H, d, L_max, prefix_len, "bf16")
    return w


def sequence_batch(w: Workload) -> tuple[Workload, np.ndarray]:
    """The sequence-based decoding baseline of SpecInfer Fig. 4 (left) / Fig. 11
    as inputs: every root-to-leaf path of every request becomes a request of its
    own -- a chain over the path's nodes, with its own copy of the prefix K/V.
    Returns the chain workload (attention inputs only) and path_nodes
    [paths][len] = (request, input node) of each chain position (-1 padding).
    Needs a workload built with attention and a parent array."""
    assert w.q is not None and w.parent is not None, "sequence_batch needs attention inputs and a parent array"
    paths = []
    for b in range(w.B):
        n = int(w.n_nodes[b])
        par = w.parent[b, :n]
        leaves = [v for v in range(n) if not np.any(par == v)]
        for leaf in leaves:
            p, u = [], leaf
            while u != -1:
                p.append(u)
                u = int(par[u])
            paths.append((b, p[::-1]))
    S = len(paths)
    n_max = max(len(p) for _, p in paths)
    P = np.array([w.prefix_len[b] for b, _ in paths], np.int32)
    L_max = _round_up(int(P.max()) + n_max, 64)
    path_nodes = np.full((S, n_max, 2), -1, np.int32)
    parent = np.full((S, n_max), -1, np.int32)
    n_nodes = np.zeros(S, np.int32)
    q = np.zeros((S, n_max) + w.q.shape[2:], w.q.dtype)
    k_new, v_new = np.zeros_like(q), np.zeros_like(q)
    k_cache = np.zeros((S, w.H, L_max, w.d), w.k_cache.dtype)
    v_cache = np.zeros_like(k_cache)
    for s, (b, p) in enumerate(paths):
        m = len(p)
        n_nodes[s] = m
        parent[s, 1:m] = np.arange(m - 1)
        path_nodes[s, :m, 0] = b
        path_nodes[s, :m, 1] = p
        q[s, :m], k_new[s, :m], v_new[s, :m] = w.q[b, p], w.k_new[b, p], w.v_new[b, p]
        k_cache[s, :, :P[s]] = w.k_cache[b, :, :P[s]]
        v_cache[s, :, :P[s]] = w.v_cache[b, :, :P[s]]
    seq = Workload(name=w.name + "-sequences", B=S, H=w.H, d=w.d, dtype=w.dtype, V=1, n_max=n_max, L_max=L_max,
                   verify="greedy", temperature=1.0, prefix_len=P, tree_mode="parent", n_nodes=n_nodes,
                   parent=parent, tokens=np.zeros((S, n_max), np.int32),
                   logits=np.zeros((S, n_max, 1), np.float32), uniforms=np.zeros((S, 2, n_max), np.float32))
    seq.q, seq.k_new, seq.v_new, seq.k_cache, seq.v_cache = q, k_new, v_new, k_cache, v_cache
    return seq, path_nodes
