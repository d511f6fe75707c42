"""Shared helpers of the GPU parity tests: oracle-side tree inputs, cached
workloads, device/oracle comparisons."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from tree_speculative_verification_gb300 import workloads as wl
from tree_speculative_verification_gb300.workloads import bf16_bits_to_f32


@functools.lru_cache(maxsize=4)
def workload(name: str, scale_down: int = 1, attention: bool = True):
    return wl.make(name, attention=attention, scale_down=scale_down)


def oracle_tree(w):
    """The oracle's own view of the tree: (parent, tokens, n_nodes, p_row, q_row),
    built with the oracle's widths/merge code, never with the library's."""
    B, n_max = w.B, w.n_max
    if w.tree_mode == "chains":
        parent = np.full((B, n_max), -1, np.int32)
        tokens = np.zeros((B, n_max), np.int32)
        p_row = np.full((B, n_max), 0, np.int32)
        q_row = np.zeros((B, n_max), np.int32)
        n_nodes = np.zeros(B, np.int32)
        for b in range(B):
            par, tok, src = oracle.merge_chains(w.chains[b], int(w.root_token[b]), n_max)
            n = len(par)
            n_nodes[b] = n
            parent[b, :n], tokens[b, :n] = par, tok
            p_row[b, :n] = src + 1
            q_row[b, :n] = np.maximum(src, 0)
        return parent, tokens, n_nodes, p_row, q_row
    if w.tree_mode == "widths":
        par = oracle.widths_parent(w.widths)
        assert np.array_equal(np.tile(par, (B, 1)), w.parent), "generator and oracle disagree on the expansion shape"
    q_row = w.q_row if w.q_row is not None else np.zeros((B, n_max), np.int32)
    return w.parent, w.tokens, w.n_nodes, None, q_row


def f64(a):
    return (bf16_bits_to_f32(a) if a.dtype == np.uint16 else a).astype(np.float64)


def device_tree(step):
    t = step.tree
    g = lambda x: x.cpu().numpy()
    W = t.anc.shape[2]
    words = g(t.anc).astype(np.uint32)
    bits = ((words[..., None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(t.B, t.n_max, W * 32)[..., :t.n_max]
    return dict(n_nodes=g(t.n_nodes), perm=g(t.perm), dfs_of=g(t.dfs_of), parent=g(t.parent), token=g(t.token),
                depth=g(t.depth), pos=g(t.pos), sub_end=g(t.sub_end), anc=bits.astype(np.uint8))


def compare_trees(dev, ref, n_nodes, prefix_len=None):
    B = len(n_nodes)
    assert dev["n_nodes"].tolist() == list(n_nodes)
    for b in range(B):
        n = int(n_nodes[b])
        for k in ("perm", "dfs_of", "parent", "token", "depth", "sub_end"):
            assert dev[k][b, :n].tolist() == ref[k][b, :n].tolist(), (k, b)
            assert (dev[k][b, n:] == -1).all(), (k, b)
        assert np.array_equal(dev["anc"][b, :n, :n], ref["anc"][b, :n, :n]), b
        assert not dev["anc"][b, n:].any() and not dev["anc"][b, :, n:].any()
        if prefix_len is not None:
            assert dev["pos"][b, :n].tolist() == (ref["depth"][b, :n] + prefix_len[b]).tolist()


def sample_rows(w, n_nodes, k, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(k):
        b = int(rng.integers(0, w.B))
        rows.append((b, int(rng.integers(0, w.H)), int(rng.integers(0, n_nodes[b]))))
    # always include the root and the last node of the first request
    rows += [(0, 0, 0), (0, w.H - 1, int(n_nodes[0]) - 1)]
    return np.array(rows, np.int32)


def attention_error(step, w, n_nodes, parent, rows):
    ref = oracle.tree_attention_rows(w.q, w.k_new, w.v_new, w.k_cache, w.v_cache, w.prefix_len, n_nodes, parent,
                                     rows, nthreads=0)
    out = step.out.float().cpu().numpy()
    got = out[rows[:, 0], rows[:, 2], rows[:, 1]].astype(np.float64)
    return float(np.max(np.abs(got - ref))), got, ref


def torch_sync():
    torch.cuda.synchronize()


def low_margin_prob(logits_row, T=1.0, eps=1e-6):
    """Probability that an inverse-CDF draw u * S from p = softmax(logits / T)
    lands within eps * S of a cumulative-sum boundary: the length of the union
    of the windows [C(x) - eps, C(x) + eps] inside [0, 1). The expected count
    of low-margin draws, from which the exclusion bounds of the sampling
    verifiers' parity checks are derived."""
    z = np.asarray(logits_row, np.float64) / T
    p = np.exp(z - z.max())
    c = np.concatenate([[0.0], np.cumsum(p / p.sum())])
    lo, hi = np.maximum(c - eps, 0.0), np.minimum(c + eps, 1.0)
    gap_start = lo[1:] > np.maximum.accumulate(hi)[:-1]       # a window that starts a new run
    run_id = np.concatenate([[0], np.cumsum(gap_start)])
    starts = np.full(run_id[-1] + 1, np.inf)
    ends = np.zeros(run_id[-1] + 1)
    np.minimum.at(starts, run_id, lo)
    np.maximum.at(ends, run_id, hi)
    return float(np.sum(ends - starts))


def exclusion_bound(probs):
    """At most this many requests may hold a low-margin decision: the expected
    number (sum of per-request probabilities) plus four standard deviations of
    the binomial-like count, plus 2."""
    e = float(np.sum(probs))
    return e + 4.0 * np.sqrt(e) + 2.0
