"""Pins of the oracle's tree attention.

SpecInfer (arXiv 2305.09781) Def. 4.1: TreeAttention(u) = Attention(S_u); the
sec. 4.2 correctness argument: the topology-aware mask gives every node exactly
the attention of its own root-to-node sequence. Checked three independent ways:
(i) every root-to-leaf path run as its own causal sequence (Eq. 1-4 in dense
matrix form), (ii) the dense masked formula softmax(QK^T/sqrt(d) + M) V of
"How Speculative Decoding in LLM Serving Actually Works" with M built from
networkx ancestors, (iii) special cases: a chain is plain causal attention,
a single node is one-query decoding.
"""
import networkx as nx
import numpy as np
import pytest

import oracle
from tree_speculative_verification_gb300.workloads import bf16_bits_to_f32, f32_to_bf16_bits


def _causal_attention(q, k, v, scale):
    """Eq. 1-4 for one head: q [l][d], k/v [l][d]; row j sees keys 0..j."""
    a = (q @ k.T) * scale
    l = a.shape[0]
    a = np.where(np.tril(np.ones((l, l), bool)), a, -np.inf)
    a = a - a.max(axis=1, keepdims=True)
    w = np.exp(a)
    w /= w.sum(axis=1, keepdims=True)
    return w @ v


def _case(rng, B, H, d, n, P, bf16=False):
    par = np.full((B, n), -1, np.int32)
    for b in range(B):
        for v in range(1, n):
            par[b, v] = rng.integers(0, v)
        perm = rng.permutation(n - 1) + 1          # keep the root at 0, shuffle the rest
        perm = np.concatenate([[0], perm])
        inv = np.argsort(perm)
        par[b] = [-1 if par[b, perm[i]] < 0 else inv[par[b, perm[i]]] for i in range(n)]
    L_max = P + n + 3
    draw = lambda *s: rng.standard_normal(s).astype(np.float32)
    q, kn, vn = draw(B, n, H, d), draw(B, n, H, d), draw(B, n, H, d)
    kc, vc = np.zeros((B, H, L_max, d), np.float32), np.zeros((B, H, L_max, d), np.float32)
    kc[:, :, :P] = draw(B, H, P, d)
    vc[:, :, :P] = draw(B, H, P, d)
    if bf16:
        q, kn, vn, kc, vc = map(f32_to_bf16_bits, (q, kn, vn, kc, vc))
    return par, q, kn, vn, kc, vc


def _f64(a):
    return (bf16_bits_to_f32(a) if a.dtype == np.uint16 else a).astype(np.float64)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("seed", range(3))
def test_paths_equal_independent_causal_sequences(seed, bf16):
    rng = np.random.default_rng(seed)
    B, H, d, n, P = 2, 2, 16, 13, 9
    par, q, kn, vn, kc, vc = _case(rng, B, H, d, n, P, bf16)
    nn = np.full(B, n, np.int32)
    pl = np.full(B, P, np.int32)
    rows = oracle.all_rows(B, H, nn)
    out = oracle.tree_attention_rows(q, kn, vn, kc, vc, pl, nn, par, rows)
    got = {tuple(r): out[i] for i, r in enumerate(rows)}
    Q, KN, VN, KC, VC = map(_f64, (q, kn, vn, kc, vc))
    scale = 1.0 / np.sqrt(d)
    for b in range(B):
        kids = {u: [v for v in range(n) if par[b, v] == u] for u in range(n)}
        for leaf in [u for u in range(n) if not kids[u]]:
            path = [leaf]
            while par[b, path[-1]] >= 0:
                path.append(int(par[b, path[-1]]))
            path = path[::-1]
            for h in range(H):
                # the sequence prefix ; path as one causal sequence
                k = np.concatenate([KC[b, h, :P], KN[b, path, h]])
                v = np.concatenate([VC[b, h, :P], VN[b, path, h]])
                qs = np.concatenate([np.zeros((P, d)), Q[b, path, h]])
                ref = _causal_attention(qs, k, v, scale)[P:]
                for j, u in enumerate(path):
                    np.testing.assert_allclose(got[(b, h, u)], ref[j], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_dense_mask_formula(seed):
    rng = np.random.default_rng(10 + seed)
    B, H, d, n, P = 1, 3, 8, 17, 5
    par, q, kn, vn, kc, vc = _case(rng, B, H, d, n, P)
    g = nx.DiGraph([(int(par[0, v]), v) for v in range(n) if par[0, v] >= 0])
    g.add_nodes_from(range(n))
    # M: prefix always visible; tree key w visible to node v iff w is v or an ancestor
    M = np.full((n, P + n), -np.inf)
    M[:, :P] = 0.0
    for v in range(n):
        for w in nx.ancestors(g, v) | {v}:
            M[v, P + w] = 0.0
    nn, pl = np.array([n], np.int32), np.array([P], np.int32)
    out = oracle.tree_attention_rows(q, kn, vn, kc, vc, pl, nn, par, oracle.all_rows(B, H, nn))
    out = out.reshape(H, n, d)
    for h in range(H):
        K = np.concatenate([kc[0, h, :P], kn[0, :, h]]).astype(np.float64)
        Vv = np.concatenate([vc[0, h, :P], vn[0, :, h]]).astype(np.float64)
        A = q[0, :, h].astype(np.float64) @ K.T / np.sqrt(d) + M
        A -= A.max(axis=1, keepdims=True)
        W = np.exp(A)
        W /= W.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(out[h], W @ Vv, rtol=1e-12, atol=1e-12)


def test_chain_is_causal_attention():
    rng = np.random.default_rng(7)
    B, H, d, n, P = 1, 1, 32, 12, 20
    par, q, kn, vn, kc, vc = _case(rng, B, H, d, n, P)
    par[0] = np.arange(-1, n - 1)
    nn, pl = np.array([n], np.int32), np.array([P], np.int32)
    out = oracle.tree_attention_rows(q, kn, vn, kc, vc, pl, nn, par, oracle.all_rows(B, H, nn))
    k = np.concatenate([kc[0, 0, :P], kn[0, :, 0]]).astype(np.float64)
    v = np.concatenate([vc[0, 0, :P], vn[0, :, 0]]).astype(np.float64)
    qs = np.concatenate([np.zeros((P, d)), q[0, :, 0]]).astype(np.float64)
    np.testing.assert_allclose(out, _causal_attention(qs, k, v, 1 / np.sqrt(d))[P:], rtol=1e-12, atol=1e-12)


def test_single_node_is_one_query_decode():
    rng = np.random.default_rng(8)
    B, H, d, n, P = 1, 2, 64, 1, 50
    par, q, kn, vn, kc, vc = _case(rng, B, H, d, n, P)
    nn, pl = np.array([1], np.int32), np.array([P], np.int32)
    out = oracle.tree_attention_rows(q, kn, vn, kc, vc, pl, nn, par, oracle.all_rows(B, H, nn))
    for h in range(H):
        k = np.concatenate([kc[0, h, :P], kn[0, :, h]]).astype(np.float64)
        v = np.concatenate([vc[0, h, :P], vn[0, :, h]]).astype(np.float64)
        s = k @ q[0, 0, h].astype(np.float64) / 8.0
        w = np.exp(s - s.max())
        np.testing.assert_allclose(out[h], (w / w.sum()) @ v, rtol=1e-12, atol=1e-12)


def test_empty_prefix_root_sees_itself_only():
    rng = np.random.default_rng(9)
    B, H, d, n, P = 1, 1, 8, 4, 0
    par, q, kn, vn, kc, vc = _case(rng, B, H, d, n, P)
    nn, pl = np.array([n], np.int32), np.array([0], np.int32)
    out = oracle.tree_attention_rows(q, kn, vn, kc, vc, pl, nn, par, np.array([[0, 0, 0]], np.int32))
    np.testing.assert_allclose(out[0], vn[0, 0, 0].astype(np.float64), rtol=0, atol=0)


def test_bad_rows_rejected():
    rng = np.random.default_rng(1)
    par, q, kn, vn, kc, vc = _case(rng, 1, 1, 8, 3, 2)
    with pytest.raises(ValueError):
        oracle.tree_attention_rows(q, kn, vn, kc, vc, np.array([2]), np.array([3]), par,
                                   np.array([[0, 0, 3]], np.int32))
