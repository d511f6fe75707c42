"""Pins of the oracle's token-tree layout against what the pages fix.

SpecInfer (arXiv 2305.09781): Fig. 3 expansion <2,2,1> (4 sequences), Def. 3.2
merge of the four Fig. 3 sequences, sec. 4.2 depth-first layout; the 6-node
tree-mask table of "How Speculative Decoding in LLM Serving Actually Works".
"""
import os

import networkx as nx
import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    out, key = {}, None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if ":" in line:
            key, _, rest = line.partition(":")
            out[key] = [rest.split()] if rest.strip() else []
        else:
            out[key].append(line.split())
    return out


def _ints(rows):
    return np.array([[int(x) for x in r] for r in rows])


def _leaves(parent):
    n = len(parent)
    has_child = np.zeros(n, bool)
    for v in range(n):
        if parent[v] >= 0:
            has_child[parent[v]] = True
    return int((~has_child).sum())


def test_expansion_221_fixture():
    fx = _read_fixture("expansion_221.txt")
    widths = _ints(fx["widths"])[0]
    par = oracle.widths_parent(widths)
    assert len(par) == int(fx["n_nodes"][0][0])
    assert _leaves(par) == int(fx["n_leaves"][0][0])
    t = oracle.tree_build(par)
    assert t["status"] == 0
    counts = np.bincount(t["depth"][: len(par)])
    assert counts.tolist() == _ints(fx["depth_counts"])[0].tolist()


@pytest.mark.parametrize("widths,n,leaves", [((1, 1, 3, 1, 1, 1, 1, 1), 21, 3), ((2, 2, 2, 2, 1), 47, 16),
                                             ((3,), 4, 3), ((1,) * 12, 13, 1)])
def test_expansion_counts(widths, n, leaves):
    # sum over levels of prod k_i nodes plus the root; prod k_i leaf sequences
    par = oracle.widths_parent(widths)
    assert len(par) == n == 1 + sum(int(np.prod(widths[: i + 1])) for i in range(len(widths)))
    assert _leaves(par) == leaves == int(np.prod(widths))


def test_merge_fig3_fixture():
    fx = _read_fixture("merge_fig3.txt")
    chains = _ints(fx["chains"])
    par, tok, src = oracle.merge_chains(chains, int(fx["root"][0][0]))
    assert len(par) == int(fx["n_nodes"][0][0])
    assert _leaves(par) == int(fx["n_leaves"][0][0])
    t = oracle.tree_build(par, tok)
    assert t["token"].tolist() == _ints(fx["dfs_tokens"])[0].tolist()
    system_nodes = [v for v in range(len(par)) if tok[v] == 4]
    assert len(system_nodes) == 2 and par[system_nodes[0]] != par[system_nodes[1]]
    # the merged tree has the shape of the <2,2,1> expansion tree of Fig. 3
    t221 = oracle.tree_build(oracle.widths_parent([2, 2, 1]))
    assert t["parent"].tolist() == t221["parent"].tolist()
    # every node was created by the lowest chain holding its sequence
    for v in range(1, len(par)):
        c, p = divmod(int(src[v]), chains.shape[1])
        assert chains[c, p] == tok[v]
        for c2 in range(c):
            assert not np.array_equal(chains[c2, : p + 1], chains[c, : p + 1])


def test_mask_6node_fixture():
    fx = _read_fixture("mask_6node.txt")
    par = _ints(fx["parent"])[0]
    mask = _ints(fx["mask"])
    t = oracle.tree_build(par)
    d = t["dfs_of"]
    n = len(par)
    got = np.array([[t["anc"][d[v], d[w]] for w in range(n)] for v in range(n)])
    assert got.tolist() == mask.tolist()


def _random_parent(rng, n, shuffle=True):
    par = np.full(n, -1, np.int32)
    for v in range(1, n):
        par[v] = rng.integers(0, v)
    if shuffle:
        # relabel so that a parent's id can exceed its child's
        perm = rng.permutation(n)
        inv = np.argsort(perm)
        par = np.array([-1 if par[perm[i]] < 0 else inv[par[perm[i]]] for i in range(n)], np.int32)
    return par


@pytest.mark.parametrize("seed", range(12))
def test_layout_against_networkx(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 90))
    par = _random_parent(rng, n)
    tok = rng.integers(0, 1000, n).astype(np.int32)
    t = oracle.tree_build(par, tok)
    assert t["status"] == 0
    root = int(np.nonzero(par == -1)[0][0])
    g = nx.DiGraph()
    g.add_nodes_from(range(n))
    for v in range(n):          # children inserted in increasing id order
        if par[v] >= 0:
            g.add_edge(int(par[v]), v)
    order = list(nx.dfs_preorder_nodes(g, source=root))
    assert t["perm"][:n].tolist() == order
    depth = nx.single_source_shortest_path_length(g, root)
    for i, v in enumerate(order):
        assert t["depth"][i] == depth[v]
        assert t["token"][i] == tok[v]
        desc = nx.descendants(g, v) | {v}
        assert set(order[i: t["sub_end"][i]]) == desc
        anc = nx.ancestors(g, v) | {v}
        for j, w in enumerate(order):
            assert t["anc"][i, j] == (w in anc)
            assert t["anc"][i, j] == (j <= i < t["sub_end"][j])
        if i > 0:
            assert t["parent"][i] == order.index(int(par[v])) < i


@pytest.mark.parametrize("par", [[-1, 2, 1], [-1, -1, 0], [0, 0, 1], [-1, 5, 0], [-1, 1]])
def test_bad_trees_rejected(par):
    t = oracle.tree_build(np.array(par, np.int32))
    assert t["status"] == oracle.OR_BAD_TREE
