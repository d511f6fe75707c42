"""GPU parity of the tree layout (tree_build), kv_append and kv_commit against
the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import DeviceStep, to_device

from _helpers import compare_trees, device_tree, oracle_tree, workload

pytestmark = pytest.mark.gpu


def _random_parents(rng, B, n_max, shuffle=True):
    par = np.full((B, n_max), -1, np.int32)
    n_nodes = rng.integers(1, n_max + 1, B).astype(np.int32)
    for b in range(B):
        n = int(n_nodes[b])
        p = np.full(n, -1, np.int32)
        for v in range(1, n):
            p[v] = rng.integers(0, v)
        if shuffle:
            perm = rng.permutation(n)
            inv = np.argsort(perm)
            p = np.array([-1 if p[perm[i]] < 0 else inv[p[perm[i]]] for i in range(n)], np.int32)
        par[b, :n] = p
    return par, n_nodes


@pytest.mark.parametrize("n_max,seed", [(1, 0), (7, 1), (33, 2), (100, 3), (256, 4)])
def test_tree_build_parent_mode(n_max, seed):
    rng = np.random.default_rng(seed)
    B = 9
    par, n_nodes = _random_parents(rng, B, n_max)
    tok = rng.integers(0, 50000, (B, n_max)).astype(np.int32)
    P = rng.integers(0, 5000, B).astype(np.int32)
    t = api.Tree(B, n_max)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.tree_build(t, to_device(tok, "cuda"), to_device(par, "cuda"), to_device(n_nodes, "cuda"),
                   prefix_len=to_device(P, "cuda"), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.tree_build(par, tok, n_nodes)
    compare_trees(device_tree(type("S", (), {"tree": t})), ref, n_nodes, P)


@pytest.mark.parametrize("widths", [(2, 2, 1), (1, 1, 3, 1, 1, 1, 1, 1), (2, 2, 2, 2, 1), (4, 4, 4), (1,) * 12])
def test_tree_build_widths_mode(widths):
    par = oracle.widths_parent(widths)
    n = len(par)
    B = 3
    rng = np.random.default_rng(n)
    tok = rng.integers(0, 32000, (B, n)).astype(np.int32)
    t = api.Tree(B, n)
    api.tree_build(t, to_device(tok, "cuda"), widths=widths)
    torch.cuda.synchronize()
    ref = oracle.tree_build(np.tile(par, (B, 1)), tok)
    compare_trees(device_tree(type("S", (), {"tree": t})), ref, [n] * B)


def test_tree_build_chains_fig3_and_merge_workload():
    # the Fig. 3 sequences (SpecInfer Def. 3.2)
    chains = np.array([[[1, 2, 3], [1, 4, 5], [6, 7, 8], [6, 4, 5]]], np.int32)
    t = api.Tree(1, 13)
    tok_out = torch.full((1, 13), -1, dtype=torch.int32, device="cuda")
    pr = torch.full((1, 13), -1, dtype=torch.int32, device="cuda")
    qr = torch.full((1, 13), -1, dtype=torch.int32, device="cuda")
    api.tree_build_chains(t, to_device(np.array([0], np.int32), "cuda"), to_device(chains, "cuda"), tok_out, pr, qr)
    torch.cuda.synchronize()
    par, tok, src = oracle.merge_chains(chains[0], 0)
    assert t.n_nodes.item() == len(par) == 11
    assert tok_out[0, :11].tolist() == tok.tolist()
    assert pr[0, :11].tolist() == (src + 1).tolist()
    assert qr[0, :11].tolist() == src.tolist()
    ref = oracle.tree_build(par[None], tok[None])
    compare_trees(device_tree(type("S", (), {"tree": t})), ref, [11])
    # the merge workload's 16 requests
    w = workload("merge", attention=False)
    s = DeviceStep(w, attention=False)
    s.build()
    torch.cuda.synchronize()
    parent, tokens, n_nodes, p_row, q_row = oracle_tree(w)
    ref = oracle.tree_build(parent, tokens, n_nodes)
    compare_trees(device_tree(s), ref, n_nodes, w.prefix_len)
    for b in range(w.B):
        n = n_nodes[b]
        assert s.p_row[b, :n].tolist() == p_row[b, :n].tolist()
        assert s.q_row[b, 1:n].tolist() == q_row[b, 1:n].tolist()
        assert s.tokens[b, :n].tolist() == tokens[b, :n].tolist()


@pytest.mark.parametrize("par", [[-1, 2, 1], [-1, -1, 0], [0, 0, 1], [-1, 5, 0]])
def test_tree_build_rejects_bad_trees(par):
    B, n = 2, len(par)
    parent = np.array([par, [-1] + [0] * (n - 1)], np.int32)
    t = api.Tree(B, n)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.tree_build(t, torch.zeros((B, n), dtype=torch.int32, device="cuda"), to_device(parent, "cuda"),
                   to_device(np.array([n, n], np.int32), "cuda"), status=st)
    torch.cuda.synchronize()
    assert st.item() & api.STATUS_BAD_TREE
    assert t.n_nodes.tolist() == [0, n]          # only the bad request is emptied
    assert (t.perm[0] == -1).all()


@pytest.mark.parametrize("name,dtype_scale", [("tiny", 1), ("llama7b", 4), ("merge", 4), ("opt30b", 16)])
def test_kv_append_and_commit(name, dtype_scale):
    w = workload(name, dtype_scale)
    s = DeviceStep(w)
    s.build()
    s.append()
    s.verify("mss" if w.verify == "mss" else "greedy")
    kind = "mss" if w.verify == "mss" else "greedy"
    torch.cuda.synchronize()
    parent, tokens, n_nodes, p_row, q_row = oracle_tree(w)
    ref = oracle.tree_build(parent, tokens, n_nodes)
    view = (lambda x: x.view(torch.int16).cpu().numpy().view(np.uint16)) if w.dtype == "bf16" else (
        lambda x: x.cpu().numpy())
    kc, vc = view(s.k_cache), view(s.v_cache)
    # appended: cache row P + dfs(v) holds node v's K/V, the prefix is untouched
    for b in range(w.B):
        P, n = int(w.prefix_len[b]), int(n_nodes[b])
        for v in range(n):
            i = ref["dfs_of"][b, v]
            assert np.array_equal(kc[b, :, P + i], w.k_new[b, v]), (b, v)
            assert np.array_equal(vc[b, :, P + i], w.v_new[b, v]), (b, v)
        assert np.array_equal(kc[b, :, :P], w.k_cache[b, :, :P])
    path = (s.mss_path if kind == "mss" else s.out_path).cpu().numpy()
    count = (s.mss_count if kind == "mss" else s.out_count).cpu().numpy()
    k_ref, v_ref, npl_ref = oracle.kv_commit(kc, vc, w.prefix_len, ref["dfs_of"], path, count)
    s.commit(kind)
    torch.cuda.synchronize()
    assert s.new_prefix_len.cpu().numpy().tolist() == npl_ref.tolist()
    assert np.array_equal(view(s.k_cache), k_ref)
    assert np.array_equal(view(s.v_cache), v_ref)
    assert s.status.item() == 0
