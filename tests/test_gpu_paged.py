"""The paged KV cache (pages of 64 keys listed per request in a block table)
against the oracle and against the dense cache: the pages, gathered through
the block table into a dense host copy, feed the oracle's fp64 tree attention
(2e-2) and its kv_commit (bit-exact); and kv_append_paged,
tree_attention_paged and kv_commit_paged give bit-identical results to the
dense calls -- the same kernels on the same values, only the row addressing
differs -- for ragged prefixes, randomly permuted pages, every attention
kernel that pages and key splits; an out-of-table page id sets
TS_STATUS_INDEX."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import to_device
from tree_speculative_verification_gb300.workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu
PK = api.PAGE_KEYS


def _pages_from_dense(rng, kc, vc, L_need, spare=5):
    """Scatter a dense cache [B][H][L_max][d] into randomly placed pages;
    block-table entries past a request's need are -1."""
    B, H, L_max, d = kc.shape
    max_pages = (L_max + PK - 1) // PK
    need = [(int(L) + PK - 1) // PK for L in L_need]
    num_pages = sum(need) + spare
    ids = rng.permutation(num_pages)
    bt = np.full((B, max_pages), -1, np.int32)
    kp = np.zeros((num_pages, H, PK, d), kc.dtype)
    vp = np.zeros_like(kp)
    nxt = 0
    for b in range(B):
        for j in range(need[b]):
            g = int(ids[nxt]); nxt += 1
            bt[b, j] = g
            rows = slice(j * PK, min((j + 1) * PK, L_max))
            m = rows.stop - rows.start
            kp[g, :, :m] = kc[b, :, rows]
            vp[g, :, :m] = vc[b, :, rows]
    return kp, vp, bt


def _dense_from_pages(kp, bt, B, H, L_max, d):
    out = np.zeros((B, H, L_max, kp.shape[3]), kp.dtype)
    for b in range(B):
        for j in range(bt.shape[1]):
            g = bt[b, j]
            if g < 0:
                continue
            m = min(PK, L_max - j * PK)
            out[b, :, j * PK: j * PK + m] = kp[g, :, :m]
    return out


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _case(rng, B, H, n, prefix, d=128):
    par = np.full((B, n), -1, np.int32)
    for b in range(B):
        for v in range(1, n):
            par[b, v] = rng.integers(max(0, v - 5), v)
    prefix = np.asarray(prefix, np.int32)
    L_max = ((int(prefix.max()) + n + PK - 1) // PK) * PK + PK
    draw = lambda *s: f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    q, kn, vn = draw(B, n, H, d), draw(B, n, H, d), draw(B, n, H, d)
    kc, vc = np.zeros((B, H, L_max, d), np.uint16), np.zeros((B, H, L_max, d), np.uint16)
    for b in range(B):
        kc[b, :, :prefix[b]] = draw(H, int(prefix[b]), d)
        vc[b, :, :prefix[b]] = draw(H, int(prefix[b]), d)
    return par, prefix, L_max, q, kn, vn, kc, vc


def _random_paths(rng, par, B, n):
    op = np.full((B, n + 1), -1, np.int32)
    oc = np.zeros(B, np.int32)
    for b in range(B):
        u, path = 0, [0]
        while True:
            kids = np.nonzero(par[b] == u)[0]
            if len(kids) == 0 or rng.random() < 0.25:
                break
            u = int(rng.choice(kids))
            path.append(u)
        op[b, :len(path)] = path
        oc[b] = len(path)
    return op, oc


@pytest.mark.parametrize("mode,n", [("mma", 21), ("splits", 21), ("mma", 150), ("tq", 21), ("tq", 40), ("tq", 100)])
def test_paged_equals_dense(mode, n, monkeypatch):
    if mode == "tq":
        monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "tq")
    if mode in ("mma", "splits"):
        monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "mma")
    if mode == "splits":
        monkeypatch.setenv("TREESPEC_ATTN_SPLITS", "3")
    rng = np.random.default_rng(n + len(mode))
    B, H, d = 5, 4, 128
    par, prefix, L_max, q, kn, vn, kc, vc = _case(rng, B, H, n, [0, 63, 64, 700, 1000])
    kp, vp, bt = _pages_from_dense(rng, kc, vc, prefix + n)
    dv = lambda a: to_device(a, "cuda", True)
    t = api.Tree(B, n)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pl = to_device(prefix, "cuda")
    api.tree_build(t, torch.zeros((B, n), dtype=torch.int32, device="cuda"), to_device(par, "cuda"),
                   to_device(np.full(B, n, np.int32), "cuda"), prefix_len=pl, status=st)
    dkc, dvc, dq, dkn, dvn = dv(kc), dv(vc), dv(q), dv(kn), dv(vn)
    kv = api.PagedKV(dv(kp), dv(vp), to_device(bt, "cuda"))
    assert kv.L_max == L_max
    ws_d = api.workspace(api.TS_OP_ATTENTION, B, H, n, d, L_max, 1)
    ws_p = api.workspace(api.TS_OP_ATTENTION, B, H, n, d, L_max, 1)
    # append
    api.kv_append(dkc, dvc, dkn, dvn, pl, t, st)
    api.kv_append_paged(kv, dkn, dvn, pl, t, st)
    torch.cuda.synchronize()
    assert np.array_equal(_dense_from_pages(_bits(kv.k_pages), bt, B, H, L_max, d), _bits(dkc))
    assert np.array_equal(_dense_from_pages(_bits(kv.v_pages), bt, B, H, L_max, d), _bits(dvc))
    # attention: the same kernel on the same values
    out_d, out_p = torch.zeros_like(dq), torch.full_like(dq, float("nan"))
    api.tree_attention(out_d, dq, dkc, dvc, pl, t, 0.0, ws_d, st)
    api.tree_attention_paged(out_p, dq, kv, pl, t, 0.0, ws_p, st)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out_p), _bits(out_d))
    # the oracle on the cache gathered through the block table
    nn = np.full(B, n, np.int32)
    gk = _dense_from_pages(_bits(kv.k_pages), bt, B, H, L_max, d)
    gv = _dense_from_pages(_bits(kv.v_pages), bt, B, H, L_max, d)
    rows = oracle.all_rows(B, H, nn)
    ref = oracle.tree_attention_rows(q, kn, vn, gk, gv, prefix, nn, par, rows)
    o = out_p.float().cpu().numpy()
    err = float(np.max(np.abs(o[rows[:, 0], rows[:, 2], rows[:, 1]] - ref)))
    assert err <= 2e-2, err
    # commit of a random accepted path per request
    op, oc = _random_paths(rng, par, B, n)
    dop, doc = to_device(op, "cuda"), to_device(oc, "cuda")
    npl_d = torch.zeros(B, dtype=torch.int32, device="cuda")
    npl_p = torch.zeros(B, dtype=torch.int32, device="cuda")
    api.kv_commit(dkc, dvc, pl, npl_d, dop, doc, t, st)
    api.kv_commit_paged(kv, pl, npl_p, dop, doc, t, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert npl_p.tolist() == npl_d.tolist() == (prefix + oc).tolist()
    # the oracle's commit of the gathered cache, with the oracle's own DFS order
    ref_t = oracle.tree_build(par, np.zeros((B, n), np.int32), nn)
    rk, rv, rnpl = oracle.kv_commit(gk, gv, prefix, ref_t["dfs_of"], op, oc)
    assert rnpl.tolist() == npl_p.tolist()
    assert np.array_equal(_dense_from_pages(_bits(kv.k_pages), bt, B, H, L_max, d), rk)
    assert np.array_equal(_dense_from_pages(_bits(kv.v_pages), bt, B, H, L_max, d), rv)
    assert np.array_equal(_dense_from_pages(_bits(kv.k_pages), bt, B, H, L_max, d), _bits(dkc))
    assert np.array_equal(_dense_from_pages(_bits(kv.v_pages), bt, B, H, L_max, d), _bits(dvc))


def test_paged_bad_page_id_sets_index():
    rng = np.random.default_rng(3)
    B, H, n, d = 2, 2, 9, 128
    par, prefix, L_max, q, kn, vn, kc, vc = _case(rng, B, H, n, [100, 200])
    kp, vp, bt = _pages_from_dense(rng, kc, vc, prefix + n)
    bt[1, 1] = kp.shape[0] + 7                         # past the page pool
    dv = lambda a: to_device(a, "cuda", True)
    t = api.Tree(B, n)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pl = to_device(prefix, "cuda")
    api.tree_build(t, torch.zeros((B, n), dtype=torch.int32, device="cuda"), to_device(par, "cuda"),
                   to_device(np.full(B, n, np.int32), "cuda"), prefix_len=pl)
    kv = api.PagedKV(dv(kp), dv(vp), to_device(bt, "cuda"))
    out = torch.zeros((B, n, H, d), dtype=torch.bfloat16, device="cuda")
    api.tree_attention_paged(out, dv(q), kv, pl, t, 0.0, api.workspace(api.TS_OP_ATTENTION, B, H, n, d, L_max, 1),
                             st)
    torch.cuda.synchronize()
    assert st.item() & api.STATUS_INDEX


def test_paged_step_equals_dense_step():
    """The merge workload's whole step (chain merge, append, attention, MSS,
    commit) on a paged cache: attention output, accepted tokens and the
    committed rows equal the dense step's bit for bit."""
    from tree_speculative_verification_gb300.step import DeviceStep
    from _helpers import workload
    w = workload("merge")
    dense, paged = DeviceStep(w), DeviceStep(w, paged=True, seed=7)
    dense.run("mss")
    paged.run("mss")
    torch.cuda.synchronize()
    assert dense.status.item() & ~api.STATUS_ZERO_RESID == 0 and paged.status.item() == dense.status.item()
    assert np.array_equal(_bits(paged.out), _bits(dense.out))
    assert torch.equal(paged.mss_tokens, dense.mss_tokens) and torch.equal(paged.mss_count, dense.mss_count)
    assert torch.equal(paged.new_prefix_len, dense.new_prefix_len)
    bt = paged.kv.block_table.cpu().numpy()
    got_k = _dense_from_pages(_bits(paged.kv.k_pages), bt, w.B, w.H, w.L_max, w.d)
    got_v = _dense_from_pages(_bits(paged.kv.v_pages), bt, w.B, w.H, w.L_max, w.d)
    npl = dense.new_prefix_len.cpu().numpy()
    ref_k, ref_v = _bits(dense.k_cache), _bits(dense.v_cache)
    for b in range(w.B):     # every row up to the new prefix length
        assert np.array_equal(got_k[b, :, :npl[b]], ref_k[b, :, :npl[b]]), b
        assert np.array_equal(got_v[b, :, :npl[b]], ref_v[b, :, :npl[b]]), b
