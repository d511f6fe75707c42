"""tree_attention_append: kv_append and tree_attention in one call. With the
persistent tcgen05 kernel it is one launch whose tenth warp writes the new
rows into the cache while the attention runs; it must leave the same cache as
kv_append, bit for bit, and produce the same output as tree_attention on that
cache, bit for bit (the same kernel arithmetic on the same keys). Small cases
(prefixes on both sides of the tile edges, trees of up to 64 nodes and of
65-128, requests without nodes, NaN rows past every request's keys), then the
full-size workloads, and the oracle on one small case."""
import numpy as np
import pytest
import torch

import oracle
from test_gpu_attention import TOL_BF16
from tree_speculative_verification_gb300 import api, workloads
from tree_speculative_verification_gb300.step import DeviceStep, to_device
from tree_speculative_verification_gb300.workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def _inputs(rng, B, H, n_max, prefix, n_nodes):
    d = 128
    par = np.full((B, n_max), -1, np.int32)
    for b in range(B):
        for v in range(1, n_nodes[b]):
            par[b, v] = rng.integers(max(0, v - 6), v)
    L_max = int(max(prefix)) + n_max + int(rng.integers(0, 70))
    draw = lambda *s: rng.standard_normal(s).astype(np.float32)
    q, kn, vn = draw(B, n_max, H, d), draw(B, n_max, H, d), draw(B, n_max, H, d)
    kc = np.full((B, H, L_max, d), np.nan, np.float32)
    vc = np.full((B, H, L_max, d), np.nan, np.float32)
    for b in range(B):
        kc[b, :, :prefix[b]] = draw(H, int(prefix[b]), d)
        vc[b, :, :prefix[b]] = draw(H, int(prefix[b]), d)
    return par, L_max, [f32_to_bf16_bits(a) for a in (q, kn, vn, kc, vc)]


def _both(B, H, n_max, prefix, n_nodes, seed):
    rng = np.random.default_rng(seed)
    n_nodes = np.asarray(n_nodes, np.int32)
    par, L_max, host = _inputs(rng, B, H, n_max, prefix, n_nodes)
    t = api.Tree(B, n_max)
    api.tree_build(t, to_device(np.zeros((B, n_max), np.int32), "cuda"), to_device(par, "cuda"),
                   to_device(n_nodes, "cuda"))
    dq, dkn, dvn, kc, vc = [to_device(a, "cuda", True) for a in host]
    pl = to_device(np.asarray(prefix, np.int32), "cuda")
    ws = api.workspace(api.TS_OP_ATTENTION, B, H, n_max, 128, L_max, 1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc1, vc1 = kc.clone(), vc.clone()
    api.kv_append(kc1, vc1, dkn, dvn, pl, t, st)
    out1 = torch.zeros_like(dq)
    api.tree_attention(out1, dq, kc1, vc1, pl, t, 0.0, ws, st)
    kc2, vc2 = kc.clone(), vc.clone()
    out2 = torch.zeros_like(dq)
    api.tree_attention_append(out2, dq, kc2, vc2, dkn, dvn, pl, t, 0.0, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return (out1, kc1, vc1), (out2, kc2, vc2), (par, host, n_nodes, prefix)


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("n_max,prefix,n_nodes", [
    (47, [1024, 0, 63, 65], [47, 21, 1, 47]),
    (64, [127, 128, 129, 700], [64, 64, 30, 0]),
    (21, [2048, 2047, 5, 300], [21, 21, 21, 21]),
    (100, [191, 192, 1000, 33], [100, 65, 99, 1]),
    (128, [16, 500], [128, 128]),
])
def test_fused_equals_separate_calls(n_max, prefix, n_nodes, monkeypatch):
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "tq")
    B, H = len(prefix), 6
    assert api.attention_kernel(B, H, n_max, 128, max(prefix) + n_max, api.TS_BF16).startswith("k_attn_tq")
    (o1, k1, v1), (o2, k2, v2), _ = _both(B, H, n_max, prefix, n_nodes, seed=n_max + sum(prefix))
    # the caches hold NaN past every request's rows: compare bit patterns
    assert _same(k1, k2) and _same(v1, v2)
    assert _same(o1, o2)


def test_fused_against_oracle():
    B, H, n_max = 3, 4, 40
    prefix, n_nodes = [300, 0, 129], [40, 17, 33]
    (_, _, _), (o2, k2, v2), (par, host, n_nodes, prefix) = _both(B, H, n_max, prefix, n_nodes, seed=5)
    q, kn, vn, kc, vc = host
    rows = oracle.all_rows(B, H, n_nodes)
    ref = oracle.tree_attention_rows(q, kn, vn, kc, vc, np.asarray(prefix), n_nodes, par, rows)
    o = o2.float().cpu().numpy()
    got = np.stack([o[b, v, h] for b, h, v in rows])
    assert float(np.max(np.abs(got - ref))) <= TOL_BF16


def test_fused_mma_path_is_two_launches_with_the_same_results(monkeypatch):
    """With the mma.sync kernel the call is kv_append then tree_attention."""
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "mma")
    (o1, k1, v1), (o2, k2, v2), _ = _both(2, 3, 21, [200, 64], [21, 9], seed=77)
    assert _same(k1, k2) and _same(v1, v2) and _same(o1, o2)


@pytest.mark.parametrize("name", ["opt30b", "merge", "long65b"])
def test_fused_full_size(name):
    w = workloads.make(name)
    s = DeviceStep(w)
    s.build()
    k0, v0 = s.k_cache.clone(), s.v_cache.clone()
    s.append()
    s.attend()
    torch.cuda.synchronize()
    out1, k1, v1 = s.out.clone(), s.k_cache.clone(), s.v_cache.clone()
    s.k_cache.copy_(k0)
    s.v_cache.copy_(v0)
    s.out.zero_()
    del k0, v0
    s.attend_append()
    torch.cuda.synchronize()
    assert s.status.item() == 0
    assert _same(s.k_cache, k1) and _same(s.v_cache, v1)
    assert _same(s.out, out1)


@pytest.mark.parametrize("d,bf16", [(64, True), (64, False), (128, False)])
def test_two_launch_forms(d, bf16):
    """head_dim 64 (the mma.sync kernel) and fp32: the call is kv_append then the
    attention, with the same results as the two calls."""
    rng = np.random.default_rng(d + 7 * bf16)
    B, H, n_max = 2, 3, 11
    prefix, n_nodes = [70, 5], np.array([11, 6], np.int32)
    par = np.full((B, n_max), -1, np.int32)
    for b in range(B):
        for v in range(1, n_nodes[b]):
            par[b, v] = rng.integers(0, v)
    L_max = max(prefix) + n_max + 3
    draw = lambda *s: rng.standard_normal(s).astype(np.float32)
    host = [draw(B, n_max, H, d), draw(B, n_max, H, d), draw(B, n_max, H, d), draw(B, H, L_max, d),
            draw(B, H, L_max, d)]
    if bf16:
        host = [f32_to_bf16_bits(a) for a in host]
    t = api.Tree(B, n_max)
    api.tree_build(t, to_device(np.zeros((B, n_max), np.int32), "cuda"), to_device(par, "cuda"),
                   to_device(n_nodes, "cuda"))
    dq, dkn, dvn, kc, vc = [to_device(a, "cuda", bf16) for a in host]
    pl = to_device(np.asarray(prefix, np.int32), "cuda")
    ws = api.workspace(api.TS_OP_ATTENTION, B, H, n_max, d, L_max, 1) if bf16 else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc1, vc1, out1 = kc.clone(), vc.clone(), torch.zeros_like(dq)
    api.kv_append(kc1, vc1, dkn, dvn, pl, t, st)
    api.tree_attention(out1, dq, kc1, vc1, pl, t, 0.0, ws, st)
    kc2, vc2, out2 = kc.clone(), vc.clone(), torch.zeros_like(dq)
    api.tree_attention_append(out2, dq, kc2, vc2, dkn, dvn, pl, t, 0.0, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    eq = (lambda a, b: torch.equal(a.view(torch.int16), b.view(torch.int16))) if bf16 else torch.equal
    assert eq(kc1, kc2) and eq(vc1, vc2) and eq(out1, out2)
