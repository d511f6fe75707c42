"""The small-tree tcgen05 tree-attention kernel (trees of up to 32 nodes,
head_dim 128: keys on the MMA's M side, the key tiles of all (request, head)
pairs cut evenly over the CTAs) against the oracle through the C ABI; selected
with TREESPEC_ATTN_KERNEL=kt. TREESPEC_ATTN_CTAS
sets the CTA count and so moves the range boundaries that cut a pair into
partials merged by the last CTA to finish. Tolerance 2e-2 (bf16 inputs, fp32
accumulation)."""
import numpy as np
import pytest

from test_gpu_attention import TOL_BF16, _run_case

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _kt(monkeypatch):
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "kt")


def test_kt_is_selected_by_name(monkeypatch):
    from tree_speculative_verification_gb300 import api
    assert api.attention_kernel(8, 32, 21, 128, 2112, api.TS_BF16) == "k_attn_kt"
    assert api.attention_kernel(8, 32, 33, 128, 2112, api.TS_BF16) != "k_attn_kt"
    assert api.attention_kernel(8, 32, 21, 64, 2112, api.TS_BF16) != "k_attn_kt"
    monkeypatch.delenv("TREESPEC_ATTN_KERNEL")
    assert api.attention_kernel(8, 32, 21, 128, 2112, api.TS_BF16).startswith("k_attn_bf16<")


@pytest.mark.parametrize("n_max", [1, 2, 5, 8, 13, 21, 24, 31, 32])
def test_kt_node_counts(n_max):
    rng = np.random.default_rng(700 + n_max)
    err, _, _ = _run_case(rng, 2, 3, 128, n_max, prefix=[int(rng.integers(0, 400)), int(rng.integers(1, 400))])
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("ctas", ["1", "2", "3", "7", "19", "64"])
def test_kt_range_boundaries(ctas, monkeypatch):
    """Prefixes at and around tile edges, a tree straddling a tile edge (so a
    range may start on keys that some nodes cannot see), one-node trees."""
    monkeypatch.setenv("TREESPEC_ATTN_CTAS", ctas)
    rng = np.random.default_rng(800 + int(ctas))
    err, _, _ = _run_case(rng, 4, 3, 128, 32, prefix=[100, 0, 127, 1000], n_nodes=[32, 1, 21, 32])
    assert err <= TOL_BF16, err


def test_kt_many_pairs_ragged():
    """128 pairs with prefixes 0..3000 and trees of 1..32 nodes: most CTAs
    start or end inside a pair."""
    rng = np.random.default_rng(901)
    B, H = 8, 16
    prefix = rng.integers(0, 3000, B).tolist()
    n_nodes = rng.integers(1, 33, B).tolist()
    err, _, _ = _run_case(rng, B, H, 128, 32, prefix=prefix, n_nodes=n_nodes)
    assert err <= TOL_BF16, err


def test_kt_fewer_tiles_than_ctas():
    rng = np.random.default_rng(902)
    err, _, _ = _run_case(rng, 1, 1, 128, 3, prefix=[5])
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("ctas", ["3", "152"])
def test_kt_large_scores_rescale(ctas, monkeypatch):
    """Scores of magnitude ~100: the reference max moves inside a segment, so O
    and the row sums are rescaled in place."""
    monkeypatch.setenv("TREESPEC_ATTN_CTAS", ctas)
    rng = np.random.default_rng(903)
    err, _, _ = _run_case(rng, 1, 2, 128, 21, prefix=[2000], value_scale=3.0)
    assert err <= 5 * TOL_BF16, err


def test_kt_with_an_empty_request():
    """A request whose tree was rejected (0 nodes) has no tiles; the pairs of
    the requests around it are still exact and its rows are untouched."""
    import torch
    import oracle
    from tree_speculative_verification_gb300 import api
    from tree_speculative_verification_gb300.step import to_device
    from tree_speculative_verification_gb300.workloads import f32_to_bf16_bits
    rng = np.random.default_rng(904)
    B, H, d, n, P = 3, 8, 128, 21, 300
    par = np.full((B, n), -1, np.int32)
    for b in range(B):
        for v in range(1, n):
            par[b, v] = rng.integers(0, v)
    par[1, 5] = 9          # request 1: a cycle, so tree_build rejects it
    par[1, 9] = 5
    L_max = P + n + 16
    draw = lambda *s: rng.standard_normal(s).astype(np.float32)
    q, kn, vn = draw(B, n, H, d), draw(B, n, H, d), draw(B, n, H, d)
    kc, vc = np.zeros((B, H, L_max, d), np.float32), np.zeros((B, H, L_max, d), np.float32)
    kc[:, :, :P], vc[:, :, :P] = draw(B, H, P, d), draw(B, H, P, d)
    q, kn, vn, kc, vc = map(f32_to_bf16_bits, (q, kn, vn, kc, vc))
    t = api.Tree(B, n)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.tree_build(t, torch.zeros((B, n), dtype=torch.int32, device="cuda"), to_device(par, "cuda"),
                   to_device(np.full(B, n, np.int32), "cuda"), status=st)
    dv = lambda a: to_device(a, "cuda", True)
    dq, dkn, dvn, dkc, dvc = map(dv, (q, kn, vn, kc, vc))
    pl = to_device(np.full(B, P, np.int32), "cuda")
    api.kv_append(dkc, dvc, dkn, dvn, pl, t, st)
    out = torch.zeros_like(dq)
    api.tree_attention(out, dq, dkc, dvc, pl, t, 0.0, api.workspace(api.TS_OP_ATTENTION, B, H, n, d, L_max, 1), st)
    torch.cuda.synchronize()
    assert st.item() == api.STATUS_BAD_TREE and t.n_nodes.tolist() == [n, 0, n]
    o = out.float().cpu().numpy()
    assert not o[1].any()
    rows = np.array([(b, h, v) for b in (0, 2) for h in range(H) for v in range(n)], np.int32)
    par_ok = par.copy()
    par_ok[1] = np.arange(-1, n - 1)
    ref = oracle.tree_attention_rows(q, kn, vn, kc, vc, np.full(B, P), np.array([n, 1, n]), par_ok, rows)
    got = np.stack([o[b, v, h] for b, h, v in rows])
    assert float(np.abs(got - ref).max()) <= TOL_BF16
