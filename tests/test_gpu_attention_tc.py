"""The tcgen05 tree-attention kernel (trees of up to 128 nodes, head_dim 128)
against the oracle, through the same C ABI call; selected with
TREESPEC_ATTN_KERNEL=tc. Tolerance 2e-2 (bf16 inputs, fp32 accumulation)."""
import numpy as np
import pytest

from test_gpu_attention import TOL_BF16, _run_case

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tc(monkeypatch):
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "tc")


@pytest.mark.parametrize("n_max", [1, 5, 21, 32, 47, 64, 100, 128])
def test_tc_node_counts(n_max):
    rng = np.random.default_rng(500 + n_max)
    err, _, _ = _run_case(rng, 2, 3, 128, n_max, prefix=[int(rng.integers(1, 400)), int(rng.integers(1, 400))])
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("splits", ["1", "3", "64"])
def test_tc_splits_ragged(splits, monkeypatch):
    monkeypatch.setenv("TREESPEC_ATTN_SPLITS", splits)
    rng = np.random.default_rng(600 + int(splits))
    err, _, _ = _run_case(rng, 4, 2, 128, 21, prefix=[0, 63, 64, 1000], n_nodes=[21, 1, 13, 21])
    assert err <= TOL_BF16, err


def test_tc_large_scores_rescale():
    rng = np.random.default_rng(9)
    err, _, _ = _run_case(rng, 1, 2, 128, 40, prefix=[900], value_scale=3.0)
    assert err <= 5 * TOL_BF16, err


def test_tp_persistent_many_items(monkeypatch):
    """More (request, head) pairs than SMs: the persistent kernel walks several
    items per CTA, with ragged prefixes and node counts (1..47) and items of one
    key tile next to long ones."""
    monkeypatch.setenv("TREESPEC_ATTN_PERSISTENT", "1")
    rng = np.random.default_rng(77)
    err, _, _ = _run_case(rng, 3, 64, 128, 47, prefix=[100, 0, 700], n_nodes=[21, 47, 1])
    assert err <= TOL_BF16, err


def test_tp_persistent_with_an_empty_request(monkeypatch):
    """A request whose tree was rejected (0 nodes) gives items with no tiles; the
    other requests' items around it are still exact."""
    monkeypatch.setenv("TREESPEC_ATTN_PERSISTENT", "1")
    import torch
    import oracle
    from tree_speculative_verification_gb300 import api
    from tree_speculative_verification_gb300.step import to_device
    from tree_speculative_verification_gb300.workloads import f32_to_bf16_bits
    rng = np.random.default_rng(78)
    B, H, d, n, P = 3, 64, 128, 30, 200
    par = np.full((B, n), -1, np.int32)
    for b in range(B):
        for v in range(1, n):
            par[b, v] = rng.integers(0, v)
    par[1, 5] = 9          # request 1: node 5 under node 9 is fine, add a cycle below
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
    assert not o[1].any()                         # the rejected request's rows are untouched
    nn = np.array([n, 0, n], np.int32)
    rows = np.array([(b, h, v) for b in (0, 2) for h in range(H) for v in range(n)], np.int32)
    par_ok = par.copy()
    par_ok[1] = np.arange(-1, n - 1)              # any valid tree for the oracle's checks
    ref = oracle.tree_attention_rows(q, kn, vn, kc, vc, np.full(B, P), np.array([n, 1, n]), par_ok, rows)
    got = np.stack([o[b, v, h] for b, h, v in rows])
    assert float(np.abs(got - ref).max()) <= TOL_BF16
