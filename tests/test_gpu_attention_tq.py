"""The persistent 128-key-tile tcgen05 tree-attention kernel (trees of up to 128
nodes, head_dim 128; Q and P in tensor memory) against the oracle, through the
same C ABI call; selected with TREESPEC_ATTN_KERNEL=tq. Tolerance 2e-2 (bf16
inputs, fp32 accumulation). Prefixes straddle the 64- and 128-key tile edges,
and NaN rows past every request's keys must not leak."""
import numpy as np
import pytest
import torch

from test_gpu_attention import TOL_BF16, _run_case
from _helpers import attention_error, oracle_tree, sample_rows, workload
from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tq(monkeypatch):
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "tq")


@pytest.mark.parametrize("n_max", [1, 5, 21, 32, 33, 47, 64, 65, 100, 128])
def test_tq_node_counts(n_max):
    rng = np.random.default_rng(700 + n_max)
    err, _, _ = _run_case(rng, 2, 3, 128, n_max, prefix=[int(rng.integers(1, 400)), int(rng.integers(1, 400))])
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("prefix", [[0, 63, 64, 65], [127, 128, 129, 191], [192, 255, 256, 1000]])
def test_tq_tile_edges(prefix):
    """Key counts P + n on both sides of 64- and 128-key boundaries (a tile with
    an empty second half, a tile with one key)."""
    rng = np.random.default_rng(sum(prefix))
    err, _, _ = _run_case(rng, 4, 2, 128, 40, prefix=prefix, n_nodes=[40, 1, 33, 7])
    assert err <= TOL_BF16, err


def test_tq_large_scores_rescale():
    rng = np.random.default_rng(19)
    err, _, _ = _run_case(rng, 1, 2, 128, 100, prefix=[1500], value_scale=3.0)
    assert err <= 5 * TOL_BF16, err


def test_tq_many_items_ragged():
    """Several items per CTA (3 x 64 pairs on the SMs), ragged prefixes and node
    counts 1..47, items of one tile next to long ones."""
    rng = np.random.default_rng(88)
    err, _, _ = _run_case(rng, 3, 64, 128, 47, prefix=[100, 0, 700], n_nodes=[21, 47, 1])
    assert err <= TOL_BF16, err


def test_tq_request_without_tree():
    """A request with no nodes gives items with no tiles, skipped by every role
    of the persistent CTAs; the other requests stay exact."""
    rng = np.random.default_rng(89)
    err, _, _ = _run_case(rng, 3, 64, 128, 30, prefix=[200, 300, 50], n_nodes=[30, 0, 12])
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("name", ["long65b", "opt30b"])
def test_tq_full_size_sampled(name):
    w = workload(name)
    assert api.attention_kernel(w.B, w.H, w.n_max, w.d, w.L_max, api.TS_BF16) == "k_attn_tq"
    s = DeviceStep(w)
    s.build(); s.append(); s.attend()
    torch.cuda.synchronize()
    assert s.status.item() == 0
    parent, tokens, n_nodes, _, _ = oracle_tree(w)
    rows = sample_rows(w, n_nodes, 48, seed=len(name) + 1)
    err, _, _ = attention_error(s, w, n_nodes, parent, rows)
    assert err <= TOL_BF16, err
    out = s.out.float()
    for b in range(w.B):
        assert torch.isfinite(out[b, : int(n_nodes[b])]).all()
