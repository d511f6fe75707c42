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
