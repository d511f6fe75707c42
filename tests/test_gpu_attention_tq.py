"""The persistent 128-key-tile tcgen05 tree-attention kernel (trees of up to 128
nodes, head_dim 128; Q and P in tensor memory) against the oracle, through the
same C ABI call; selected with TREESPEC_ATTN_KERNEL=tq. Tolerance 2e-2 (bf16
inputs, fp32 accumulation). Prefixes straddle the 64- and 128-key tile edges,
and NaN rows past every request's keys must not leak."""
import numpy as np
import pytest
import torch

from test_gpu_attention import TOL_BF16, _run_case, full_size_every_row
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


@pytest.mark.parametrize("n_max,prefix", [(5, 3), (30, 20)])
def test_tq_cache_shorter_than_a_tile(n_max, prefix):
    """One request and one head whose whole cache (at most 119 rows) is shorter
    than one 128-key tile: the tile is loaded past the end of the cache."""
    rng = np.random.default_rng(31 + n_max)
    err, _, _ = _run_case(rng, 1, 1, 128, n_max, prefix=[prefix])
    assert err <= TOL_BF16, err


def test_tq_large_scores_rescale():
    rng = np.random.default_rng(19)
    err, _, _ = _run_case(rng, 1, 2, 128, 100, prefix=[1500], value_scale=3.0)
    print(f"value scale 3: max-abs error {err:.4f}")
    assert err <= 3.0 * TOL_BF16, err    # the bound scales with the magnitude of V


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


@pytest.mark.parametrize("name", ["llama7b", "merge"])
def test_tq_full_size_every_row_small_trees(name):
    """The persistent kernel forced onto the 21-node and merged-chain layers:
    256 and 512 items on 152 CTAs (most CTAs take several items from the
    queue), ragged prefixes U[512, 4096]; every output row checked."""
    full_size_every_row(name, "k_attn_tq")
