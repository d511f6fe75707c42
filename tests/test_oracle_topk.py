"""Pins of the oracle's top-k expansion (SpecInfer sec. 3, Fig. 3: the SSM
expands every node of depth i-1 into its k_i most likely next tokens):
numpy's stable sort as the definition of "k largest, ties to the lower id",
a hand-made tie fixture, and the tokens the synthetic expansion workloads
draft with their own (independent) numpy code."""
import numpy as np
import pytest

import oracle
from tree_speculative_verification_gb300 import workloads as wl


def _expected(widths, root, ssm):
    par = oracle.widths_parent(widths)
    n = len(par)
    B = ssm.shape[0]
    tok = np.full((B, n), -1, np.int32)
    tok[:, 0] = root
    for b in range(B):
        for u in range(n):
            kids = np.nonzero(par == u)[0]
            if len(kids):
                tok[b, kids] = np.argsort(-ssm[b, u].astype(np.float64), kind="stable")[: len(kids)]
    return tok


@pytest.mark.parametrize("widths", [(2,), (3, 2), (2, 2, 2, 2, 1), (1, 1, 3, 1)])
def test_topk_matches_stable_sort(widths):
    rng = np.random.default_rng(len(widths))
    n_internal = int(np.max(oracle.widths_parent(widths))) + 1
    B, V = 5, 300
    z = rng.standard_normal((B, n_internal, V))
    ssm = (np.exp(z) / np.exp(z).sum(-1, keepdims=True)).astype(np.float32)
    root = rng.integers(0, V, B).astype(np.int32)
    tok, st = oracle.topk_expand(widths, root, ssm)
    assert st == 0
    assert np.array_equal(tok, _expected(widths, root, ssm))


def test_topk_ties_go_to_the_lower_id():
    ssm = np.array([[[0.1, 0.3, 0.2, 0.3, 0.1]]], np.float32)   # tokens 1 and 3 tie, then 2
    tok, _ = oracle.topk_expand((3,), np.array([4], np.int32), ssm)
    assert tok[0].tolist() == [4, 1, 3, 2]


def test_topk_nonfinite_row():
    ssm = np.full((2, 1, 6), 1 / 6, np.float32)
    ssm[1, 0, 2] = np.nan
    tok, st = oracle.topk_expand((2,), np.array([0, 0], np.int32), ssm)
    assert st & 4 and tok[1, 1:].tolist() == [-1, -1] and tok[0, 1:].tolist() == [0, 1]


@pytest.mark.parametrize("name", ["tiny", "opt30b"])
def test_topk_reproduces_the_workload_drafts(name):
    w = wl.make(name, attention=False, scale_down=16)
    tok, st = oracle.topk_expand(w.widths, w.tokens[:, 0], w.ssm)
    assert st == 0 and np.array_equal(tok, w.tokens)
