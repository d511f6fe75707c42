"""tree_expand_topk (the drafter's top-k expansion, SpecInfer sec. 3, Fig. 3) on
the GPU against the oracle's or_topk_expand: integer tokens, bit-exact (both
sides order the same fp32 values); then the drafted tokens feed tree_build."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300 import workloads as wl
from tree_speculative_verification_gb300.step import to_device

pytestmark = pytest.mark.gpu


def _gpu(widths, root, ssm, n_max):
    B = ssm.shape[0]
    tok = torch.full((B, n_max), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.tree_expand_topk(tok, to_device(root, "cuda"), to_device(ssm, "cuda"), widths, status=st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("widths,V", [((2,), 8), ((3, 2), 257), ((2, 2, 2, 2, 1), 50272), ((1, 1, 3, 1, 1, 1, 1, 1), 32000),
                                      ((5, 3), 1000), ((), 64)])
def test_expand_matches_oracle(widths, V):
    rng = np.random.default_rng(V + len(widths))
    par = oracle.widths_parent(widths)
    n = len(par)
    n_internal = max(1, int(np.max(par)) + 1)
    B = 6
    z = rng.standard_normal((B, n_internal, V)) * 2
    ssm = (np.exp(z) / np.exp(z).sum(-1, keepdims=True)).astype(np.float32)
    ssm[0, 0, :4] = ssm[0, 0, 4]                       # ties at the top of one row
    root = rng.integers(0, V, B).astype(np.int32)
    got, st = _gpu(widths, root, ssm, n + 2)
    ref, rst = oracle.topk_expand(widths, root, ssm, n + 2)
    assert st == rst == 0
    assert np.array_equal(got[:, :n], ref[:, :n])
    assert (got[:, n:] == -7).all()                    # past the tree: not written


def test_expand_nonfinite_row():
    ssm = np.full((2, 3, 16), 1 / 16, np.float32)
    ssm[1, 2, 5] = np.inf
    got, st = _gpu((2, 1), np.array([3, 4], np.int32), ssm, 5)
    ref, rst = oracle.topk_expand((2, 1), np.array([3, 4], np.int32), ssm, 5)
    assert st & api.STATUS_NONFINITE and rst & 4
    assert np.array_equal(got, ref)


def test_expand_then_build_reproduces_the_workload_tree():
    """The OPT-30B-shaped layer drafts its tree by top-k on the host: the device
    expansion + tree_build gives the same linearised tree."""
    w = wl.make("opt30b", attention=False)
    got, st = _gpu(w.widths, w.tokens[:, 0].copy(), w.ssm, w.n_max)
    assert st == 0 and np.array_equal(got, w.tokens)
    t = api.Tree(w.B, w.n_max)
    api.tree_build(t, to_device(got, "cuda"), widths=w.widths)
    ref_t = oracle.tree_build(w.parent, w.tokens)
    torch.cuda.synchronize()
    assert np.array_equal(t.token.cpu().numpy(), ref_t["token"])
