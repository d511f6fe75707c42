"""tree_build_append (tree_build in widths mode and kv_append in one launch)
against the two separate calls: every tree array and every cache byte
identical, for expansion configurations of one to eight levels, bf16 and fp32
caches, prefixes at 0 and at tile edges, and a request past the cache's end
(TS_STATUS_INDEX, its rows left alone)."""
import numpy as np
import pytest
import torch

from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import to_device

pytestmark = pytest.mark.gpu

FIELDS = ("n_nodes", "perm", "dfs_of", "parent", "token", "depth", "pos", "sub_end", "anc")


def _arrays(t):
    return {f: getattr(t, f).cpu().numpy().copy() for f in FIELDS}


@pytest.mark.parametrize("widths", [(1,), (3, 2), (2, 2, 1), (2, 2, 2, 2, 1), (1, 1, 3, 1, 1, 1, 1, 1)])
@pytest.mark.parametrize("bf16", [True, False])
def test_fused_equals_separate(widths, bf16):
    rng = np.random.default_rng(len(widths) * 7 + bf16)
    B, H = 4, 3
    d = 128 if bf16 else 64
    n = 1 + sum(int(np.prod(widths[:l + 1])) for l in range(len(widths)))
    n_max = n + 3
    prefix = np.array([0, 63, 200, 260], np.int32)
    L_max = 256 + n_max                       # request 3 runs past the cache's end
    dt = torch.bfloat16 if bf16 else torch.float32
    tok = to_device(rng.integers(0, 1000, (B, n_max)).astype(np.int32), "cuda")
    kn = torch.randn(B, n_max, H, d, device="cuda").to(dt)
    vn = torch.randn(B, n_max, H, d, device="cuda").to(dt)
    kc0 = torch.randn(B, H, L_max, d, device="cuda").to(dt)
    vc0 = torch.randn(B, H, L_max, d, device="cuda").to(dt)
    pl = to_device(prefix, "cuda")
    # separate calls
    t1, st1 = api.Tree(B, n_max), torch.zeros(1, dtype=torch.int32, device="cuda")
    kc1, vc1 = kc0.clone(), vc0.clone()
    api.tree_build(t1, tok, widths=widths, prefix_len=pl, status=st1)
    api.kv_append(kc1, vc1, kn, vn, pl, t1, st1)
    # one launch
    t2, st2 = api.Tree(B, n_max), torch.zeros(1, dtype=torch.int32, device="cuda")
    kc2, vc2 = kc0.clone(), vc0.clone()
    api.tree_build_append(t2, tok, widths, pl, kc2, vc2, kn, vn, st2)
    torch.cuda.synchronize()
    a1, a2 = _arrays(t1), _arrays(t2)
    for f in FIELDS:
        assert np.array_equal(a1[f], a2[f]), f
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert st1.item() == st2.item() == api.STATUS_INDEX
