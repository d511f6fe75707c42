"""verify_greedy in each of its launch forms against the oracle (SpecInfer
Algorithm 2, VerifyGreedy): tokens, path, count and per-node argmax bit-exact.

The shapes pick the forms: each (row, part) segment taken by one bulk copy
into shared memory (8 x 21 x 32000, the LLaMA-7B-shaped rows; 1 x 8 x 50272;
12 x 19 x 40000, about 36 MB of logits) and the 128-thread form with float4
loads (2 x 21 x 32000, whose 16 KB parts are below the bulk-copy size;
4 x 128 x 32000, too many rows for one wave of bulk-copy CTAs). Each case has
ragged trees, a request with no nodes (batches of three and more), a NaN and
an infinity in rows of two other requests (batches of four and more), maxima
planted at children's tokens so that the walks go deep, and pairs of equal
maxima in adjacent entries (the lower index wins) placed where a row cut
into 2..8 equal parts, or the rows' logits taken as one array cut into equal
parts for two CTAs per SM, would be split. The call runs twice, so that the second one finds the counters the
first one left."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import to_device

pytestmark = pytest.mark.gpu

CASES = [(8, 21, 32000), (2, 21, 32000), (1, 8, 50272), (12, 19, 40000), (4, 128, 32000)]


def _inputs(B, n_max, V, seed):
    rng = np.random.default_rng(seed)
    n_nodes = rng.integers(max(1, n_max // 2), n_max + 1, size=B).astype(np.int32)
    n_nodes[rng.integers(0, B)] = n_max
    if B > 2:
        n_nodes[1] = 0                                        # an empty request
    parent = np.full((B, n_max), -1, np.int32)
    tokens = np.zeros((B, n_max), np.int32)
    logits = rng.standard_normal((B, n_max, V)).astype(np.float32)
    for b in range(B):
        n = int(n_nodes[b])
        for v in range(1, n):
            parent[b, v] = rng.integers(max(0, v - 4), v)     # bushy, a few levels deep
        tokens[b, :n] = rng.integers(0, V, size=n)
        for v in range(n):
            kids = [c for c in range(1, n) if parent[b, c] == v]
            if kids and rng.random() < 0.9:                   # the walk continues through v
                logits[b, v, tokens[b, kids[rng.integers(0, len(kids))]]] = 20.0
    # equal maxima in adjacent entries, at the edges of equal parts of the flattened rows
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    V4 = V // 4
    F = B * n_max * V4
    per = max(-(-F // (2 * sms)), (V4 + 6) // 7)
    for edge in range(per, F, per):
        r, x = divmod(4 * edge, V)
        b, v = divmod(r, n_max)
        if 0 < x < V and rng.random() < 0.5:
            logits[b, v, x - 1] = logits[b, v, x] = 12.0
    # and at the edges of a row cut into s equal parts of float4s (s = 2..8)
    for b in range(B):
        for v in range(n_max):
            s = int(rng.integers(2, 9))
            x = 4 * (-(-V4 // s))
            if x < V and rng.random() < 0.3:
                logits[b, v, x - 1] = logits[b, v, x] = 12.0
    if B >= 4:                                                # two requests emptied by non-finite rows
        good = [b for b in range(B) if n_nodes[b] > 1]
        logits[good[0], n_nodes[good[0]] - 1, V // 3] = np.nan
        logits[good[-1], 0, V - 1] = np.inf
    return parent, tokens, n_nodes, logits


@pytest.mark.parametrize("B,n_max,V", CASES)
def test_greedy_forms_match_oracle(B, n_max, V):
    parent, tokens, n_nodes, logits = _inputs(B, n_max, V, seed=B * 1000 + n_max)
    ref = oracle.verify_greedy(logits, parent, tokens, n_nodes)
    d = lambda a: to_device(a, "cuda")
    t = api.Tree(B, n_max)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.tree_build(t, d(tokens), d(parent), d(n_nodes), status=st)
    ws = api.workspace(api.TS_OP_VERIFY_GREEDY, B, n_max=n_max, V=V)
    lg = d(logits)
    for call in range(2):
        ot = torch.full((B, n_max + 1), -1, dtype=torch.int32, device="cuda")
        op = torch.full((B, n_max + 1), -1, dtype=torch.int32, device="cuda")
        oc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        am = torch.full((B, n_max), -1, dtype=torch.int32, device="cuda")
        api.verify_greedy(ot, op, oc, lg, t, am, ws, st)
        torch.cuda.synchronize()
        cnt = oc.cpu().numpy()
        assert cnt.tolist() == ref["count"].tolist(), call
        ot, op, am = ot.cpu().numpy(), op.cpu().numpy(), am.cpu().numpy()
        for b in range(B):
            c = int(cnt[b])
            assert ot[b, :c].tolist() == ref["tokens"][b, :c].tolist(), (call, b)
            assert op[b, :c].tolist() == ref["path"][b, :c].tolist(), (call, b)
            if ref["status"][b] == 0:
                n = int(n_nodes[b])
                assert am[b, :n].tolist() == ref["argmax"][b, :n].tolist(), (call, b)
    bits = st.item()
    assert bool(bits & api.STATUS_NONFINITE) == (B >= 4)
    assert not bits & api.STATUS_TIMEOUT
    clean = ref["status"] == 0
    assert (ref["count"][clean] >= 3).any()                   # deep walks were exercised
