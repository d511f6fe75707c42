"""GPU parity of the verifiers against the oracle (SpecInfer Algorithm 2).

Greedy: tokens, path, count and per-node argmax bit-exact. MSS: the same
supplied uniforms on both sides; tokens bit-exact up to the oracle's first
decision whose margin is under 1e-6 (those requests are counted and printed);
counts equal where no low-margin decision occurred."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import DeviceStep, to_device

from _helpers import exclusion_bound, low_margin_prob, oracle_tree, workload

pytestmark = pytest.mark.gpu


def _greedy_check(w, s):
    parent, tokens, n_nodes, _, _ = oracle_tree(w)
    ref = oracle.verify_greedy(w.logits, parent, tokens, n_nodes)
    cnt = s.out_count.cpu().numpy()
    assert cnt.tolist() == ref["count"].tolist()
    ot, op, am = s.out_tokens.cpu().numpy(), s.out_path.cpu().numpy(), s.argmax.cpu().numpy()
    for b in range(w.B):
        c, n = int(cnt[b]), int(n_nodes[b])
        assert ot[b, :c].tolist() == ref["tokens"][b, :c].tolist()
        assert op[b, :c].tolist() == ref["path"][b, :c].tolist()
        assert am[b, :n].tolist() == ref["argmax"][b, :n].tolist()
    return ref


def _mss_check(w, s):
    """Tokens, path and count bit-exact against the oracle up to the oracle's
    first decision with a margin under 1e-6. Every request whose result
    differs from the oracle's at all must carry a low-margin count from the
    device (a decision flips only where the device's own margin is below its
    rounding error, far below 1e-6). The number of requests the oracle flags
    is bounded by the expected number of low-margin final draws (the measure
    of u within 1e-6 of a cumulative-sum boundary at each request's last
    node) plus four standard deviations."""
    parent, tokens, n_nodes, p_row, q_row = oracle_tree(w)
    ref = oracle.verify_mss(w.logits, w.ssm, q_row, w.uniforms, parent, tokens, n_nodes, w.temperature, p_row=p_row)
    cnt, ot, op = s.mss_count.cpu().numpy(), s.mss_tokens.cpu().numpy(), s.mss_path.cpu().numpy()
    lowm = s.mss_lowmargin.cpu().numpy()
    excluded, probs = 0, []
    for b in range(w.B):
        lm = int(ref["lm_pos"][b])
        rc = int(ref["count"][b])
        last = int(ref["path"][b, rc - 1])
        row = last if p_row is None else int(p_row[b, last])
        probs.append(low_margin_prob(w.logits[b, row], w.temperature) + 2e-6 * rc)
        if lm < rc:
            excluded += 1
        k = min(lm, rc)
        assert ot[b, :k].tolist() == ref["tokens"][b, :k].tolist(), (b, ot[b, :rc], ref["tokens"][b, :rc], lm)
        assert op[b, :k].tolist() == ref["path"][b, :k].tolist(), b
        if lm >= rc:
            assert cnt[b] == rc, (b, cnt[b], rc)
            assert ot[b, :rc].tolist() == ref["tokens"][b, :rc].tolist()
        same = cnt[b] == rc and ot[b, :rc].tolist() == ref["tokens"][b, :rc].tolist()
        assert same or lowm[b] > 0, f"request {b} differs from the oracle with no low-margin decision reported"
    bound = exclusion_bound(probs)
    print(f"[{w.name}] MSS requests with an oracle low-margin decision: {excluded} of {w.B} (bound {bound:.1f}); "
          f"device-reported: {int((lowm > 0).sum())}; min margin {ref['min_margin'].min():.3g}")
    assert excluded <= bound
    return ref


@pytest.mark.parametrize("name", ["tiny", "llama7b", "long65b"])
def test_greedy_full_size(name):
    w = workload(name, attention=False)
    s = DeviceStep(w, attention=False)
    s.build()
    s.verify("greedy")
    torch.cuda.synchronize()
    assert s.status.item() == 0
    ref = _greedy_check(w, s)
    if name == "llama7b":
        # the 0.68 plant rate shows in the accepted lengths
        assert ref["count"].mean() > 1.5


@pytest.mark.parametrize("name", ["tiny", "merge", "long65b", "opt30b"])
def test_mss_full_size(name):
    w = workload(name, attention=False)
    s = DeviceStep(w, attention=False)
    s.build()
    s.verify("mss")
    torch.cuda.synchronize()
    assert s.status.item() & ~api.STATUS_ZERO_RESID == 0
    _mss_check(w, s)


def _tiny_tree_case(rng, B, n, V, k_per_node=None):
    par = np.full((B, n), -1, np.int32)
    for b in range(B):
        for v in range(1, n):
            par[b, v] = rng.integers(0, v)
    tok = rng.integers(0, V, (B, n)).astype(np.int32)
    return par, tok


@pytest.mark.parametrize("V", [8, 257, 1000, 32000])
def test_mss_random_trees_many_seeds(V):
    """Random topologies and distributions, children drawn i.i.d. from q at the
    parent; V = 257 exercises the scalar (non-float4) path."""
    rng = np.random.default_rng(V)
    B, n = 64, 12
    par, _ = _tiny_tree_case(rng, B, n, V)
    logits = (rng.standard_normal((B, n, V)) * 2.0).astype(np.float32)
    z = logits + rng.standard_normal((B, n, V)).astype(np.float32)
    q = np.exp(z - z.max(-1, keepdims=True)); q /= q.sum(-1, keepdims=True); q = q.astype(np.float32)
    tok = np.zeros((B, n), np.int32)
    for b in range(B):
        for v in range(1, n):
            u = par[b, v]
            cdf = np.cumsum(q[b, u].astype(np.float64))
            tok[b, v] = min(int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right")), V - 1)
    q_row = np.where(par >= 0, par, 0).astype(np.int32)
    uni = rng.random((B, 2, n)).astype(np.float32)
    t = api.Tree(B, n)
    d = lambda a: to_device(a, "cuda")
    api.tree_build(t, d(tok), d(par), d(np.full(B, n, np.int32)))
    ot = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
    op = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
    oc = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.verify_mss(ot, op, oc, d(logits), d(q), d(q_row), d(uni), 1.0, t, status=st)
    torch.cuda.synchronize()
    ref = oracle.verify_mss(logits, q, q_row, uni, par, tok, np.full(B, n))
    got = oc.cpu().numpy()
    ex = 0
    for b in range(B):
        lm, rc = int(ref["lm_pos"][b]), int(ref["count"][b])
        k = min(lm, rc)
        ex += lm < rc
        assert ot[b, :k].tolist() == ref["tokens"][b, :k].tolist()
        if lm >= rc:
            assert got[b] == rc
    assert ex <= 3


def test_mss_temperature_and_leaf_bonus():
    rng = np.random.default_rng(5)
    B, n, V = 32, 6, 64
    par = np.tile(np.array([-1, 0, 1, 2, 3, 4], np.int32), (B, 1))       # chains: leaf bonus when all accepted
    logits = (rng.standard_normal((B, n, V)) * 3).astype(np.float32)
    tok = rng.integers(0, V, (B, n)).astype(np.int32)
    # half the requests draft the target's own favourite token at every node, so
    # p(x)/q(x) > 1 there and the walk reaches the leaf
    tok[: B // 2, 1:] = np.argmax(logits[: B // 2, :-1], axis=-1)
    q = np.full((B, n, V), 1.0 / V, np.float32)
    uni = (rng.random((B, 2, n)) * 0.05).astype(np.float32)             # small accept uniforms: deep walks
    t = api.Tree(B, n)
    d = lambda a: to_device(a, "cuda")
    api.tree_build(t, d(tok), d(par), d(np.full(B, n, np.int32)))
    outs = [torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda") for _ in range(2)]
    oc = torch.zeros(B, dtype=torch.int32, device="cuda")
    api.verify_mss(outs[0], outs[1], oc, d(logits), d(q), d(np.where(par >= 0, par, 0).astype(np.int32)), d(uni),
                   0.7, t)
    torch.cuda.synchronize()
    ref = oracle.verify_mss(logits, q, np.where(par >= 0, par, 0), uni, par, tok, np.full(B, n), temperature=0.7)
    for b in range(B):
        lm, rc = int(ref["lm_pos"][b]), int(ref["count"][b])
        assert outs[0][b, :min(lm, rc)].tolist() == ref["tokens"][b, :min(lm, rc)].tolist()
    assert (ref["count"] == n).any()        # some walk reached the leaf and drew the bonus token


def test_greedy_ties_nan_and_scalar_path():
    B, n, V = 3, 3, 13                                                   # V % 4 != 0: scalar path
    logits = np.zeros((B, n, V), np.float32)
    logits[:, 0, [4, 9]] = 2.0                                           # tie -> token 4
    par = np.tile(np.array([-1, 0, 0], np.int32), (B, 1))
    tok = np.tile(np.array([0, 4, 4], np.int32), (B, 1))                 # duplicate children -> first
    logits[2, 2, 7] = np.nan                                             # request 2 emptied
    t = api.Tree(B, n)
    d = lambda a: to_device(a, "cuda")
    api.tree_build(t, d(tok), d(par), d(np.full(B, n, np.int32)))
    ot = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
    op = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
    oc = torch.zeros(B, dtype=torch.int32, device="cuda")
    am = torch.full((B, n), -1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = api.workspace(api.TS_OP_VERIFY_GREEDY, B, n_max=n, V=V)
    api.verify_greedy(ot, op, oc, d(logits), t, am, ws, st)
    torch.cuda.synchronize()
    ref = oracle.verify_greedy(logits, par, tok, np.full(B, n))
    assert oc.tolist() == ref["count"].tolist() == [2, 2, 0]
    assert am[0].tolist() == ref["argmax"][0].tolist()
    assert op[0, :2].tolist() == [0, 1]
    assert st.item() & api.STATUS_NONFINITE
    assert int(ws.count_nonzero()) == 0 or int(ws[: (B * 4 + 255) // 256 * 256].count_nonzero()) == 0


def test_mss_zero_residual_guard_and_nonfinite():
    V = 2
    B = 2
    logits = np.zeros((B, 2, V), np.float32)
    ssm = np.full((B, 1, V), 0.6, np.float32)
    par = np.array([[-1, 0]] * B, np.int32)
    tok = np.array([[0, 0]] * B, np.int32)
    uni = np.array([[[0.0, 0.9], [0.3, 0.0]]] * B, np.float32)
    logits[1, 0, 1] = np.inf
    t = api.Tree(B, 2)
    d = lambda a: to_device(a, "cuda")
    api.tree_build(t, d(tok), d(par), d(np.full(B, 2, np.int32)))
    ot = torch.full((B, 3), -1, dtype=torch.int32, device="cuda")
    op = torch.full((B, 3), -1, dtype=torch.int32, device="cuda")
    oc = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.verify_mss(ot, op, oc, d(logits), d(ssm), d(np.zeros((B, 2), np.int32)), d(uni), 1.0, t, status=st)
    torch.cuda.synchronize()
    ref = oracle.verify_mss(logits, ssm, np.zeros((B, 2)), uni, par, tok, [2, 2])
    assert oc.tolist() == ref["count"].tolist() == [1, 0]
    assert ot[0, 0].item() == ref["tokens"][0, 0] == 0
    assert st.item() & api.STATUS_ZERO_RESID and st.item() & api.STATUS_NONFINITE


def test_mss_bad_row_index():
    B, n, V = 1, 2, 8
    t = api.Tree(B, n)
    d = lambda a: to_device(a, "cuda")
    api.tree_build(t, d(np.zeros((B, n), np.int32)), d(np.array([[-1, 0]], np.int32)), d(np.array([2], np.int32)))
    ot = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
    oc = torch.ones(B, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.verify_mss(ot, ot.clone(), oc, d(np.zeros((B, n, V), np.float32)), d(np.zeros((B, 1, V), np.float32)),
                   d(np.array([[0, 3]], np.int32)), d(np.zeros((B, 2, n), np.float32)), 1.0, t, status=st)
    torch.cuda.synchronize()
    assert oc.item() == 0 and st.item() & api.STATUS_INDEX


def test_mss_fast_walk_zero_residual_rebuild_and_nonfinite():
    """The shared-memory walk (V a multiple of 4): a rejection whose residual
    max(0, p - q) is zero everywhere keeps the residual (status ZERO_RESID) and
    the walk goes on with the next child, then samples; compared with the
    oracle. Request 0 accepts the second child, request 1 rejects both and
    samples from p, request 2 meets a NaN in the second child's drafter row."""
    V, B, n = 8, 3, 3
    logits = np.zeros((B, n, V), np.float32)          # p uniform: 1/8 at every node
    logits[:, 2, 6] = 2.0
    ssm = np.full((B, 2, V), 0.6, np.float32)           # q >= p everywhere: zero residual
    ssm[:, 1, :] = 0.125
    ssm[:, 1, 5] = 0.3
    ssm[2, 1, 4] = np.nan
    q_row = np.array([[0, 0, 1]] * B, np.int32)
    par = np.array([[-1, 0, 0]] * B, np.int32)
    tok = np.array([[0, 3, 5]] * B, np.int32)
    uni = np.zeros((B, 2, n), np.float32)
    uni[:, 0, 1] = 0.9                                   # child 1: p/q = 0.208, rejected
    uni[0, 0, 2] = 0.1                                   # child 2: p/q = 0.417, accepted for request 0
    uni[1, 0, 2] = 0.8                                   # rejected for request 1
    uni[2, 0, 2] = 0.8
    uni[:, 1, 0] = 0.55                                  # the final sample at the root
    uni[:, 1, 2] = 0.3
    t = api.Tree(B, n)
    d = lambda a: to_device(a, "cuda")
    api.tree_build(t, d(tok), d(par), d(np.full(B, n, np.int32)))
    ot = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
    op = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
    oc = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.verify_mss(ot, op, oc, d(logits), d(ssm), d(q_row), d(uni), 1.0, t, status=st)
    torch.cuda.synchronize()
    ref = oracle.verify_mss(logits, ssm, q_row, uni, par, tok, [n] * B)
    assert oc.tolist() == ref["count"].tolist()
    assert ref["count"].tolist()[2] == 0 and ref["count"].tolist()[0] == 2 and ref["count"].tolist()[1] == 1
    for b in range(2):
        c = int(ref["count"][b])
        assert ot[b, :c].tolist() == ref["tokens"][b, :c].tolist()
    assert st.item() & api.STATUS_ZERO_RESID and st.item() & api.STATUS_NONFINITE
