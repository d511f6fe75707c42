"""Pins of the oracle's verifiers against what the pages and the mathematics fix.

SpecInfer (arXiv 2305.09781) sec. 4.3, Algorithm 2:
 (ii)  VerifyGreedy yields exactly the tokens of incremental greedy decoding;
 (iv)  Theorem 4.2: multi-step speculative sampling (MSS) leaves the target law
       unchanged -- exact enumeration over i.i.d. child draws on a vocabulary of
       8, plus a chi-square test on 10^6 seeded runs; k = 1 is the single-step
       proof of "How Speculative Decoding in LLM Serving Actually Works";
 (v)   Theorem 4.3: MSS rejects no more often than naive sampling, exactly and
       measured;
 and the "Speculative decoding" concept page: with one-hot (greedy) target and
 drafter, the stochastic rule reduces to the exact-match test.
"""
import itertools
import os
import zlib

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- #
# greedy
# --------------------------------------------------------------------------- #
def _model_logits(seq, V, sigma=3.0):
    """A deterministic synthetic 'model': logits are N(0, sigma^2) draws seeded
    by a hash of the whole token sequence."""
    h = zlib.crc32(np.asarray(seq, np.int64).tobytes())
    return (np.random.default_rng(h).standard_normal(V) * sigma).astype(np.float32)


def _greedy_tree(rng, prefix, n, V, plant=0.68):
    par = np.full(n, -1, np.int32)
    tok = np.zeros(n, np.int32)
    tok[0] = prefix[-1]
    seqs = {0: list(prefix)}
    for v in range(1, n):
        u = int(rng.integers(0, v))
        par[v] = u
        am = int(np.argmax(_model_logits(seqs[u], V)))
        first_child = not any(par[w] == u for w in range(1, v))
        if first_child and rng.random() < plant:
            t = am
        else:
            t = int(rng.integers(0, V))
        tok[v] = t
        seqs[v] = seqs[u] + [t]
    logits = np.stack([_model_logits(seqs[v], V) for v in range(n)])
    return par, tok, logits


@pytest.mark.parametrize("seed", range(20))
def test_greedy_equals_sequential_greedy_decoding(seed):
    rng = np.random.default_rng(seed)
    V, n = 64, int(rng.integers(1, 30))
    prefix = list(rng.integers(0, V, 5))
    par, tok, logits = _greedy_tree(rng, prefix, n, V)
    r = oracle.verify_greedy(logits[None], par[None], tok[None], np.array([n]))
    cnt = int(r["count"][0])
    seq = list(prefix)
    ref = []
    for _ in range(cnt):
        x = int(np.argmax(_model_logits(seq, V)))
        ref.append(x)
        seq.append(x)
    assert r["tokens"][0, :cnt].tolist() == ref
    # the walk stops only where the target's choice is not among the children
    u = int(r["path"][0, cnt - 1])
    kids = [v for v in range(n) if par[v] == u]
    assert all(tok[c] != ref[-1] for c in kids)


def test_greedy_full_chain_accepts_everything():
    V, n = 50, 9
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((n, V)).astype(np.float32)
    par = np.arange(-1, n - 1, dtype=np.int32)
    tok = np.zeros(n, np.int32)
    for v in range(1, n):
        tok[v] = np.argmax(logits[v - 1])
    r = oracle.verify_greedy(logits[None], par[None], tok[None], np.array([n]))
    assert r["count"][0] == n
    assert r["tokens"][0, : n - 1].tolist() == tok[1:].tolist()
    assert r["tokens"][0, n - 1] == np.argmax(logits[n - 1])
    assert r["path"][0, :n].tolist() == list(range(n))


def test_greedy_ties_and_duplicate_children():
    V = 8
    logits = np.zeros((3, V), np.float32)
    logits[0, [2, 5]] = 1.0            # tie between tokens 2 and 5 -> 2
    par = np.array([-1, 0, 0], np.int32)
    tok = np.array([7, 2, 2], np.int32)  # duplicate children -> the first (node 1)
    r = oracle.verify_greedy(logits[None], par[None], tok[None], np.array([3]))
    assert r["argmax"][0, 0] == 2
    assert r["path"][0, 1] == 1
    assert r["count"][0] == 2 and r["tokens"][0, :2].tolist() == [2, 0]


def test_greedy_rejects_nonfinite():
    logits = np.zeros((1, 2, 4), np.float32)
    logits[0, 1, 3] = np.nan
    r = oracle.verify_greedy(logits, np.array([[-1, 0]]), np.array([[0, 1]]), np.array([2]))
    assert r["status"][0] & oracle.OR_NONFINITE and r["count"][0] == 0


# --------------------------------------------------------------------------- #
# MSS: worked example, exact law, statistics
# --------------------------------------------------------------------------- #
def _fixture(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, _, v = line.partition(":")
            out[k] = np.array([float(x) for x in v.split()])
    return out


def test_mss_worked_example():
    fx = _fixture("mss_worked_example.txt")
    toks = [int(fx["child1_token"][0]), int(fx["child2_token"][0])]
    a, r, g = oracle.mss_node_trace(fx["p"], toks, np.stack([fx["q1"], fx["q2"]]))
    assert g == 0
    np.testing.assert_allclose(a, [fx["a1"][0], fx["a2"][0]], rtol=1e-7)
    np.testing.assert_allclose(r, fx["r2"], atol=1e-7)
    a1, r1, _ = oracle.mss_node_trace(fx["p"], toks[:1], fx["q1"][None])
    np.testing.assert_allclose(r1, fx["r1"], atol=1e-7)
    law = np.zeros(4)
    law[toks[0]] += a[0]
    law[toks[1]] += (1 - a[0]) * a[1]
    law += (1 - a[0]) * (1 - a[1]) * r / r.sum()
    np.testing.assert_allclose(law, fx["law"], atol=1e-7)


def _walk_law(p, q, k):
    """Exact law of one MSS node's output when its k children are drawn i.i.d.
    from q: enumerate all V^k draws, weight each by prod q(x_i)."""
    V = len(p)
    law = np.zeros(V)
    qf = q.astype(np.float32)
    for xs in itertools.product(range(V), repeat=k):
        w = float(np.prod([q[x] for x in xs]))
        if w == 0.0:
            continue
        a, r, _ = oracle.mss_node_trace(p, list(xs), np.tile(qf, (k, 1)))
        reach = 1.0
        for i, x in enumerate(xs):
            law[x] += w * reach * a[i]
            reach *= 1.0 - a[i]
        law += w * reach * r / r.sum()
    return law


def _dist(rng, V, sharp=1.5, zero=False):
    z = rng.standard_normal(V) * sharp
    p = np.exp(z - z.max())
    if zero:
        p[rng.integers(0, V)] = 0.0
    return p / p.sum()


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("seed", range(4))
def test_mss_exact_law_is_target(k, seed):
    rng = np.random.default_rng(seed)
    V = 8
    p = _dist(rng, V, zero=(seed == 3))
    # q in float32, as the drafter's probabilities arrive; the law is exact for q as stored
    q = _dist(rng, V, sharp=2.0).astype(np.float32).astype(np.float64)
    q /= q.sum()
    q = q.astype(np.float32).astype(np.float64)
    law = _walk_law(p, q / q.sum(), k)
    np.testing.assert_allclose(law, p, atol=1e-7 if k else 0)


def test_mss_exact_law_float64_q():
    # with q exactly normalised in double the identity holds to rounding
    rng = np.random.default_rng(42)
    V = 8
    p = _dist(rng, V)
    q = np.full(V, 1.0 / V)      # exact in float32 and float64
    for k in (1, 2, 3):
        np.testing.assert_allclose(_walk_law(p, q, k), p, atol=1e-12)


def _one_node_batch(rng, B, V, k, p_logits, q, child_iid=True):
    n_max = 1 + k
    par = np.tile(np.array([-1] + [0] * k, np.int32), (B, 1))
    tok = np.zeros((B, n_max), np.int32)
    cdf = np.cumsum(q)
    draws = np.searchsorted(cdf, rng.random((B, k)) * cdf[-1], side="right")
    tok[:, 1:] = np.minimum(draws, V - 1)
    logits = np.tile(p_logits.astype(np.float32), (B, n_max, 1))
    ssm = np.tile(q.astype(np.float32), (B, 1, 1))
    q_row = np.zeros((B, n_max), np.int32)
    uni = rng.random((B, 2, n_max)).astype(np.float32)
    return par, tok, logits, ssm, q_row, uni


@pytest.mark.parametrize("k", [1, 2, 3])
def test_mss_chi_square_first_token(k):
    rng = np.random.default_rng(1000 + k)
    V = 8
    z = rng.standard_normal(V) * 1.5
    p = np.exp(z - z.max()); p /= p.sum()
    q = _dist(rng, V, sharp=2.0)
    counts = np.zeros(V)
    total = 0
    for _ in range(5):
        B = 200_000
        par, tok, logits, ssm, q_row, uni = _one_node_batch(rng, B, V, k, z, q)
        r = oracle.verify_mss(logits, ssm, q_row, uni, par, tok, np.full(B, 1 + k))
        counts += np.bincount(r["tokens"][:, 0], minlength=V)
        total += B
    pval = stats.chisquare(counts, p * total).pvalue
    assert pval > 1e-3, (pval, counts / total, p)


def test_mss_chi_square_detects_wrong_law():
    # the same test rejects the drafter's own law, so it has power here
    rng = np.random.default_rng(5)
    V = 8
    z = rng.standard_normal(V) * 1.5
    p = np.exp(z - z.max()); p /= p.sum()
    q = _dist(rng, V, sharp=2.0)
    B = 200_000
    par, tok, logits, ssm, q_row, uni = _one_node_batch(rng, B, V, 2, z, q)
    r = oracle.verify_mss(logits, ssm, q_row, uni, par, tok, np.full(B, 3))
    counts = np.bincount(r["tokens"][:, 0], minlength=V)
    assert stats.chisquare(counts, q * B).pvalue < 1e-6


def test_mss_two_level_law():
    """Law of the first two tokens: the tree's tokens, extended where the step
    emitted only one token by one plain draw from the target at that context,
    must follow p(y1) * p(y2 | y1). Exact enumeration over children drawn i.i.d.
    from the drafter at each node (root: 2 children, each with 1 child)."""
    V = 4
    rng = np.random.default_rng(77)
    p_root = _dist(rng, V)
    p_next = {y: _dist(rng, V) for y in range(V)}
    q_root = np.full(V, 0.25)
    q_next = {y: _dist(rng, V, sharp=1.0).astype(np.float32).astype(np.float64) for y in range(V)}
    for y in range(V):
        q_next[y] = (q_next[y] / q_next[y].sum()).astype(np.float32).astype(np.float64)
        q_next[y] /= q_next[y].sum()
    law = np.zeros((V, V))
    for x1, x2 in itertools.product(range(V), repeat=2):          # root's two children
        w_root = q_root[x1] * q_root[x2]
        a, r, _ = oracle.mss_node_trace(p_root, [x1, x2], np.tile(q_root.astype(np.float32), (2, 1)))
        # child c accepted with probability reach * a_c; then its own child y ~ q_next[x_c]
        reach = 1.0
        for i, xc in enumerate((x1, x2)):
            pa = w_root * reach * a[i]
            reach *= 1 - a[i]
            for y in range(V):
                wy = q_next[xc][y]
                a2, r2, _ = oracle.mss_node_trace(p_next[xc], [y], q_next[xc].astype(np.float32)[None])
                law[xc, y] += pa * wy * a2[0]
                law[xc] += pa * wy * (1 - a2[0]) * r2 / r2.sum()
        # all rejected: correction token y1 from the residual, then y2 ~ p(. | y1)
        rr = r / r.sum()
        for y1 in range(V):
            law[y1] += w_root * reach * rr[y1] * p_next[y1]
    ref = p_root[:, None] * np.stack([p_next[y] for y in range(V)])
    np.testing.assert_allclose(law, ref, atol=1e-7)


# --------------------------------------------------------------------------- #
# Theorem 4.3
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("seed", range(5))
def test_mss_rejects_no_more_than_naive_exact(k, seed):
    rng = np.random.default_rng(300 + seed)
    V = 8
    p = _dist(rng, V)
    q = _dist(rng, V, sharp=2.0).astype(np.float32).astype(np.float64)
    q /= q.sum()
    mss = naive = 0.0
    for xs in itertools.product(range(V), repeat=k):
        w = float(np.prod([q[x] for x in xs]))
        a, _, _ = oracle.mss_node_trace(p, list(xs), np.tile(q.astype(np.float32), (k, 1)))
        mss += w * float(np.prod(1 - a))
        naive += w * (1.0 - sum(p[x] for x in set(xs)))
    assert mss <= naive + 1e-12


def test_mss_rejects_no_more_than_naive_measured():
    rng = np.random.default_rng(11)
    V, k, B = 8, 3, 200_000
    z = rng.standard_normal(V) * 1.5
    q = _dist(rng, V, sharp=2.0)
    par, tok, logits, ssm, q_row, uni = _one_node_batch(rng, B, V, k, z, q)
    nn = np.full(B, 1 + k)
    m = oracle.verify_mss(logits, ssm, q_row, uni, par, tok, nn)
    nv = oracle.verify_naive(logits, par, tok, nn, uni)
    rej_m = np.mean(m["count"] == 1)
    rej_n = np.mean(nv["count"] == 1)
    se = np.sqrt(rej_m * (1 - rej_m) / B + rej_n * (1 - rej_n) / B)
    assert rej_m <= rej_n + 4 * se
    assert rej_m < rej_n          # strictly better on this case


# --------------------------------------------------------------------------- #
# limits, guards, conventions
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("seed", range(6))
def test_mss_one_hot_limit_is_greedy(seed):
    """Greedy as the one-hot limit of the stochastic rule: target one-hot at its
    argmax (tiny temperature), each child's drafter one-hot at its own token."""
    rng = np.random.default_rng(seed)
    V, n = 16, 14
    par = np.full(n, -1, np.int32)
    for v in range(1, n):
        par[v] = rng.integers(0, v)
    logits = rng.standard_normal((n, V)).astype(np.float32) * 4
    tok = np.zeros(n, np.int32)
    for v in range(1, n):
        tok[v] = np.argmax(logits[par[v]]) if rng.random() < 0.6 else rng.integers(0, V)
    ssm = np.zeros((n, V), np.float32)
    ssm[np.arange(n), tok] = 1.0
    q_row = np.arange(n, dtype=np.int32)
    uni = rng.uniform(1e-3, 1 - 1e-3, (2, n)).astype(np.float32)
    m = oracle.verify_mss(logits[None], ssm[None], q_row[None], uni[None], par[None], tok[None], [n],
                          temperature=1e-3)
    g = oracle.verify_greedy(logits[None], par[None], tok[None], [n])
    c = int(g["count"][0])
    assert m["count"][0] == c
    assert m["tokens"][0, :c].tolist() == g["tokens"][0, :c].tolist()


def test_mss_zero_normaliser_guard():
    # drafter rows that over-cover the target (unnormalised q) leave max(0, p - q) = 0
    V = 2
    logits = np.zeros((1, 2, V), np.float32)          # p = (1/2, 1/2)
    ssm = np.full((1, 1, V), 0.6, np.float32)
    par = np.array([[-1, 0]], np.int32)
    tok = np.array([[0, 0]], np.int32)
    uni = np.array([[[0.0, 0.9], [0.3, 0.0]]], np.float32)   # accept test of node 1 fails (0.9 > 5/6)
    r = oracle.verify_mss(logits, ssm, np.zeros((1, 2), np.int32), uni, par, tok, [2])
    assert r["status"][0] & oracle.OR_ZERO_RESID
    assert r["count"][0] == 1 and r["tokens"][0, 0] == 0    # residual kept = p, u = 0.3 -> token 0


def test_mss_leaf_root_samples_bonus_from_target():
    V = 5
    logits = np.log(np.array([[[0.1, 0.2, 0.3, 0.2, 0.2]]], np.float32))
    for u, want in ((0.05, 0), (0.15, 1), (0.31, 2), (0.61, 3), (0.95, 4)):
        uni = np.array([[[0.0], [u]]], np.float32)
        r = oracle.verify_mss(logits, np.zeros((1, 1, V), np.float32), np.zeros((1, 1), np.int32), uni,
                              np.array([[-1]]), np.array([[0]]), [1])
        assert r["count"][0] == 1 and r["tokens"][0, 0] == want


def test_mss_zero_q_accepts():
    V = 4
    logits = np.zeros((1, 2, V), np.float32)
    ssm = np.array([[[0.5, 0.5, 0.0, 0.0]]], np.float32)
    uni = np.array([[[0.0, 0.999], [0.1, 0.1]]], np.float32)
    r = oracle.verify_mss(logits, ssm, np.zeros((1, 2), np.int32), uni, np.array([[-1, 0]]),
                          np.array([[0, 3]]), [2])
    assert r["path"][0, 1] == 1 and r["tokens"][0, 0] == 3


def test_mss_margin_reporting():
    V = 4
    logits = np.zeros((1, 2, V), np.float32)          # p = 1/4 each
    ssm = np.array([[[0.1, 0.1, 0.3, 0.5]]], np.float32)
    a = 0.25 / np.float64(np.float32(0.5))              # a for token 3 = 0.5
    uni = np.array([[[0.0, np.float32(a + 4e-7)], [0.5, 0.5]]], np.float32)
    r = oracle.verify_mss(logits, ssm, np.zeros((1, 2), np.int32), uni, np.array([[-1, 0]]),
                          np.array([[0, 3]]), [2])
    assert r["lm_pos"][0] == 0 and r["min_margin"][0] < 1e-6


def test_mss_bad_q_row_flagged():
    r = oracle.verify_mss(np.zeros((1, 2, 4), np.float32), np.zeros((1, 1, 4), np.float32),
                          np.array([[0, 5]], np.int32), np.zeros((1, 2, 2), np.float32),
                          np.array([[-1, 0]]), np.array([[0, 1]]), [2])
    assert r["status"][0] & oracle.OR_INDEX and r["count"][0] == 0


def test_mss_nonfinite_only_where_read():
    V = 4
    logits = np.zeros((2, 3, V), np.float32)
    ssm = np.full((2, 1, V), 0.25, np.float32)
    par = np.array([[-1, 0, 1]] * 2, np.int32)
    tok = np.array([[0, 1, 2]] * 2, np.int32)
    uni = np.zeros((2, 2, 3), np.float32)          # every child accepted
    logits[0, 2, 1] = np.nan                         # on the walk (node 2 is reached)
    ssm[1, 0, 3] = np.inf                            # drafter row never fully read: children accepted
    r = oracle.verify_mss(logits, ssm, np.zeros((2, 3), np.int32), uni, par, tok, [3, 3])
    assert r["status"][0] & oracle.OR_NONFINITE and r["count"][0] == 0
    assert r["status"][1] == 0 and r["count"][1] == 3


def test_naive_law_and_rejection_closed_form():
    """Naive sampling (SpecInfer sec. 4.3): the first token is a draw from p, and
    the walk stops at the root exactly when that draw is not a child token, so
    the rejection rate is 1 - sum_{x in children} p(x)."""
    rng = np.random.default_rng(21)
    V, B = 8, 200_000
    z = rng.standard_normal(V) * 1.5
    p = np.exp(z - z.max()); p /= p.sum()
    kids = np.array([1, 4, 4], np.int32)           # a duplicate child token counts once
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    tok = np.tile(np.concatenate([[0], kids]).astype(np.int32), (B, 1))
    logits = np.tile(z.astype(np.float32), (B, 4, 1))
    uni = rng.random((B, 2, 4)).astype(np.float32)
    r = oracle.verify_naive(logits, par, tok, np.full(B, 4), uni)
    first = r["tokens"][:, 0]
    assert stats.chisquare(np.bincount(first, minlength=V), p * B).pvalue > 1e-3
    rej = np.mean(r["count"] == 1)
    expect = 1.0 - p[1] - p[4]
    assert abs(rej - expect) < 4 * np.sqrt(expect * (1 - expect) / B)


def test_kv_commit_hand_built():
    """Only the accepted path keeps its cache entries (SpecInfer sec. 4.2): path
    node i moves to row P + i; every other row is untouched."""
    B, H, L, d, n_max, P = 1, 2, 16, 4, 6, 5
    cache = np.arange(B * H * L * d, dtype=np.float32).reshape(B, H, L, d)
    dfs_of = np.array([[0, 3, 1, 5, 2, 4]], np.int32)      # input id -> DFS index
    path = np.full((1, n_max + 1), -1, np.int32)
    path[0, :3] = [0, 1, 3]                                  # root, then nodes at DFS 3 and 5
    k2, v2, npl = oracle.kv_commit(cache, cache + 1000, [P], dfs_of, path, [3])
    assert npl.tolist() == [P + 3]
    for h in range(H):
        assert np.array_equal(k2[0, h, P + 0], cache[0, h, P + 0])
        assert np.array_equal(k2[0, h, P + 1], cache[0, h, P + 3])
        assert np.array_equal(k2[0, h, P + 2], cache[0, h, P + 5])
        assert np.array_equal(v2[0, h, P + 2], cache[0, h, P + 5] + 1000)
        untouched = [r for r in range(L) if r not in (P, P + 1, P + 2)]
        assert np.array_equal(k2[0, h, untouched], cache[0, h, untouched])
