"""The arithmetic behind tree_build_append: in an expansion tree <k_1..k_m>
numbered level by level, node v of level d with index idx has the child ranks
of its root path as the mixed-radix digits of idx (radices k_1..k_d), and its
depth-first position is the sum over the path of 1 + rank * (size of a subtree
one level below). Pinned here to the oracle's depth-first linearisation (a
plain DFS over parent[]), so a wrong digit order or subtree size fails."""
import numpy as np
import pytest

import oracle


def _arith_dfs(widths):
    m = len(widths)
    sub = [1] * (m + 1)
    for l in range(m - 1, -1, -1):
        sub[l] = 1 + widths[l] * sub[l + 1]
    starts, n, level_n = [0, 1], 1, 1
    for k in widths:
        level_n *= k
        n += level_n
        starts.append(n)
    out = []
    for v in range(n):
        d = max(l for l in range(m + 1) if starts[l] <= v)
        idx, pos = v - starts[d], 0
        for l in range(d - 1, -1, -1):   # digits from the last level up
            c = idx % widths[l]
            idx //= widths[l]
            pos += 1 + c * sub[l + 1]
        out.append(pos)
    return np.array(out)


@pytest.mark.parametrize("widths", [(), (1,), (3,), (2, 2, 1), (3, 2), (2, 2, 2, 2, 1), (1, 1, 3, 1, 1, 1, 1, 1),
                                    (4, 1, 3)])
def test_dfs_positions_match_the_oracle(widths):
    par = oracle.widths_parent(widths)
    ref = oracle.tree_build(par[None, :], np.zeros((1, len(par)), np.int32))["dfs_of"][0]
    assert np.array_equal(_arith_dfs(widths), ref)
