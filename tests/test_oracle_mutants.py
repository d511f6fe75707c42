"""The pins have teeth: each planted mistake in the oracle (compiled with
-DOR_MUTANT=k, on the CPU) must make at least one oracle pin fail.

  1 residual subtracts q only at the rejected token (one-hot drafter)
  2 acceptance ratio uses the original target instead of the current residual
  3 depth-first order visits children in decreasing id order
  4 mask drops the node itself (strict ancestors only)
  5 attention scale 1/d instead of 1/sqrt(d)
  6 argmax ties go to the highest token id
  7 greedy walk stops after the first accepted child
  8 inverse CDF returns the next token id
  9 residual without the max(0, .) clamp
 11 merge unifies equal tokens regardless of their prefix
 12 temperature multiplies the logits instead of dividing
 13 expansion gives depth-2 nodes one child too many
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
PINS = [os.path.join(HERE, f) for f in ("test_oracle_tree.py", "test_oracle_attention.py", "test_oracle_verify.py")]


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 6, 7, 8, 9, 11, 12, 13])
def test_planted_mistake_is_caught(k, tmp_path):
    so = oracle.build_mutant(k, str(tmp_path / f"liboracle_m{k}.so"))
    env = dict(os.environ, TREESPEC_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"mutant {k} survived the pins:\n{r.stdout[-2000:]}"
