"""Longest-first dispatch of the attention CTAs (grid row r takes the request
with the r-th largest key count): only the order in which (request, head)
pairs are scheduled changes, so the output must be bit-identical to request
order, with and without key splits; the persistent tcgen05 kernel takes its
items from a queue and must not depend on the switch."""
import numpy as np
import pytest
import torch

from tree_speculative_verification_gb300 import workloads as wl
from tree_speculative_verification_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu


def _attend(w, monkeypatch, lpt):
    monkeypatch.setenv("TREESPEC_ATTN_LPT", "1" if lpt else "0")
    s = DeviceStep(w)
    s.build(); s.append(); s.attend()
    torch.cuda.synchronize()
    assert s.status.item() == 0
    return s.out.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("kernel,splits", [("mma", ""), ("mma", "3"), ("tq", "")])
def test_longest_first_is_bit_identical(kernel, splits, monkeypatch):
    """Merge-based trees over ragged prefixes U[512, 4096] (batch 16)."""
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", kernel)
    if splits:
        monkeypatch.setenv("TREESPEC_ATTN_SPLITS", splits)
    w = wl.make("merge")
    assert len(set(int(p) for p in w.prefix_len)) > 1
    a = _attend(w, monkeypatch, True)
    b = _attend(w, monkeypatch, False)
    assert np.array_equal(a, b)
