"""The sequence-based baseline (SpecInfer Fig. 4 left: one sequence and one KV
copy per root-to-leaf path) against the oracle and the tree kernel: every
chain's output must equal the oracle's fp64 causal attention of that chain
(2e-2), and since TreeAttention(u) is the causal attention of u's path at u
(Def. 4.1), every path position must reproduce the tree output of its node
(both bf16 results of fp32 accumulation in different kernels: 2e-2)."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verification_gb300 import workloads as wl
from tree_speculative_verification_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,sd", [("llama7b", 1), ("long65b", 16), ("opt30b", 16)])
def test_sequences_reproduce_tree_attention(name, sd):
    """Full llama7b layer; the 128-node random tree (64 paths) and the OPT-30B
    expansion tree at a 1024-key prefix, which keeps the 64 prefix copies near 2 GB."""
    w = wl.make(name, scale_down=sd)
    tree = DeviceStep(w)
    tree.build(); tree.append(); tree.attend()
    seq_w, path_nodes = wl.sequence_batch(w)
    seq = DeviceStep(seq_w)
    seq.build(); seq.append(); seq.attend()
    torch.cuda.synchronize()
    assert tree.status.item() == 0 and seq.status.item() == 0
    t_out = tree.out.float().cpu().numpy()     # [B][n_max][H][d]
    s_out = seq.out.float().cpu().numpy()      # [paths][len][H][d]
    rows = oracle.all_rows(seq_w.B, seq_w.H, seq_w.n_nodes)
    ref = oracle.tree_attention_rows(seq_w.q, seq_w.k_new, seq_w.v_new, seq_w.k_cache, seq_w.v_cache,
                                     seq_w.prefix_len, seq_w.n_nodes, seq_w.parent, rows)
    err_o = float(np.max(np.abs(s_out[rows[:, 0], rows[:, 2], rows[:, 1]] - ref)))
    print(f"[{name}] {seq_w.B} chains, max-abs error against the oracle {err_o:.4g}")
    assert err_o <= 2e-2, err_o
    S, L = path_nodes.shape[:2]
    err = 0.0
    for s in range(S):
        for i in range(L):
            b, v = path_nodes[s, i]
            if b < 0:
                break
            err = max(err, float(np.abs(s_out[s, i] - t_out[b, v]).max()))
    assert err <= 2e-2, err
