"""Several verification steps in a row on the GPU, each committed into the
shared KV cache that the next step attends (SpecInfer sec. 4.2: the tree's
K/V sit after the verified prefix; after verification only the accepted path
keeps its entries and the verified length grows by the accepted count + 1).
The oracle replays the same steps on a host copy of the cache: attention
outputs within 2e-2, accepted tokens and the committed cache bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import to_device
from tree_speculative_verification_gb300.workloads import bf16_bits_to_f32, f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", ["greedy", "mss"])
def test_step_loop_commits_feed_the_next_step(kind):
    rng = np.random.default_rng(2025 if kind == "greedy" else 2026)
    B, H, d, V, widths = 2, 4, 128, 512, (2, 2, 1)
    par1 = oracle.widths_parent(widths)
    n = len(par1)
    steps, P0 = 4, 90
    L_max = P0 + steps * (n + 1) + n
    parent = np.tile(par1, (B, 1))
    kc = np.zeros((B, H, L_max, d), np.uint16)
    vc = np.zeros((B, H, L_max, d), np.uint16)
    kc[:, :, :P0] = f32_to_bf16_bits(rng.standard_normal((B, H, P0, d)).astype(np.float32))
    vc[:, :, :P0] = f32_to_bf16_bits(rng.standard_normal((B, H, P0, d)).astype(np.float32))
    dkc, dvc = to_device(kc, "cuda", True), to_device(vc, "cuda", True)
    prefix = np.full(B, P0, np.int32)
    t = api.Tree(B, n)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_a = api.workspace(api.TS_OP_ATTENTION, B, H, n, d, L_max, V)
    ws_g = api.workspace(api.TS_OP_VERIFY_GREEDY, B, n_max=n, V=V)
    host_k, host_v = kc.copy(), vc.copy()
    for step in range(steps):
        tok = rng.integers(0, V, (B, n)).astype(np.int32)
        q, kn, vn = (f32_to_bf16_bits(rng.standard_normal((B, n, H, d)).astype(np.float32)) for _ in range(3))
        logits = (rng.standard_normal((B, n, V)) * 2).astype(np.float32)
        for b in range(B):                        # plant the target's choice as first child
            for u in range(n):
                kids = np.nonzero(par1 == u)[0]
                if len(kids) and rng.random() < 0.7:
                    tok[b, kids[0]] = np.argmax(logits[b, u])
        z = logits + rng.standard_normal((B, n, V)).astype(np.float32)
        ssm = np.exp(z - z.max(-1, keepdims=True)).astype(np.float64)
        ssm = (ssm / ssm.sum(-1, keepdims=True)).astype(np.float32)
        q_row = np.where(parent >= 0, parent, 0).astype(np.int32)
        uni = rng.random((B, 2, n)).astype(np.float32)
        # ---- GPU step
        dpl = to_device(prefix, "cuda")
        api.tree_build(t, to_device(tok, "cuda"), widths=widths, prefix_len=dpl, status=st)
        api.kv_append(dkc, dvc, to_device(kn, "cuda", True), to_device(vn, "cuda", True), dpl, t, st)
        out = torch.zeros((B, n, H, d), dtype=torch.bfloat16, device="cuda")
        api.tree_attention(out, to_device(q, "cuda", True), dkc, dvc, dpl, t, 0.0, ws_a, st)
        ot = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
        op = torch.full((B, n + 1), -1, dtype=torch.int32, device="cuda")
        oc = torch.zeros(B, dtype=torch.int32, device="cuda")
        if kind == "greedy":
            api.verify_greedy(ot, op, oc, to_device(logits, "cuda"), t, ws=ws_g, status=st)
        else:
            api.verify_mss(ot, op, oc, to_device(logits, "cuda"), to_device(ssm, "cuda"), to_device(q_row, "cuda"),
                           to_device(uni, "cuda"), 1.0, t, status=st)
        npl = torch.zeros(B, dtype=torch.int32, device="cuda")
        api.kv_commit(dkc, dvc, dpl, npl, op, oc, t, st)
        torch.cuda.synchronize()
        assert st.item() & ~api.STATUS_ZERO_RESID == 0
        # ---- oracle replay on the host cache
        ref_t = oracle.tree_build(parent, tok)
        rows = oracle.all_rows(B, H, np.full(B, n))
        ref_out = oracle.tree_attention_rows(q, kn, vn, host_k, host_v, prefix, np.full(B, n), parent, rows)
        o = out.float().cpu().numpy()
        got = np.stack([o[b, v, h] for b, h, v in rows])
        assert float(np.abs(got - ref_out).max()) <= 2e-2, step
        if kind == "greedy":
            ref = oracle.verify_greedy(logits, parent, tok, np.full(B, n))
            lm = ref["count"]
        else:
            ref = oracle.verify_mss(logits, ssm, q_row, uni, parent, tok, np.full(B, n))
            lm = ref["lm_pos"]
            if (lm < ref["count"]).any():
                pytest.skip("a low-margin MSS decision; the replay would diverge")
        assert oc.cpu().tolist() == ref["count"].tolist(), step
        for b in range(B):
            c = int(ref["count"][b])
            assert ot[b, :c].tolist() == ref["tokens"][b, :c].tolist()
            for v in range(n):                      # append by definition: row P + dfs(v) holds node v
                host_k[b, :, prefix[b] + ref_t["dfs_of"][b, v]] = kn[b, v]
                host_v[b, :, prefix[b] + ref_t["dfs_of"][b, v]] = vn[b, v]
        host_k, host_v, new_prefix = oracle.kv_commit(host_k, host_v, prefix, ref_t["dfs_of"], ref["path"],
                                                      ref["count"])
        assert npl.cpu().tolist() == new_prefix.tolist()
        gk = dkc.view(torch.int16).cpu().numpy().view(np.uint16)
        gv = dvc.view(torch.int16).cpu().numpy().view(np.uint16)
        for b in range(B):                          # the verified region is bit-exact
            assert np.array_equal(gk[b, :, : new_prefix[b]], host_k[b, :, : new_prefix[b]]), step
            assert np.array_equal(gv[b, :, : new_prefix[b]], host_v[b, :, : new_prefix[b]]), step
        prefix = new_prefix.astype(np.int32)
    assert (prefix >= P0 + steps).all()             # every step appends at least one token
