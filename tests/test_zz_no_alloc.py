"""tree_attention_noalloc: tree attention for callers that cannot allocate
device memory (plugin or callback code inside a host framework that owns all
device allocations, serving loops that must not allocate once warm). It takes
no workspace; the library's built-in scratch array holds the split-KV partials.

Called through the C ABI and compared with tree_attention given a caller
workspace, on two calls in a row with different inputs (the scratch keeps the
previous call's contents, which must not leak into the next result). This file
is collected last on purpose."""
import ctypes as C

import numpy as np
import pytest
import torch

from tree_speculative_verification_gb300 import api
from tree_speculative_verification_gb300.step import to_device
from tree_speculative_verification_gb300.workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def _inputs(rng, B, H, d, n, L_max):
    draw = lambda *s: torch.from_numpy(f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32)).view(np.int16)
                                       ).cuda().view(torch.bfloat16)
    q, kn, vn = draw(B, n, H, d), draw(B, n, H, d), draw(B, n, H, d)
    kc, vc = draw(B, H, L_max, d), draw(B, H, L_max, d)
    return q, kn, vn, kc, vc


# (widths, kernel): the LLaMA-7B-shaped expansion tree (21 nodes) on few heads
# with the mma.sync kernel, which then splits the key axis so that its partials
# really go to the scratch; the OPT-30B-shaped (47 nodes) and the 21-node tree
# with the persistent tcgen05 kernel, which keeps its item queue in the scratch
CASES = [((1, 1, 3, 1, 1, 1, 1, 1), "k_attn_bf16<"), ((2, 2, 2, 2, 1), "k_attn_tq"), ((1, 1, 3, 1, 1, 1, 1, 1), "k_attn_tq")]


@pytest.mark.parametrize("widths,kernel", CASES)
def test_noalloc_matches_workspace_entry_point_twice(widths, kernel, monkeypatch):
    """Same kernel, same plan, same inputs: the outputs must be bit-identical to
    tree_attention with a caller workspace, on two calls in a row (the second
    call must not see what the first left in the scratch)."""
    for var in ("TREESPEC_ATTN_KERNEL", "TREESPEC_ATTN_SPLITS"):
        monkeypatch.delenv(var, raising=False)
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", "mma" if kernel.startswith("k_attn_bf16") else "tq")
    lib = api.load_library()
    B, H, d, L_max = 2, 4, 128, 1600
    n = 1
    level = 1
    for k in widths:
        level *= k
        n += level
    assert api.attention_kernel(B, H, n, d, L_max, api.TS_BF16).startswith(kernel)
    need = api.workspace_size(api.TS_OP_ATTENTION, B, H, n, d, L_max, 1)
    assert 0 < need <= api.NOALLOC_SCRATCH_BYTES
    rng = np.random.default_rng(2024 + n)
    t = api.Tree(B, n)
    api.tree_build(t, torch.zeros((B, n), dtype=torch.int32, device="cuda"), widths=widths)
    ws = api.workspace(api.TS_OP_ATTENTION, B, H, n, d, L_max, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, prefix in enumerate(([1500, 1200], [900, 1577 - n])):
        q, kn, vn, kc, vc = _inputs(rng, B, H, d, n, L_max)
        pl = to_device(np.array(prefix, np.int32), "cuda")
        api.kv_append(kc, vc, kn, vn, pl, t)
        ref = torch.zeros_like(q)
        api.tree_attention(ref, q, kc, vc, pl, t, 0.0, ws, status)
        out = torch.full_like(q, float("nan"))
        rc = lib.tree_attention_noalloc(C.c_void_p(out.data_ptr()), C.c_void_p(q.data_ptr()),
                                        C.c_void_p(kc.data_ptr()), C.c_void_p(vc.data_ptr()),
                                        C.c_void_p(pl.data_ptr()), t.c, H, d, L_max, api.TS_BF16, 0.0,
                                        C.c_void_p(status.data_ptr()), stream)
        assert rc == api.TS_OK, lib.treespec_last_error()
        torch.cuda.synchronize()
        assert status.item() == 0
        assert torch.isfinite(out.float()).all(), f"call {call}"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}"


def test_noalloc_rejects_sizes_beyond_the_scratch():
    lib = api.load_library()
    B, H, d, n, L_max = 2, 2, 128, 256, 65536      # few heads, long keys, big tree: many key splits
    need = api.workspace_size(api.TS_OP_ATTENTION, B, H, n, d, L_max, 1)
    assert need > api.NOALLOC_SCRATCH_BYTES
    t = api.Tree(B, n)
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")     # never touched: the call is refused first
    p = C.c_void_p(x.data_ptr())
    rc = lib.tree_attention_noalloc(p, p, p, p, p, t.c, H, d, L_max, api.TS_BF16, 0.0, None,
                                    C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == api.TS_ERR_INVALID_ARG
    assert b"scratch" in lib.treespec_last_error()
