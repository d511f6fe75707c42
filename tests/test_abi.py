"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
function that include/treespec.h declares, and rejects bad arguments on the
host before anything is launched."""
import ctypes as C
import os
import re

import pytest

from tree_speculative_verification_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treespec.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert set(api.EXPORTS) == set(names), names
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert "sm_103a" in api.version()


def _tree(B=2, n_max=8):
    fake = 0x10000    # never dereferenced: every call below fails validation first
    return api.ts_tree(B, n_max, *([fake] * 9))


def test_null_tree_rejected(lib):
    rc = lib.tree_build(None, None, None, None, None, 0, None, None, None)
    assert rc == api.TS_ERR_INVALID_ARG
    assert b"tree" in lib.treespec_last_error()


@pytest.mark.parametrize("n_max", [0, 257])
def test_tree_size_limits(lib, n_max):
    t = _tree(n_max=n_max)
    rc = lib.tree_build(C.byref(t), C.c_void_p(0x10000), C.c_void_p(0x10000), C.c_void_p(0x10000), None, 0, None,
                        None, None)
    assert rc == api.TS_ERR_INVALID_ARG


def test_expansion_larger_than_n_max(lib):
    t = _tree(n_max=10)
    w = (C.c_int32 * 3)(2, 2, 1)     # 11 nodes
    rc = lib.tree_build(C.byref(t), C.c_void_p(0x10000), None, None, w, 3, None, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"n_max" in lib.treespec_last_error()


def test_unsupported_head_dim(lib):
    t = _tree()
    p = C.c_void_p(0x10000)
    rc = lib.tree_attention(p, p, p, p, p, C.byref(t), 4, 96, 64, api.TS_BF16, 0.0, p, 1 << 20, None, None)
    assert rc == api.TS_ERR_UNSUPPORTED


def test_misaligned_cache(lib):
    t = _tree()
    p, bad = C.c_void_p(0x10000), C.c_void_p(0x10008)
    rc = lib.tree_attention(p, p, bad, p, p, C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, p, 1 << 20, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"aligned" in lib.treespec_last_error()


def test_workspace_too_small(lib):
    t = _tree()
    p = C.c_void_p(0x10000)
    rc = lib.tree_attention(p, p, p, p, p, C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, p, 0, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"workspace" in lib.treespec_last_error()


def test_mss_bad_temperature(lib):
    t = _tree()
    p = C.c_void_p(0x10000)
    rc = lib.verify_mss(p, p, p, None, p, None, 8, p, p, 1, p, 0.0, C.byref(t), 16, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"temperature" in lib.treespec_last_error()


def test_commit_alias_rejected(lib):
    t = _tree()
    p = C.c_void_p(0x10000)
    rc = lib.kv_commit(p, p, p, p, p, p, C.byref(t), 2, 128, 64, api.TS_BF16, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"alias" in lib.treespec_last_error()


def test_chains_too_many_nodes(lib):
    t = _tree(n_max=24)
    p = C.c_void_p(0x10000)
    rc = lib.tree_build_chains(C.byref(t), p, p, 3, 8, None, None, None, None, None, None)
    assert rc == api.TS_ERR_INVALID_ARG


def test_workspace_sizes(lib):
    assert api.workspace_size(api.TS_OP_ATTENTION, 8, 32, 21, 128, 2112, 32000) > 0
    assert api.workspace_size(api.TS_OP_VERIFY_GREEDY, 8, 1, 21, 128, 1, 32000) >= 8 * 21 * 8
    assert api.workspace_size(api.TS_OP_VERIFY_MSS, 8, 1, 21, 128, 1, 32000) == 0
    assert api.workspace_size(api.TS_OP_ATTENTION, 8, 32, 300, 128, 2112, 32000) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    saved = api._lib
    try:
        api._lib = None
        with pytest.raises(api.TreespecError):
            api.load_library(str(tmp_path / "missing.so"))
    finally:
        api._lib = saved


@pytest.mark.parametrize("n_max,d,expect", [
    (21, 128, "k_attn_bf16<"),      # the LLaMA-7B-shaped expansion tree: mma.sync
    (32, 128, "k_attn_bf16<"),
    (33, 128, "k_attn_tq"),         # 33..128 nodes: persistent tcgen05, 128-key tiles
    (47, 128, "k_attn_tq"),
    (128, 128, "k_attn_tq"),
    (129, 128, "k_attn_bf16<"),
    (47, 64, "k_attn_bf16<"),       # head_dim 64: mma.sync only
])
def test_kernel_choice(lib, n_max, d, expect, monkeypatch):
    """attn_plan's default choice is host logic: the same without a GPU."""
    for var in ("TREESPEC_ATTN_KERNEL", "TREESPEC_ATTN_SPLITS"):
        monkeypatch.delenv(var, raising=False)
    name = api.attention_kernel(8, 32, n_max, d, 2048 + n_max, api.TS_BF16)
    assert name.startswith(expect), name
    assert api.attention_kernel(8, 32, n_max, d, 2048 + n_max, api.TS_F32) == "k_attn_f32"


@pytest.mark.parametrize("B,expect", [(1, "k_attn_tq"), (4, "k_attn_tq"), (5, "k_attn_bf16<"), (8, "k_attn_bf16<"),
                                      (9, "k_attn_bf16<"), (10, "k_attn_tq"), (16, "k_attn_tq")])
def test_kernel_choice_small_trees_by_batch(lib, B, expect, monkeypatch):
    """Trees of up to 32 nodes at head_dim 128 (32 heads, 152 SMs when no GPU
    is present): the mma.sync kernel only when the (request, head) pairs fill
    one wave of its two CTAs per SM, 152 < B*H <= 304."""
    for var in ("TREESPEC_ATTN_KERNEL", "TREESPEC_ATTN_SPLITS"):
        monkeypatch.delenv(var, raising=False)
    assert api.attention_kernel(B, 32, 21, 128, 2048 + 21, api.TS_BF16).startswith(expect)


@pytest.mark.parametrize("force,n_max,expect", [("mma", 47, "k_attn_bf16<"), ("tq", 21, "k_attn_tq"),
                                                 ("mma", 21, "k_attn_bf16<")])
def test_kernel_override(lib, force, n_max, expect, monkeypatch):
    monkeypatch.setenv("TREESPEC_ATTN_KERNEL", force)
    assert api.attention_kernel(8, 32, n_max, 128, 2048 + n_max, api.TS_BF16).startswith(expect)


def test_build_append_rejects_before_launch(lib):
    """tree_build_append checks like tree_build (widths) and kv_append together."""
    t = _tree(n_max=10)
    p, bad = C.c_void_p(0x10000), C.c_void_p(0x10008)
    w = (C.c_int32 * 3)(2, 2, 1)     # 11 nodes > n_max
    rc = lib.tree_build_append(C.byref(t), p, w, 3, p, p, p, p, p, 2, 128, 64, api.TS_BF16, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"n_max" in lib.treespec_last_error()
    w2 = (C.c_int32 * 2)(2, 2)       # 7 nodes
    rc = lib.tree_build_append(C.byref(t), p, w2, 2, p, p, bad, p, p, 2, 128, 64, api.TS_BF16, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"aligned" in lib.treespec_last_error()
    rc = lib.tree_build_append(C.byref(t), p, w2, 2, None, p, p, p, p, 2, 128, 64, api.TS_BF16, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"NULL" in lib.treespec_last_error()


def test_noalloc_rejects_before_touching_the_device(lib):
    """tree_attention_noalloc runs every check of tree_attention before it looks
    up or clears its scratch: with no GPU here, any device call would return
    TS_ERR_CUDA, so an argument error coming back as TS_ERR_INVALID_ARG (or
    TS_ERR_UNSUPPORTED) shows that nothing was enqueued."""
    t = _tree()
    p, bad = C.c_void_p(0x10000), C.c_void_p(0x10008)
    rc = lib.tree_attention_noalloc(None, p, p, p, p, C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"NULL" in lib.treespec_last_error()
    rc = lib.tree_attention_noalloc(p, p, bad, p, p, C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"aligned" in lib.treespec_last_error()
    rc = lib.tree_attention_noalloc(p, p, p, p, None, C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, None, None)
    assert rc == api.TS_ERR_INVALID_ARG
    rc = lib.tree_attention_noalloc(p, p, p, p, p, C.byref(t), 4, 96, 64, api.TS_BF16, 0.0, None, None)
    assert rc == api.TS_ERR_UNSUPPORTED
    rc = lib.tree_attention_noalloc(p, p, p, p, p, None, 4, 128, 64, api.TS_BF16, 0.0, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"tree" in lib.treespec_last_error()


def test_attention_append_rejects_before_touching_the_device(lib):
    """tree_attention_append runs the checks of tree_attention and of kv_append
    (new K/V present and 16-byte aligned, the workspace) before anything is
    enqueued: with no GPU here a device call would come back as TS_ERR_CUDA."""
    t = _tree()
    p, bad = C.c_void_p(0x10000), C.c_void_p(0x10008)
    ws = C.c_void_p(0x20000)
    args = lambda **kw: [kw.get(k, p) for k in ("out", "q", "kc", "vc", "kn", "vn", "pl")]
    rc = lib.tree_attention_append(*args(kn=None), C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, ws, 1 << 20, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"NULL" in lib.treespec_last_error()
    rc = lib.tree_attention_append(*args(vn=bad), C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, ws, 1 << 20, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"aligned" in lib.treespec_last_error()
    rc = lib.tree_attention_append(*args(kc=bad), C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, ws, 1 << 20, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"aligned" in lib.treespec_last_error()
    rc = lib.tree_attention_append(*args(), C.byref(t), 4, 128, 64, api.TS_BF16, 0.0, ws, 16, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"workspace" in lib.treespec_last_error()
    rc = lib.tree_attention_append(*args(), C.byref(t), 4, 96, 64, api.TS_BF16, 0.0, ws, 1 << 20, None, None)
    assert rc == api.TS_ERR_UNSUPPORTED
    rc = lib.tree_attention_append(*args(), None, 4, 128, 64, api.TS_BF16, 0.0, ws, 1 << 20, None, None)
    assert rc == api.TS_ERR_INVALID_ARG and b"tree" in lib.treespec_last_error()


@pytest.mark.parametrize("B,H,n_max", [(32768, 128, 33), (8, 32, 64), (64, 56, 47)])
def test_persistent_kernel_workspace_is_its_queue(lib, B, H, n_max, monkeypatch):
    """The persistent tcgen05 plan keeps only its item queue in the workspace,
    whatever the batch (no per-(request, head) counters), so the scratch-free
    entry point's clear stays inside the plan's bytes even at B*H > 2^21."""
    monkeypatch.delenv("TREESPEC_ATTN_KERNEL", raising=False)
    assert api.attention_kernel(B, H, n_max, 128, 64 + n_max, api.TS_BF16) == "k_attn_tq"
    assert api.workspace_size(api.TS_OP_ATTENTION, B, H, n_max, 128, 64 + n_max, 1) == 256
