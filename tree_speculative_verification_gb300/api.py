"""Python binding of libtreespec (the C ABI declared in include/treespec.h).

Argument marshalling only: every function here checks shapes/dtypes of torch
tensors, passes raw device pointers and the current CUDA stream to the
function of the same name in libtreespec.so, and raises TreespecError when it
returns an error. All computation happens in the library's CUDA kernels; there
is no CPU fallback -- without the built library every call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtreespec.so")

TS_OK, TS_ERR_INVALID_ARG, TS_ERR_CUDA, TS_ERR_UNSUPPORTED = 0, 1, 2, 3
TS_F32, TS_BF16 = 0, 1
TS_OP_ATTENTION, TS_OP_VERIFY_GREEDY, TS_OP_VERIFY_MSS = 0, 1, 2
STATUS_BAD_TREE, STATUS_NONFINITE, STATUS_ZERO_RESID, STATUS_INDEX, STATUS_TIMEOUT = 1, 2, 4, 8, 16
MAX_NODES = 256
PAGE_KEYS = 64   # TS_PAGE_KEYS

#: every entry point of the C ABI (include/treespec.h)
EXPORTS = ("tree_build", "tree_build_chains", "kv_append", "tree_attention", "verify_greedy", "verify_mss",
           "kv_commit", "treespec_workspace_size", "treespec_workspace_init", "treespec_last_error",
           "treespec_version", "tree_attention_noalloc", "treespec_attention_kernel", "verify_naive",
           "tree_expand_topk", "kv_append_paged", "tree_attention_paged", "kv_commit_paged", "tree_build_append",
           "tree_attention_append")
#: bytes of the scratch array compiled into the library (TS_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 8 << 20


class TreespecError(RuntimeError):
    pass


class ts_tree(C.Structure):
    _fields_ = [("B", C.c_int32), ("n_max", C.c_int32)] + [
        (name, C.c_void_p) for name in ("n_nodes", "perm", "dfs_of", "parent", "token", "depth", "pos", "sub_end",
                                        "anc")]


class ts_paged_kv(C.Structure):
    _fields_ = [("k_pages", C.c_void_p), ("v_pages", C.c_void_p), ("block_table", C.c_void_p),
                ("num_pages", C.c_int32), ("max_pages", C.c_int32)]


_lib = None


def load_library(path: str | None = None):
    """Load libtreespec.so (built by tree_speculative_verification_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise TreespecError(f"{path} is missing: build the CUDA library first "
                            "(python -m tree_speculative_verification_gb300.build)")
    lib = C.CDLL(path)
    P, I, F, Z = C.c_void_p, C.c_int, C.c_float, C.c_size_t
    T = C.POINTER(ts_tree)
    sig = {
        "tree_build": [T, P, P, P, P, I, P, P, P],
        "tree_build_chains": [T, P, P, I, I, P, P, P, P, P, P],
        "kv_append": [P, P, P, P, P, T, I, I, I, I, P, P],
        "tree_build_append": [T, P, P, I, P, P, P, P, P, I, I, I, I, P, P],
        "tree_attention": [P, P, P, P, P, T, I, I, I, I, F, P, Z, P, P],
        "tree_attention_append": [P, P, P, P, P, P, P, T, I, I, I, I, F, P, Z, P, P],
        "verify_greedy": [P, P, P, P, P, T, I, P, Z, P, P],
        "verify_mss": [P, P, P, P, P, P, I, P, P, I, P, F, T, I, P, P],
        "verify_naive": [P, P, P, P, P, P, I, P, F, T, I, P, P],
        "tree_expand_topk": [P, P, P, I, I, I, P, I, I, P, P],
        "kv_append_paged": [C.POINTER(ts_paged_kv), P, P, P, T, I, I, P, P],
        "tree_attention_paged": [P, P, C.POINTER(ts_paged_kv), P, T, I, I, F, P, Z, P, P],
        "kv_commit_paged": [C.POINTER(ts_paged_kv), P, P, P, P, T, I, I, P, P],
        "kv_commit": [P, P, P, P, P, P, T, I, I, I, I, P, P],
        "treespec_workspace_init": [P, Z, P],
        "tree_attention_noalloc": [P, P, P, P, P, T, I, I, I, I, F, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = C.c_int
    lib.treespec_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.treespec_workspace_size.restype = C.c_size_t
    lib.treespec_attention_kernel.argtypes = [I, I, I, I, I, I]
    lib.treespec_attention_kernel.restype = C.c_char_p
    lib.treespec_last_error.restype = C.c_char_p
    lib.treespec_version.restype = C.c_char_p
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != TS_OK:
        msg = load_library().treespec_last_error().decode()
        raise TreespecError(f"{what} failed ({rc}): {msg}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise TreespecError("tensors passed to the library must live on a CUDA device")
    if not t.is_contiguous():
        raise TreespecError("tensors passed to the library must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _i32(t, name):
    if t is not None and t.dtype != torch.int32:
        raise TreespecError(f"{name} must be int32")
    return t


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return TS_BF16
    if t.dtype == torch.float32:
        return TS_F32
    raise TreespecError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


class Tree:
    """Device arrays of a linearised tree batch (the ts_tree of the C ABI)."""

    def __init__(self, B: int, n_max: int, device="cuda"):
        if not 1 <= n_max <= MAX_NODES:
            raise TreespecError(f"n_max={n_max} outside [1, {MAX_NODES}]")
        self.B, self.n_max = B, n_max
        W = (n_max + 31) // 32
        z = lambda *s: torch.full(s, -1, dtype=torch.int32, device=device)
        self.n_nodes = torch.zeros(B, dtype=torch.int32, device=device)
        self.perm, self.dfs_of, self.parent, self.token = z(B, n_max), z(B, n_max), z(B, n_max), z(B, n_max)
        self.depth, self.pos, self.sub_end = z(B, n_max), z(B, n_max), z(B, n_max)
        self.anc = torch.zeros(B, n_max, W, dtype=torch.int32, device=device)   # uint32 bit patterns
        self._c = ts_tree(B, n_max, *[t.data_ptr() for t in (self.n_nodes, self.perm, self.dfs_of, self.parent,
                                                              self.token, self.depth, self.pos, self.sub_end,
                                                              self.anc)])

    @property
    def c(self):
        return C.byref(self._c)


def tree_build(tree: Tree, tokens, parent=None, n_nodes=None, widths=None, prefix_len=None, status=None,
               stream=None):
    lib = load_library()
    w_arr, m = None, 0
    if widths is not None:
        m = len(widths)
        w_arr = (C.c_int32 * max(1, m))(*[int(k) for k in widths])
    _check(lib.tree_build(tree.c, _ptr(_i32(tokens, "tokens")), _ptr(_i32(parent, "parent")),
                          _ptr(_i32(n_nodes, "n_nodes")), w_arr, m, _ptr(_i32(prefix_len, "prefix_len")),
                          _ptr(status), _stream(stream)), "tree_build")


def tree_build_append(tree: Tree, tokens, widths, prefix_len, k_cache, v_cache, k_new, v_new, status=None,
                      stream=None):
    """tree_build (widths mode) and kv_append in one launch (dense cache)."""
    lib = load_library()
    m = len(widths)
    w_arr = (C.c_int32 * max(1, m))(*[int(k) for k in widths])
    B, H, L_max, d = k_cache.shape
    _check(lib.tree_build_append(tree.c, _ptr(_i32(tokens, "tokens")), w_arr, m, _ptr(_i32(prefix_len, "prefix_len")),
                                 _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), H, d, L_max,
                                 _dtype(k_cache), _ptr(status), _stream(stream)), "tree_build_append")


def tree_build_chains(tree: Tree, root_token, chains, tokens_out=None, p_row=None, q_row=None, prefix_len=None,
                      status=None, stream=None):
    lib = load_library()
    Cn, ln = chains.shape[1], chains.shape[2]
    _check(lib.tree_build_chains(tree.c, _ptr(_i32(root_token, "root_token")), _ptr(_i32(chains, "chains")), Cn, ln,
                                 _ptr(_i32(tokens_out, "tokens_out")), _ptr(_i32(p_row, "p_row")),
                                 _ptr(_i32(q_row, "q_row")), _ptr(_i32(prefix_len, "prefix_len")), _ptr(status),
                                 _stream(stream)), "tree_build_chains")


def tree_expand_topk(tokens, root_token, ssm_probs, widths, status=None, stream=None):
    """Draft the expansion tree <widths> from drafter rows into tokens [B][n_max]."""
    lib = load_library()
    B, n_max = tokens.shape
    NQ, V = ssm_probs.shape[1], ssm_probs.shape[2]
    m = len(widths)
    w_arr = (C.c_int32 * max(1, m))(*[int(k) for k in widths])
    _check(lib.tree_expand_topk(_ptr(_i32(tokens, "tokens")), _ptr(_i32(root_token, "root_token")), _ptr(ssm_probs),
                                NQ, B, n_max, w_arr, m, V, _ptr(status), _stream(stream)), "tree_expand_topk")


def kv_append(k_cache, v_cache, k_new, v_new, prefix_len, tree: Tree, status=None, stream=None):
    lib = load_library()
    B, H, L_max, d = k_cache.shape
    _check(lib.kv_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(_i32(prefix_len, "prefix_len")),
                         tree.c, H, d, L_max, _dtype(k_cache), _ptr(status), _stream(stream)), "kv_append")


def workspace_size(op: int, B: int, H: int, n_max: int, d: int, L_max: int, V: int) -> int:
    return int(load_library().treespec_workspace_size(op, B, H, n_max, d, L_max, V))


def attention_kernel(B: int, H: int, n_max: int, d: int, L_max: int, dtype: int) -> str:
    """Name of the kernel tree_attention launches for these sizes ("" if rejected)."""
    return load_library().treespec_attention_kernel(B, H, n_max, d, L_max, dtype).decode()


def workspace(op: int, B: int, H: int = 1, n_max: int = 1, d: int = 128, L_max: int = 1, V: int = 1,
              device="cuda"):
    """A zero-filled workspace of the size the op needs (at least 256 bytes)."""
    return torch.zeros(max(256, workspace_size(op, B, H, n_max, d, L_max, V)), dtype=torch.uint8, device=device)


def tree_attention(out, q, k_cache, v_cache, prefix_len, tree: Tree, scale: float = 0.0, ws=None, status=None,
                   stream=None):
    lib = load_library()
    B, H, L_max, d = k_cache.shape
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.tree_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(_i32(prefix_len, "prefix_len")),
                              tree.c, H, d, L_max, _dtype(k_cache), float(scale), _ptr(ws), nbytes, _ptr(status),
                              _stream(stream)), "tree_attention")


def tree_attention_append(out, q, k_cache, v_cache, k_new, v_new, prefix_len, tree: Tree, scale: float = 0.0,
                          ws=None, status=None, stream=None):
    """kv_append and tree_attention in one call (one launch with the persistent
    tcgen05 kernel, else the two launches)."""
    lib = load_library()
    B, H, L_max, d = k_cache.shape
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.tree_attention_append(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                     _ptr(_i32(prefix_len, "prefix_len")), tree.c, H, d, L_max, _dtype(k_cache),
                                     float(scale), _ptr(ws), nbytes, _ptr(status), _stream(stream)),
           "tree_attention_append")


def tree_attention_noalloc(out, q, k_cache, v_cache, prefix_len, tree: Tree, scale: float = 0.0, status=None,
                           stream=None):
    """tree_attention without a workspace argument, for callers that cannot
    allocate device memory: the library's built-in scratch array (shared by all
    calls on a device; calls must not overlap on the GPU) holds the partials."""
    lib = load_library()
    B, H, L_max, d = k_cache.shape
    _check(lib.tree_attention_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(_i32(prefix_len, "prefix_len")), tree.c, H, d, L_max, _dtype(k_cache),
                                      float(scale), _ptr(status), _stream(stream)), "tree_attention_noalloc")


def verify_greedy(out_tokens, out_path, out_count, logits, tree: Tree, argmax_out=None, ws=None, status=None,
                  stream=None):
    lib = load_library()
    V = logits.shape[-1]
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.verify_greedy(_ptr(out_tokens), _ptr(out_path), _ptr(out_count), _ptr(argmax_out), _ptr(logits),
                             tree.c, V, _ptr(ws), nbytes, _ptr(status), _stream(stream)), "verify_greedy")


def verify_mss(out_tokens, out_path, out_count, target_logits, ssm_probs, q_row, uniforms, temperature, tree: Tree,
               p_row=None, status=None, stream=None, lowmargin=None):
    """lowmargin: optional int32 [B], the number of decisions per request taken
    with a margin below 1e-6."""
    lib = load_library()
    NP, V = target_logits.shape[1], target_logits.shape[2]
    NQ = ssm_probs.shape[1]
    _check(lib.verify_mss(_ptr(out_tokens), _ptr(out_path), _ptr(out_count), _ptr(_i32(lowmargin, "lowmargin")),
                          _ptr(target_logits),
                          _ptr(_i32(p_row, "p_row")), NP, _ptr(ssm_probs), _ptr(_i32(q_row, "q_row")), NQ,
                          _ptr(uniforms), float(temperature), tree.c, V, _ptr(status), _stream(stream)), "verify_mss")


def verify_naive(out_tokens, out_path, out_count, target_logits, uniforms, temperature, tree: Tree, p_row=None,
                 status=None, stream=None, lowmargin=None):
    lib = load_library()
    NP, V = target_logits.shape[1], target_logits.shape[2]
    _check(lib.verify_naive(_ptr(out_tokens), _ptr(out_path), _ptr(out_count), _ptr(_i32(lowmargin, "lowmargin")),
                            _ptr(target_logits),
                            _ptr(_i32(p_row, "p_row")), NP, _ptr(uniforms), float(temperature), tree.c, V,
                            _ptr(status), _stream(stream)), "verify_naive")


def kv_commit(k_cache, v_cache, prefix_len, new_prefix_len, out_path, out_count, tree: Tree, status=None,
              stream=None):
    lib = load_library()
    B, H, L_max, d = k_cache.shape
    _check(lib.kv_commit(_ptr(k_cache), _ptr(v_cache), _ptr(_i32(prefix_len, "prefix_len")),
                         _ptr(_i32(new_prefix_len, "new_prefix_len")), _ptr(out_path), _ptr(out_count), tree.c, H, d,
                         L_max, _dtype(k_cache), _ptr(status), _stream(stream)), "kv_commit")


class PagedKV:
    """A paged KV cache (the ts_paged_kv of the C ABI): k_pages / v_pages
    [num_pages][H][PAGE_KEYS][d] bf16 and block_table [B][max_pages] int32."""

    def __init__(self, k_pages, v_pages, block_table):
        if k_pages.dtype != torch.bfloat16 or v_pages.shape != k_pages.shape:
            raise TreespecError("pages must be two bf16 tensors of one shape [num_pages][H][64][d]")
        if k_pages.shape[2] != PAGE_KEYS:
            raise TreespecError(f"a page holds {PAGE_KEYS} keys")
        self.k_pages, self.v_pages, self.block_table = k_pages, v_pages, _i32(block_table, "block_table")
        self.H, self.d = k_pages.shape[1], k_pages.shape[3]
        self._c = ts_paged_kv(k_pages.data_ptr(), v_pages.data_ptr(), block_table.data_ptr(), k_pages.shape[0],
                              block_table.shape[1])

    @property
    def c(self):
        return C.byref(self._c)

    @property
    def L_max(self) -> int:
        return self.block_table.shape[1] * PAGE_KEYS


def kv_append_paged(kv: PagedKV, k_new, v_new, prefix_len, tree: Tree, status=None, stream=None):
    _check(load_library().kv_append_paged(kv.c, _ptr(k_new), _ptr(v_new), _ptr(_i32(prefix_len, "prefix_len")), tree.c,
                                          kv.H, kv.d, _ptr(status), _stream(stream)), "kv_append_paged")


def tree_attention_paged(out, q, kv: PagedKV, prefix_len, tree: Tree, scale=0.0, ws=None, status=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load_library().tree_attention_paged(_ptr(out), _ptr(q), kv.c, _ptr(_i32(prefix_len, "prefix_len")), tree.c,
                                               kv.H, kv.d, float(scale), _ptr(ws), nbytes, _ptr(status),
                                               _stream(stream)), "tree_attention_paged")


def kv_commit_paged(kv: PagedKV, prefix_len, new_prefix_len, out_path, out_count, tree: Tree, status=None,
                    stream=None):
    _check(load_library().kv_commit_paged(kv.c, _ptr(_i32(prefix_len, "prefix_len")),
                                          _ptr(_i32(new_prefix_len, "new_prefix_len")), _ptr(out_path),
                                          _ptr(out_count), tree.c, kv.H, kv.d, _ptr(status), _stream(stream)),
           "kv_commit_paged")


def version() -> str:
    return load_library().treespec_version().decode()
