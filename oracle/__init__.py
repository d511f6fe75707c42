"""The oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow fp64 CPU restatement of one tree-based speculative verification
step (SpecInfer, arXiv 2305.09781: Def. 3.1/3.2, Def. 4.1, sec. 4.2 mask,
Algorithm 2), written in C99 (``oracle.c``) and wrapped here with ctypes and
numpy. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import it; the library under
``tree_speculative_verification_gb300`` never does, and the two share no code.

Every function takes numpy arrays and returns numpy arrays. The shared library
is compiled on first use (gcc, OpenMP) next to this file.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OR_OK, OR_BAD_TREE, OR_INDEX, OR_NONFINITE, OR_ZERO_RESID, OR_BAD_ARG = 0, 1, 2, 4, 8, 16


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # TREESPEC_ORACLE_LIB lets the mutation tests load a planted-mistake build
            alt = os.environ.get("TREESPEC_ORACLE_LIB")
            if alt:
                _lib = C.CDLL(alt)
            else:
                build()
                _lib = C.CDLL(_SO)
    return _lib


def build_mutant(k: int, path: str) -> str:
    """Compile the oracle with planted mistake number k (see OR_MUTANT in oracle.c)."""
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", f"-DOR_MUTANT={int(k)}", "-shared", "-fPIC",
                    _SRC, "-o", path, "-lm"], check=True)
    return path


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def num_threads() -> int:
    return int(_load().or_num_threads())


# --------------------------------------------------------------------------- #
# tree layout
# --------------------------------------------------------------------------- #
def widths_parent(widths, n_cap: int = 4096) -> np.ndarray:
    """Level-order parent array of the expansion tree <k1..km> (Fig. 3)."""
    lib = _load()
    w = _i32(widths)
    par = np.full(n_cap, -1, np.int32)
    n = lib.or_widths_parent(C.c_int(len(w)), _p(w), C.c_int(n_cap), _p(par))
    if n < 0:
        raise ValueError("expansion tree larger than n_cap")
    return par[:n].copy()


def topk_expand(widths, root_token, ssm, n_max: int | None = None):
    """Tokens of the expansion tree <k1..km> drafted by top-k (sec. 3, Fig. 3):
    node u's children are the k most probable tokens of ssm[b][u], ties to the
    lower id. Returns (tokens [B][n_max], status bits)."""
    lib = _load()
    w = _i32(widths)
    q = _f32(ssm)
    B, NQ, V = q.shape
    n = len(widths_parent(widths))
    n_max = n if n_max is None else n_max
    rt = _i32(root_token)
    tok = np.full((B, n_max), -1, np.int32)
    st = lib.or_topk_expand(C.c_int(B), C.c_int(n_max), C.c_int(NQ), C.c_int(V), C.c_int(len(w)), _p(w), _p(rt),
                            _p(q), _p(tok))
    return tok, int(st)


def merge_chains(chains, root_token: int, n_cap: int | None = None):
    """Trie merge of C chains of equal length (Def. 3.2).
    Returns (parent, tokens, src) in creation order; src = chain*len + pos."""
    lib = _load()
    ch = _i32(chains)
    Cn, ln = ch.shape
    n_cap = n_cap or 1 + Cn * ln
    par = np.full(n_cap, -1, np.int32)
    tok = np.zeros(n_cap, np.int32)
    src = np.full(n_cap, -1, np.int32)
    n = lib.or_merge_chains(C.c_int(Cn), C.c_int(ln), _p(ch), C.c_int(int(root_token)),
                            C.c_int(n_cap), _p(par), _p(tok), _p(src))
    if n < 0:
        raise ValueError("merged tree larger than n_cap")
    return par[:n].copy(), tok[:n].copy(), src[:n].copy()


def tree_build(parent, tokens=None, n_nodes=None):
    """Batched linearisation. parent: [B][n_max] (or [n]). Returns a dict of
    arrays (perm, dfs_of, parent, token, depth, sub_end: [B][n_max]; anc:
    [B][n_max][n_max] uint8; status: [B])."""
    lib = _load()
    par = _i32(parent)
    squeeze = par.ndim == 1
    if squeeze:
        par = par[None]
    B, n_max = par.shape
    tok = _i32(tokens if tokens is not None else np.zeros_like(par)).reshape(B, n_max)
    nn = _i32(n_nodes if n_nodes is not None else np.full(B, n_max)).reshape(B)
    out = {k: np.full((B, n_max), -1, np.int32) for k in ("perm", "dfs_of", "parent", "token", "depth", "sub_end")}
    anc = np.zeros((B, n_max, n_max), np.uint8)
    st = np.zeros(B, np.int32)
    lib.or_tree_build_batch(C.c_int(B), C.c_int(n_max), _p(nn), _p(par), _p(tok), _p(out["perm"]),
                            _p(out["dfs_of"]), _p(out["parent"]), _p(out["token"]), _p(out["depth"]),
                            _p(out["sub_end"]), _p(anc), _p(st))
    out["anc"] = anc
    out["status"] = st
    if squeeze:
        out = {k: v[0] for k, v in out.items()}
    return out


# --------------------------------------------------------------------------- #
# tree attention
# --------------------------------------------------------------------------- #
def tree_attention_rows(q, k_new, v_new, k_cache, v_cache, prefix_len, n_nodes, parent, rows,
                        scale=None, nthreads: int = 0) -> np.ndarray:
    """fp64 TreeAttention(u) = Attention(S_u) for the (b, h, v) triples in rows.
    q/k_new/v_new: [B][n_max][H][d]; caches: [B][H][L_max][d]; float32 arrays,
    or uint16 arrays holding bfloat16 bits."""
    lib = _load()
    dtype = 1 if q.dtype == np.uint16 else 0
    conv = (lambda a: np.ascontiguousarray(a, np.uint16)) if dtype else _f32
    q, k_new, v_new, k_cache, v_cache = map(conv, (q, k_new, v_new, k_cache, v_cache))
    B, n_max, H, d = q.shape
    L_max = k_cache.shape[2]
    rows = _i32(rows).reshape(-1, 3)
    out = np.zeros((rows.shape[0], d), np.float64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    pl, nn, par = _i32(prefix_len), _i32(n_nodes), _i32(parent)
    rc = lib.or_tree_attention_rows(C.c_int(B), C.c_int(H), C.c_int(d), C.c_int(n_max), C.c_int(L_max),
                                    C.c_int(dtype), _p(q), _p(k_new), _p(v_new), _p(k_cache), _p(v_cache),
                                    _p(pl), _p(nn), _p(par), C.c_double(scale), C.c_int(rows.shape[0]),
                                    _p(rows), _p(out), C.c_int(nthreads))
    if rc:
        raise ValueError(f"oracle tree attention rejected its arguments (code {rc})")
    return out


def all_rows(B, H, n_nodes) -> np.ndarray:
    return np.array([(b, h, v) for b in range(B) for h in range(H) for v in range(int(n_nodes[b]))],
                    np.int32).reshape(-1, 3)


# --------------------------------------------------------------------------- #
# verification
# --------------------------------------------------------------------------- #
def verify_greedy(logits, parent, tokens, n_nodes):
    lib = _load()
    lg, par, tok, nn = _f32(logits), _i32(parent), _i32(tokens), _i32(n_nodes)
    B, n_max, V = lg.shape
    ot = np.full((B, n_max + 1), -1, np.int32)
    op = np.full((B, n_max + 1), -1, np.int32)
    oc = np.zeros(B, np.int32)
    am = np.full((B, n_max), -1, np.int32)
    st = np.zeros(B, np.int32)
    lib.or_verify_greedy(C.c_int(B), C.c_int(n_max), C.c_int(V), _p(nn), _p(par), _p(tok), _p(lg),
                         _p(ot), _p(op), _p(oc), _p(am), _p(st))
    return dict(tokens=ot, path=op, count=oc, argmax=am, status=st)


def verify_mss(logits, ssm, q_row, uniforms, parent, tokens, n_nodes, temperature=1.0, p_row=None,
               margin_eps=1e-6):
    lib = _load()
    lg, sm, qr, un = _f32(logits), _f32(ssm), _i32(q_row), _f32(uniforms)
    par, tok, nn = _i32(parent), _i32(tokens), _i32(n_nodes)
    B, n_max = par.shape
    NP, V = lg.shape[1], lg.shape[2]
    NQ = sm.shape[1]
    pr = None if p_row is None else _i32(p_row)
    ot = np.full((B, n_max + 1), -1, np.int32)
    op = np.full((B, n_max + 1), -1, np.int32)
    oc = np.zeros(B, np.int32)
    lm = np.zeros(B, np.int32)
    mm = np.zeros(B, np.float64)
    st = np.zeros(B, np.int32)
    rc = lib.or_verify_mss(C.c_int(B), C.c_int(n_max), C.c_int(V), _p(nn), _p(par), _p(tok), _p(lg), _p(pr),
                           C.c_int(NP), _p(sm), _p(qr), C.c_int(NQ), _p(un), C.c_double(temperature),
                           _p(ot), _p(op), _p(oc), _p(lm), _p(mm), _p(st), C.c_double(margin_eps))
    if rc & OR_BAD_ARG:
        raise ValueError("oracle MSS rejected its arguments")
    return dict(tokens=ot, path=op, count=oc, lm_pos=lm, min_margin=mm, status=st)


def mss_node_trace(p, child_tokens, q_rows):
    """(a_1..a_k, final residual) of one MSS node for exact-law checks."""
    lib = _load()
    p = np.ascontiguousarray(p, np.float64)
    ct = _i32(child_tokens)
    q = _f32(q_rows).reshape(len(ct), -1)
    V = p.shape[0]
    a = np.zeros(len(ct), np.float64)
    r = np.zeros(V, np.float64)
    g = lib.or_mss_node_trace(C.c_int(V), _p(p), C.c_int(len(ct)), _p(ct), _p(q), _p(a), _p(r))
    return a, r, int(g)


def verify_naive(logits, parent, tokens, n_nodes, uniforms, temperature=1.0):
    lib = _load()
    lg, par, tok, nn, un = _f32(logits), _i32(parent), _i32(tokens), _i32(n_nodes), _f32(uniforms)
    B, n_max, V = lg.shape
    ot = np.full((B, n_max + 1), -1, np.int32)
    oc = np.zeros(B, np.int32)
    lib.or_verify_naive(C.c_int(B), C.c_int(n_max), C.c_int(V), _p(nn), _p(par), _p(tok), _p(lg),
                        C.c_double(temperature), _p(un), _p(ot), _p(oc))
    return dict(tokens=ot, count=oc)


def kv_commit(k_cache, v_cache, prefix_len, dfs_of, out_path, out_count):
    """Returns (k_cache', v_cache', new_prefix_len) on copies of the caches."""
    lib = _load()
    k = np.array(k_cache, copy=True, order="C")
    v = np.array(v_cache, copy=True, order="C")
    B, H, L_max, d = k.shape
    n_max = dfs_of.shape[1]
    npl = np.zeros(B, np.int32)
    lib.or_kv_commit(C.c_int(B), C.c_int(H), C.c_int(d), C.c_int(L_max), C.c_int(n_max),
                     C.c_int(k.dtype.itemsize), _p(k), _p(v), _p(_i32(prefix_len)), _p(_i32(dfs_of)),
                     _p(_i32(out_path)), _p(_i32(out_count)), _p(npl))
    return k, v, npl

