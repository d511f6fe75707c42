"""One tree-verification step on the GPU, driven through the C ABI.

DeviceStep holds a workload's tensors on the device (KV cache, Q / new K/V,
logits, drafter probabilities, uniforms) and the output buffers, and runs the
hot path: tree_build -> kv_append -> tree_attention -> verify (greedy and/or
MSS, or naive sampling) -> kv_commit. kv_commit writes the new prefix lengths into a separate
array, so repeating a step on the same inputs is idempotent.
"""
from __future__ import annotations

import numpy as np
import torch

from . import api
from .workloads import Workload


def to_device(a: np.ndarray, device, bf16: bool = False) -> torch.Tensor:
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceStep:
    """paged: keep the KV cache in pages of api.PAGE_KEYS rows (randomly placed,
    listed per request in a block table) and run the paged calls.
    serial_verify: run verification after the attention on the main stream
    (the order a verification that also commits would need)."""

    def __init__(self, w: Workload, device="cuda", attention: bool = True, paged: bool = False,
                 serial_verify: bool = False, seed: int = 0):
        self.w = w
        self.device = device
        self.paged = paged
        self.serial_verify = serial_verify
        dev = device
        B, n_max = w.B, w.n_max
        i32 = lambda a: to_device(np.asarray(a, np.int32), dev)
        self.tree = api.Tree(B, n_max, dev)
        self.prefix_len = i32(w.prefix_len)
        self.new_prefix_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        if w.tree_mode == "chains":
            self.chains = i32(w.chains)
            self.root_token = i32(w.root_token)
            self.tokens = torch.full((B, n_max), -1, dtype=torch.int32, device=dev)
            self.p_row = torch.full((B, n_max), -1, dtype=torch.int32, device=dev)
            self.q_row = torch.full((B, n_max), -1, dtype=torch.int32, device=dev)
        else:
            self.tokens = i32(w.tokens)
            self.parent = i32(w.parent)
            self.n_nodes_in = i32(w.n_nodes)
            self.p_row = None
            self.q_row = i32(w.q_row) if w.q_row is not None else None
        self.logits = to_device(w.logits, dev)
        self.ssm = to_device(w.ssm, dev) if w.ssm is not None else None
        self.uniforms = to_device(w.uniforms, dev)
        self.out_tokens = torch.full((B, n_max + 1), -1, dtype=torch.int32, device=dev)
        self.out_path = torch.full((B, n_max + 1), -1, dtype=torch.int32, device=dev)
        self.out_count = torch.zeros(B, dtype=torch.int32, device=dev)
        self.mss_tokens = torch.full((B, n_max + 1), -1, dtype=torch.int32, device=dev)
        self.mss_path = torch.full((B, n_max + 1), -1, dtype=torch.int32, device=dev)
        self.mss_count = torch.zeros(B, dtype=torch.int32, device=dev)
        self.mss_lowmargin = torch.zeros(B, dtype=torch.int32, device=dev)
        self.argmax = torch.full((B, n_max), -1, dtype=torch.int32, device=dev)
        self.ws_greedy = api.workspace(api.TS_OP_VERIFY_GREEDY, B, n_max=n_max, V=w.V, device=dev)
        self._side = None   # verification stream, created on first use
        self._fused = w.tree_mode == "widths"   # tree_build_append applies
        self._append_in_attention = False       # tree_attention_append is one launch
        self.attention = attention and w.q is not None
        if self.attention:
            bf = w.dtype == "bf16"
            self.q = to_device(w.q, dev, bf)
            self.k_new = to_device(w.k_new, dev, bf)
            self.v_new = to_device(w.v_new, dev, bf)
            self.out = torch.zeros_like(self.q)
            self.ws_attn = api.workspace(api.TS_OP_ATTENTION, B, w.H, n_max, w.d, w.L_max, w.V, device=dev)
            if paged:
                self.kv = self._pages(np.random.default_rng(seed))
                self.k_cache = self.v_cache = None
                self._fused = False
            else:
                self.k_cache = to_device(w.k_cache, dev, bf)
                self.v_cache = to_device(w.v_cache, dev, bf)
                # the fused append for the tcgen05 kernel's form for trees of up to 64 nodes (with more,
                # long-context layer: 361.7 us fused against 5.6 + 347.8 us as two launches)
                kern = api.attention_kernel(w.B, w.H, w.n_max, w.d, w.L_max, api.TS_BF16 if bf else api.TS_F32)
                self._append_in_attention = kern.startswith("k_attn_tq") and w.n_max <= 64

    def _pages(self, rng):
        """The prefix cache scattered into randomly placed pages of PAGE_KEYS rows."""
        w, PK = self.w, api.PAGE_KEYS
        if w.dtype != "bf16":
            raise ValueError("the paged cache holds bf16 rows")
        max_pages = (w.L_max + PK - 1) // PK
        need = [(int(w.prefix_len[b]) + w.n_max + PK - 1) // PK for b in range(w.B)]
        ids = rng.permutation(sum(need))
        bt = np.full((w.B, max_pages), -1, np.int32)
        kp = np.zeros((len(ids), w.H, PK, w.d), np.uint16)
        vp = np.zeros_like(kp)
        nxt = 0
        for b in range(w.B):
            for j in range(need[b]):
                g = int(ids[nxt])
                nxt += 1
                bt[b, j] = g
                lo, hi = j * PK, min((j + 1) * PK, w.L_max)
                kp[g, :, :hi - lo] = w.k_cache[b, :, lo:hi]
                vp[g, :, :hi - lo] = w.v_cache[b, :, lo:hi]
        dv = self.device
        return api.PagedKV(to_device(kp, dv, True), to_device(vp, dv, True), to_device(bt, dv))

    # -- the five rows of the hot path ----------------------------------------
    def build(self, stream=None):
        w = self.w
        if w.tree_mode == "chains":
            api.tree_build_chains(self.tree, self.root_token, self.chains, self.tokens, self.p_row, self.q_row,
                                  self.prefix_len, self.status, stream)
        elif w.tree_mode == "widths":
            api.tree_build(self.tree, self.tokens, widths=w.widths, prefix_len=self.prefix_len, status=self.status,
                           stream=stream)
        else:
            api.tree_build(self.tree, self.tokens, self.parent, self.n_nodes_in, prefix_len=self.prefix_len,
                           status=self.status, stream=stream)

    def append(self, stream=None):
        if self.paged:
            api.kv_append_paged(self.kv, self.k_new, self.v_new, self.prefix_len, self.tree, self.status, stream)
            return
        api.kv_append(self.k_cache, self.v_cache, self.k_new, self.v_new, self.prefix_len, self.tree, self.status,
                      stream)

    def attend(self, stream=None):
        if self.paged:
            api.tree_attention_paged(self.out, self.q, self.kv, self.prefix_len, self.tree, 0.0, self.ws_attn,
                                     self.status, stream)
            return
        api.tree_attention(self.out, self.q, self.k_cache, self.v_cache, self.prefix_len, self.tree, 0.0,
                           self.ws_attn, self.status, stream)

    def attend_append(self, stream=None):
        """kv_append and tree_attention in one call (dense cache)."""
        api.tree_attention_append(self.out, self.q, self.k_cache, self.v_cache, self.k_new, self.v_new,
                                  self.prefix_len, self.tree, 0.0, self.ws_attn, self.status, stream)

    def verify(self, kind: str | None = None, stream=None):
        kind = kind or self.w.verify
        if kind in ("greedy", "both"):
            api.verify_greedy(self.out_tokens, self.out_path, self.out_count, self.logits, self.tree, self.argmax,
                              self.ws_greedy, self.status, stream)
        if kind in ("mss", "both"):
            api.verify_mss(self.mss_tokens, self.mss_path, self.mss_count, self.logits, self.ssm, self.q_row,
                           self.uniforms, self.w.temperature, self.tree, p_row=self.p_row, status=self.status,
                           stream=stream, lowmargin=self.mss_lowmargin)
        if kind == "naive":
            api.verify_naive(self.mss_tokens, self.mss_path, self.mss_count, self.logits, self.uniforms,
                             self.w.temperature, self.tree, p_row=self.p_row, status=self.status, stream=stream,
                             lowmargin=self.mss_lowmargin)

    def commit(self, kind: str | None = None, stream=None):
        kind = kind or self.w.verify
        path, count = ((self.mss_path, self.mss_count) if kind in ("mss", "both", "naive")
                       else (self.out_path, self.out_count))
        if self.paged:
            api.kv_commit_paged(self.kv, self.prefix_len, self.new_prefix_len, path, count, self.tree, self.status,
                                stream)
            return
        api.kv_commit(self.k_cache, self.v_cache, self.prefix_len, self.new_prefix_len, path, count, self.tree,
                      self.status, stream)

    def run(self, kind: str | None = None, stream=None):
        """One step. Verification reads only the tree and the logits, so it runs on
        a second stream beside the KV append and the attention; the commit, which
        needs the accepted path and the appended rows, waits for both.

        With the persistent tcgen05 kernel for trees of up to 64 nodes the append
        rides in the attention launch (tree_attention_append), and the tree is
        built on the second stream, the verification following it there as a
        programmatic dependent launch: its CTAs take their SMs while the build
        runs, before the persistent attention (launched on the main stream once
        the build is done) fills every SM. Launched side by side, the attention's
        CTAs came first and the walk ran after it (OPT-30B-shaped step 384 us;
        built on the second stream 356 us; 369 us with the append a launch of
        its own). Otherwise the tree is built on the main stream: greedy
        verification (many small CTAs) forks after the append, so that the
        attention's CTAs are placed first, MSS right after the build, and with
        the mma.sync kernel and an expansion tree the append rides in the
        tree_build launch (tree_build_append)."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if not self.attention:
            self.build(main)
            self.verify(kind, main)
            return
        if self.serial_verify:   # one stream: build, append, attention, verification, commit
            self.build(main)
            self.append(main)
            self.attend(main)
            self.verify(kind, main)
            self.commit(kind, main)
            return
        if self._side is None:
            self._side = torch.cuda.Stream(self.device)
            self._fork, self._built, self._join = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        side = self._side
        if self._append_in_attention:
            self._fork.record(main)          # the previous step's commit
            side.wait_event(self._fork)
            self.build(side)
            self._built.record(side)
            self.verify(kind, side)
            self._join.record(side)
            main.wait_event(self._built)
            self.attend_append(main)
            main.wait_event(self._join)
            self.commit(kind, main)
            return
        late = (kind or self.w.verify) == "greedy"
        if late and self._fused:   # expansion tree: tree_build and kv_append in one launch
            api.tree_build_append(self.tree, self.tokens, self.w.widths, self.prefix_len, self.k_cache, self.v_cache,
                                  self.k_new, self.v_new, self.status, main)
        else:
            self.build(main)
            if late:
                self.append(main)
        self._fork.record(main)
        side.wait_event(self._fork)
        self.verify(kind, side)
        self._join.record(side)
        if not late:
            self.append(main)
        self.attend(main)
        main.wait_event(self._join)
        self.commit(kind, main)

    def accepted(self, kind: str | None = None) -> int:
        """Tokens the last verification produced, over all requests."""
        kind = kind or self.w.verify
        count = self.mss_count if kind in ("mss", "both", "naive") else self.out_count
        return int(count.sum().item())

    def launches_per_step(self, kind: str | None = None) -> int:
        """Kernel launches of one step: tree_build (with the append when it rides
        there), the append when it is a launch of its own, the attention (with
        the append when it rides there; "a+b" names a call of two launches), the
        commit, and one launch per verification."""
        kind = kind or self.w.verify
        n = 1 + (2 if kind == "both" else 1)
        if self.attention:
            w = self.w
            name = api.attention_kernel(w.B, w.H, w.n_max, w.d, w.L_max,
                                        api.TS_BF16 if w.dtype == "bf16" else api.TS_F32)
            append_rides = self._append_in_attention or (self._fused and kind == "greedy" and not self.serial_verify)
            n += len(name.split("+")) + 1 + (0 if append_rides else 1)
        return n
