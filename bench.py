"""Benchmark of one tree-verification step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config opt30b] [--impl ours|reference]

A step is the whole hot path over one batch of synthetic input, all through
the C ABI: tree_build -> kv_append -> tree_attention -> verify -> kv_commit.
Prints ONE JSON line (rank 0). Metric: verified tree nodes per second (the
speculated-tree nodes, root included, that one step verifies), whole job.
The headline workload is the largest single-GPU one (OPT-30B-shaped, 3008
nodes and about 3 GB of K/V and logits per step); the line also carries the
other four workloads measured in the same run (per_config).
Under torchrun every rank runs an independent replica on its own GPU (the path
needs no exchange); value = nodes of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tree nodes/s (tree-attn+verify) on 1 GB300; attn HBM GB/s vs peak"
L2_BYTES = 129 * 2**20
DESCR = {
    "tiny": "Tiny: 1 request, prefix 64, widths (2,2,1) -> 11 nodes, 4 heads x 64, fp32, vocab 256, greedy+MSS",
    "llama7b": "LLaMA-7B-shaped layer: batch 8, 32 heads x 128, bf16, prefix 2048, widths (1,1,3,1,1,1,1,1) -> 21 "
               "nodes, greedy verify over vocab 32000",
    "merge": "merge-based trees: batch 16, 32 heads x 128, bf16, prefixes U[512,4096], 3 chains x 8 merged, MSS "
             "over vocab 32000",
    "long65b": "long-context LLaMA-65B-shaped layer: batch 4, 64 heads x 128, bf16, prefix 16384, random tree of "
               "128 nodes, greedy+MSS over vocab 32000",
    "opt30b": "OPT-30B-shaped high batch: batch 64, 56 heads x 128, bf16, prefix 1024, widths (2,2,2,2,1) -> 47 "
              "nodes, MSS over vocab 50272",
}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def attention_bytes(w) -> int:
    """Algorithmic bytes of one tree_attention launch: every visible K and V row
    once (prefix + tree, per head), Q read and the output written once."""
    esz = 2 if w.dtype == "bf16" else 4
    n = w.n_nodes_dev
    kv = sum(int(w.prefix_len[b] + n[b]) for b in range(w.B)) * w.H * w.d * esz * 2
    qo = int(sum(n)) * w.H * w.d * esz * 2
    return kv + qo


def append_bytes(w) -> int:
    """Bytes a launch that also appends writes on top of attention_bytes: the
    tree's new K and V rows into the cache (the attention already counts them
    read once)."""
    esz = 2 if w.dtype == "bf16" else 4
    return int(sum(w.n_nodes_dev)) * w.H * w.d * esz * 2


def attention_launch(s):
    """The kernel name ncu summaries use for the step's attention launch, and
    whether that launch also appends the new K/V rows."""
    from tree_speculative_verification_gb300 import api
    w = s.w
    kernel = api.attention_kernel(w.B, w.H, w.n_max, w.d, w.L_max, api.TS_BF16 if w.dtype == "bf16" else api.TS_F32)
    fused = bool(getattr(s, "_append_in_attention", False))
    return (kernel + "+append" if fused else kernel), fused


def _profile_keys(path):
    kv = {}
    with open(path) as fh:
        for line in fh:
            if line.startswith("- ") and ":" in line:
                k, _, v = line[2:].partition(":")
                kv[k.strip()] = v.strip()
    return kv


def _traffic_from_profile(w, kernel):
    """DRAM bytes per full attention launch from a committed ncu summary under
    profiles/: the summary must name this workload and the kernel this run
    launches (`kernel`), and the hash of that kernel's source file (`source`)
    must equal the one recorded at capture time (`source_sha256_16`).
    Returns (bytes, summary file name) or (None, None)."""
    pdir = os.path.join(ROOT, "profiles")
    try:
        names = sorted(os.listdir(pdir))
    except OSError:
        return None, None
    for name in names:
        if not name.endswith(".md"):
            continue
        try:
            kv = _profile_keys(os.path.join(pdir, name))
        except OSError:
            continue
        if kv.get("kernel") != kernel or kv.get("workload") != w.name or "source" not in kv:
            continue
        try:
            src = os.path.join(ROOT, kv["source"])
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            if kv.get("source_sha256_16") == h:
                return float(kv["dram_bytes_per_full_launch"]), name
        except (OSError, KeyError, ValueError):
            continue
    return None, None


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the GPU is loaded."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.rows, self.proc = [], None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.rows:
            return None
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        window = "timed region"
        if not inside:
            inside = [r for _, r in self.rows]
            window = "loaded window around the timed region (shorter than one 200 ms sample)"
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in inside if num(r[1]) is not None]
        mx = [num(r[2]) for r in inside if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window}


def _oracle_tree(w):
    import oracle
    if w.tree_mode == "chains":
        B, n_max = w.B, w.n_max
        parent = np.full((B, n_max), -1, np.int32)
        tokens = np.zeros((B, n_max), np.int32)
        p_row = np.zeros((B, n_max), np.int32)
        q_row = np.zeros((B, n_max), np.int32)
        n_nodes = np.zeros(B, np.int32)
        for b in range(B):
            par, tok, src = oracle.merge_chains(w.chains[b], int(w.root_token[b]), n_max)
            n = len(par)
            n_nodes[b] = n
            parent[b, :n], tokens[b, :n], p_row[b, :n], q_row[b, :n] = par, tok, src + 1, np.maximum(src, 0)
        return parent, tokens, n_nodes, p_row, q_row
    return w.parent, w.tokens, w.n_nodes, None, w.q_row


def run_oracle_sample(w, heads: int, verify: bool = True, nthreads: int = 0):
    """One bounded oracle pass: attention rows of request 0 for `heads` heads
    (on `nthreads` threads, 0 = all cores), then (optionally) the step's
    verifier on every request. Returns seconds spent in attention and in
    verification."""
    import oracle
    parent, tokens, n_nodes, p_row, q_row = _oracle_tree(w)
    n0 = int(n_nodes[0])
    rows = np.array([(0, h, v) for h in range(heads) for v in range(n0)], np.int32)
    t0 = time.perf_counter()
    if w.q is not None and heads > 0:
        oracle.tree_attention_rows(w.q, w.k_new, w.v_new, w.k_cache, w.v_cache, w.prefix_len, n_nodes, parent, rows,
                                   nthreads=nthreads)
    t1 = time.perf_counter()
    if verify:
        if w.verify == "naive":
            oracle.verify_naive(np.stack([w.logits[b][p_row[b]] for b in range(w.B)]) if p_row is not None
                                else w.logits, parent, tokens, n_nodes, w.uniforms, w.temperature)
        if w.verify in ("greedy", "both"):
            oracle.verify_greedy(w.logits, parent, tokens, n_nodes)
        if w.verify in ("mss", "both"):
            oracle.verify_mss(w.logits, w.ssm, q_row, w.uniforms, parent, tokens, n_nodes, w.temperature,
                              p_row=p_row)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1, n_nodes


def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo, or lscpu on Arm hosts)."""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_nodes_per_s(w, budget_s: float, nthreads: int = 0):
    """Time the oracle on a bounded sample and extrapolate to the whole step.
    nthreads: attention threads (0 = all cores; verification is serial C)."""
    import oracle
    ta, tv, n_nodes = run_oracle_sample(w, heads=1, nthreads=nthreads)
    heads = max(1, min(w.H, int(budget_s / max(ta, 1e-4))))
    ta, tv2, n_nodes = run_oracle_sample(w, heads=heads, verify=False, nthreads=nthreads)
    # attention cost per node-head from the sample, applied to every node-head of the step
    per_node_head = ta / (heads * int(n_nodes[0]))
    # rows of longer prefixes cost proportionally more keys
    keys = np.array([w.prefix_len[b] + n_nodes[b] for b in range(w.B)], np.float64)
    scale = float(np.sum(n_nodes * keys) / (n_nodes[0] * keys[0]))
    t_step = per_node_head * w.H * int(n_nodes[0]) * scale + tv
    sample = (f"oracle tree attention for request 0 ({int(n_nodes[0])} nodes) x {heads} of {w.H} heads "
              f"({ta:.2f} s), scaled by key count to all {w.B} requests and heads; oracle verification of all "
              f"{w.B} requests ({tv:.2f} s)")
    return float(np.sum(n_nodes)) / t_step, t_step, (nthreads or oracle.num_threads()), sample


def _events(n, external):
    import torch
    kw = {"enable_timing": True}
    if external:
        kw["external"] = True     # record nodes inside a captured graph
    return [torch.cuda.Event(**kw) for _ in range(n)]


def replica_rate(ms_per_step, units_per_step, dist=None, device="cpu"):
    """Whole-job rate of N independent replicas (one per rank, no exchange): the
    slowest rank's time per step (max over ranks) and every rank's units over it.
    Returns (ms per step, units per second)."""
    import torch
    ws = 1
    if dist is not None:
        ws = dist.get_world_size()
        t = torch.tensor([float(ms_per_step)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_per_step = float(t.item())
    return ms_per_step, ws * units_per_step / (ms_per_step * 1e-3)


def config_dict(w, name, kind, ws, scale_down=1):
    """The workload description both arms print (identical for the same run)."""
    return {"workload": DESCR[name] + (f" (batch and long prefix / {scale_down})" if scale_down > 1 else ""),
            "name": name, "batch": w.B, "heads": w.H, "head_dim": w.d, "vocab": w.V,
            "nodes_per_step": int(np.sum(w.n_nodes_dev)), "verify": kind,
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    """--impl reference: the oracle as it stands on the host cores, same config,
    metric and unit; each step a bounded sample sized to finish in minutes."""
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    from tree_speculative_verification_gb300 import workloads
    w = workloads.make(args.config)
    if args.verify:
        w.verify = args.verify
    w.n_nodes_dev = _oracle_tree(w)[2]
    per_step_budget = max(0.05, min(2.0, 90.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_nodes_per_s(w, per_step_budget)
    vals, times = [], []
    for _ in range(args.steps):
        v, t_step, cores, sample = oracle_nodes_per_s(w, per_step_budget)
        vals.append(v)
        times.append(t_step)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "nodes/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, args.config, w.verify, args.gpus),
            "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _load_step(name, args, device, verify=None, paged=False, serial_verify=False):
    from tree_speculative_verification_gb300 import api, workloads
    from tree_speculative_verification_gb300.step import DeviceStep
    w = workloads.make(name, scale_down=args.scale_down)
    if verify:
        if verify in ("mss", "both") and w.ssm is None:
            raise SystemExit(f"--verify {verify}: the {name} workload has no drafter distributions")
        w.verify = verify
    s = DeviceStep(w, device, paged=paged, serial_verify=serial_verify)
    s.run(w.verify)
    import torch
    torch.cuda.synchronize()
    w.n_nodes_dev = s.tree.n_nodes.cpu().numpy()
    if s.status.item() not in (0, api.STATUS_ZERO_RESID):
        raise RuntimeError(f"{name}: device status {s.status.item()} after the first step")
    return w, s


def _timed_graphs(s, kind, K, device, stream, eager=False):
    """The K steps as one CUDA graph (the step's library calls; the graph
    removes the host launch overhead between them) with events at its two ends
    only -- an event-record node between two kernels of a graph costs a few
    microseconds -- and two more graphs of K back-to-back launches of the
    attention call and of the verify call alone on the same inputs (the time
    between two launches counts, so those figures are conservative).
    Returns (events per pass, a function replaying a pass, launch mode)."""
    import torch
    passes = {
        "step": lambda: [s.run(kind) for _ in range(K)],
        # the step's attention launch (with the KV append when it rides there)
        "attend": lambda: [(s.attend_append() if s._append_in_attention else s.attend()) for _ in range(K)],
        "verify": lambda: [s.verify(kind) for _ in range(K)],
    }
    evs = {k: _events(2, not eager) for k in passes}
    graphs, mode = None, "eager launches"
    if not eager:
        try:
            graphs = {}
            for k, body in passes.items():
                g = torch.cuda.CUDAGraph()
                cs = torch.cuda.Stream(device)
                cs.wait_stream(stream)
                with torch.cuda.graph(g, stream=cs, capture_error_mode="relaxed"):
                    cur = torch.cuda.current_stream(device)
                    evs[k][0].record(cur)
                    body()
                    evs[k][1].record(cur)
                stream.wait_stream(cs)
                g.replay()
                torch.cuda.synchronize()
                graphs[k] = g
            mode = "CUDA graph of the K steps"
        except Exception as exc:     # no graph support for event nodes: time eager launches
            graphs = None
            mode = f"eager launches ({type(exc).__name__} capturing a graph)"
            torch.cuda.synchronize()
            evs = {k: _events(2, False) for k in passes}

    def replay(k="step"):
        if graphs is not None:
            graphs[k].replay()
        else:
            evs[k][0].record(stream)
            passes[k]()
            evs[k][1].record(stream)

    return evs, replay, mode


def _roofline(w, t_att_ms, kernel, fused=False):
    peak, peak_kind = _peaks()
    abytes = attention_bytes(w) + (append_bytes(w) if fused else 0)
    achieved = abytes / (t_att_ms * 1e-3) / 1e9
    traffic, prof = _traffic_from_profile(w, kernel)
    call = "tree_attention_append" if fused else "tree_attention"
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "traffic_source": prof, "kernel": f"{call} ({kernel})",
            "algorithmic_bytes_per_launch": abytes, "peak_kind": peak_kind, "avg_launch_us": t_att_ms * 1e3}


def measure_other_config(name, args, device, stream):
    """A workload other than the headline one, measured in the same run with
    the same method (graphs of K steps and of K back-to-back attention /
    verify launches); no end-to-end leg, no CPU baseline."""
    import torch
    from tree_speculative_verification_gb300 import api
    w, s = _load_step(name, args, device)
    kind = w.verify
    K = max(10, min(args.steps, 100))
    for _ in range(3):
        s.run(kind)
    torch.cuda.synchronize()
    evs, replay, _ = _timed_graphs(s, kind, K, device, stream, args.eager)
    out = {}
    for k in ("step", "attend", "verify"):
        replay(k)
        torch.cuda.synchronize()
        replay(k)
        torch.cuda.synchronize()
        out[k] = evs[k][0].elapsed_time(evs[k][1]) / K
    nodes = int(w.n_nodes_dev.sum())
    kernel, fused = attention_launch(s)
    roof = _roofline(w, out["attend"], kernel, fused)
    line = {"value": nodes / (out["step"] * 1e-3), "unit": "nodes/s", "ms_per_step": out["step"],
            "nodes_per_step": nodes, "attention_ms": out["attend"], "verify_ms": out["verify"], "verify": kind,
            "attention_kernel": kernel, "roofline_frac": roof["frac"], "attention_gbs": roof["achieved"],
            "attention_traffic_bytes": roof["traffic"],
            "accepted_tokens_per_step": s.accepted(kind), "steps": K, "workload": DESCR[name]}
    del s, w
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def run_ours(args):
    import torch
    ws, rank, local = _dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    from tree_speculative_verification_gb300 import api, workloads
    api.load_library()
    stream = torch.cuda.current_stream(device)
    w, s = _load_step(args.config, args, device, args.verify, paged=args.paged, serial_verify=args.serial_verify)
    kind = w.verify
    nodes_per_step = int(w.n_nodes_dev.sum())
    accepted_per_step = s.accepted(kind)

    def barrier():
        if dist:
            dist.barrier()

    # ---- warm-up, then K timed steps (device time, CUDA events on the launch stream)
    for _ in range(args.warmup):
        s.run(kind)
    torch.cuda.synchronize()
    K = args.steps
    evs, timed_pass, launch_mode = _timed_graphs(s, kind, K, device, stream, args.eager)
    sampler = ClockSampler(device.index if device.index is not None else 0) if rank == 0 else None
    t_load0 = time.time()
    while time.time() - t_load0 < 0.6:      # keep the GPU loaded while the sampler starts
        timed_pass()
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    timed_pass()
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    ms = evs["step"][0].elapsed_time(evs["step"][1])
    timed_pass("attend")
    timed_pass("verify")
    torch.cuda.synchronize()
    t_load1 = time.time()
    while time.time() - t_load1 < 0.4:
        timed_pass()
        torch.cuda.synchronize()
    if sampler:
        sampler.stop()
    t_att = evs["attend"][0].elapsed_time(evs["attend"][1]) / K
    t_ver = evs["verify"][0].elapsed_time(evs["verify"][1]) / K
    seq_line = None
    if args.sequence_baseline and rank == 0:
        seq_line = measure_sequence_baseline(w, K, device, stream, t_att)
    sweep = measure_sequence_sweep(K, device, stream) if args.sequence_sweep and rank == 0 else None
    ms_per_step, value = replica_rate(ms / args.steps, nodes_per_step, dist, device)

    # ---- end to end through the C ABI with host buffers: pinned inputs in, results out
    # every rank runs it (replicas); the slowest rank's time sets the job's figure
    barrier()
    e2e = measure_e2e(s, w, kind, args, stream)
    e2e["ms_per_step"], e2e["value"] = replica_rate(e2e["ms_per_step"], nodes_per_step, dist, device)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    kernel, fused = attention_launch(s)
    roof = _roofline(w, t_att, kernel, fused)
    launches = args.steps * s.launches_per_step(kind)
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    host_w = w
    del s
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    per_config = None
    if ws == 1 and not args.no_per_config and args.scale_down == 1:
        per_config = {}
        for name in workloads.CONFIG_NAMES:
            if name != args.config:
                per_config[name] = measure_other_config(name, args, device, stream)
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        v, t_step, cores, sample = oracle_nodes_per_s(host_w, 12.0)
        v1, t1, _, sample1 = oracle_nodes_per_s(host_w, 6.0, nthreads=1)
        cpu = {"value": v, "unit": "nodes/s", "cores": cores, "kind": "oracle", "sample": sample,
               "cpu_model": cpu_model(),
               "single_thread": {"value": v1, "unit": "nodes/s", "cores": 1, "sample": sample1}}
    line = {"metric": METRIC, "value": value, "unit": "nodes/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_dict(w, args.config, kind, ws, args.scale_down),
            "timing": {"launch": launch_mode,
                       "kernel_timing": "attention and verify durations from graphs of K back-to-back launches "
                                        "of that call on the same inputs, events at both ends",
                       "l2": f"inputs larger than L2: {attention_bytes(w) / 2**20:.0f} MiB of K/V+Q per step vs "
                             f"129 MiB"},
            "nodes_per_s_attn_verify": ws * nodes_per_step / ((t_att + t_ver) * 1e-3),
            "attention_ms": t_att, "verify_ms": t_ver,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "accepted_tokens_per_step": accepted_per_step,
            **({"sequence_baseline": seq_line} if seq_line else {}),
            "accepted_tokens_per_s": ws * accepted_per_step / (ms_per_step * 1e-3),
            "gpu_launches": launches,
            **({"per_config": per_config} if per_config else {}),
            **({"sequence_sweep": sweep} if sweep else {}),
            **({"cache": "paged (pages of 64 keys, randomly placed)"} if args.paged else {}),
            **({"step_order": "verification after attention on one stream"} if args.serial_verify else {})}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def _graph_time(fn, K, device, stream):
    """Milliseconds per call of fn from a CUDA graph of K back-to-back calls."""
    import torch
    ge = _events(2, True)
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(device)
    cs.wait_stream(stream)
    with torch.cuda.graph(g, stream=cs, capture_error_mode="relaxed"):
        cur = torch.cuda.current_stream(device)
        ge[0].record(cur)
        for _ in range(K):
            fn()
        ge[1].record(cur)
    stream.wait_stream(cs)
    g.replay()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    return ge[0].elapsed_time(ge[1]) / K


def measure_sequence_sweep(K, device, stream, batches=(1, 2, 4, 8, 16)):
    """SpecInfer Fig. 11 on this GPU, for the attention layer: the LLaMA-7B-shaped
    layer (32 heads x 128, prefix 2048, expansion tree (1,1,3,1,1,1,1,1), 21
    nodes and 3 root-to-leaf paths per request) at several batch sizes, tree
    attention against sequence-based attention (one sequence and one prefix
    copy per path), each timed as a graph of K back-to-back launches."""
    import torch
    from tree_speculative_verification_gb300 import api, workloads
    from tree_speculative_verification_gb300.step import DeviceStep
    rows = []
    for B in batches:
        w = workloads.make("llama7b", batch=B)
        tree = DeviceStep(w, device)
        tree.build()
        tree.append()
        seq_w, _ = workloads.sequence_batch(w)
        seq_w.n_nodes_dev = seq_w.n_nodes
        seq = DeviceStep(seq_w, device)
        seq.build()
        seq.append()
        torch.cuda.synchronize()
        t_tree = _graph_time(tree.attend, K, device, stream)
        t_seq = _graph_time(seq.attend, K, device, stream)
        w.n_nodes_dev = w.n_nodes
        bf = api.TS_BF16
        rows.append({"batch": B, "tree_ms": t_tree, "sequence_ms": t_seq, "ratio": t_seq / t_tree,
                     "paths": int(seq_w.B), "tree_bytes": attention_bytes(w), "sequence_bytes": attention_bytes(seq_w),
                     "tree_kernel": api.attention_kernel(w.B, w.H, w.n_max, w.d, w.L_max, bf),
                     "sequence_kernel": api.attention_kernel(seq_w.B, seq_w.H, seq_w.n_max, seq_w.d, seq_w.L_max, bf)})
        del tree, seq
        torch.cuda.empty_cache()
    return rows


def measure_sequence_baseline(w, K, device, stream, t_att):
    """SpecInfer Fig. 4 (left) / Fig. 11: one sequence and one prefix copy per
    root-to-leaf path, the same attention call on the chains."""
    import torch
    from tree_speculative_verification_gb300 import api, workloads
    from tree_speculative_verification_gb300.step import DeviceStep
    seq_w, path_nodes = workloads.sequence_batch(w)
    seq_w.n_nodes_dev = seq_w.n_nodes
    sq = DeviceStep(seq_w, device)
    sq.build()
    sq.append()
    torch.cuda.synchronize()
    ge = _events(2, True)
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(device)
    cs.wait_stream(stream)
    with torch.cuda.graph(g, stream=cs, capture_error_mode="relaxed"):
        cur = torch.cuda.current_stream(device)
        ge[0].record(cur)
        for _ in range(K):
            sq.attend()
        ge[1].record(cur)
    stream.wait_stream(cs)
    g.replay()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    t_seq = ge[0].elapsed_time(ge[1]) / K
    line = {"paths": int(seq_w.B), "path_nodes": int(seq_w.n_nodes.sum()), "attention_ms": t_seq,
            "algorithmic_bytes_per_launch": attention_bytes(seq_w),
            "tree_speedup": t_seq / t_att,
            "kernel": api.attention_kernel(seq_w.B, seq_w.H, seq_w.n_max, seq_w.d, seq_w.L_max,
                                           api.TS_BF16 if seq_w.dtype == "bf16" else api.TS_F32)}
    del sq, g
    return line


def measure_e2e(s, w, kind, args, stream):
    """Same metric through the public API with HOST buffers: per step, the
    step's inputs (tokens, prefix lengths, Q / new K / new V, logits and, for
    MSS, drafter rows and uniforms) go host->device from pinned memory, the
    step runs, and the verified tokens and counts come back device->host.

    The copies are pipelined the way a serving loop would run them: two sets of
    device input/output buffers, step i+1's inputs copied on a copy stream while
    step i computes, step i's results read back on a third stream.  The compute
    of the steps stays serialised on one stream (they share the KV cache); every
    copy of every timed step, the first step's inputs and the last step's
    results included, lies inside the timed region."""
    import copy
    import torch
    pinned = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
    in_names = {"chains": ["chains", "root_token"], "widths": ["tokens"],
                "parent": ["tokens", "parent", "n_nodes_in"]}[w.tree_mode]
    in_names += ["prefix_len", "q", "k_new", "v_new", "logits"]
    if kind in ("mss", "both"):
        in_names += ["ssm", "uniforms"] + (["q_row"] if w.tree_mode != "chains" else [])
    if kind == "naive":
        in_names += ["uniforms"]
    in_names = [n for n in in_names if getattr(s, n, None) is not None]
    out_names = ["mss_tokens", "mss_count"] if kind in ("mss", "naive") else ["out_tokens", "out_count"]
    out_names.append("new_prefix_len")
    # the second buffer set shares the KV cache, tree and workspaces (only the
    # compute stream touches them) and owns its inputs and outputs
    s2 = copy.copy(s)
    for n in in_names + out_names + ["out_path", "mss_path"]:
        setattr(s2, n, torch.empty_like(getattr(s, n)))
    sets = [s, s2]
    host_in = [pinned(getattr(s, n)) for n in in_names]
    host_out = [[torch.empty(getattr(s, n).shape, dtype=getattr(s, n).dtype, pin_memory=True) for n in out_names]
                for _ in sets]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    steps = max(3, min(args.steps, 200))
    cs, rs = torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in sets]
    computed = [torch.cuda.Event() for _ in sets]
    read = [torch.cuda.Event() for _ in sets]

    def h2d_copy(j):
        with torch.cuda.stream(cs):
            for n, host in zip(in_names, host_in):
                getattr(sets[j], n).copy_(host, non_blocking=True)
            copied[j].record(cs)

    def run(n_steps, start):
        cs.wait_event(start)
        h2d_copy(0)
        for i in range(n_steps):
            j = i & 1
            if i + 1 < n_steps:
                if i >= 1:                       # set j^1 was last used by step i-1
                    cs.wait_event(computed[j ^ 1])
                h2d_copy(j ^ 1)
            stream.wait_event(copied[j])
            if i >= 2:                           # its results of step i-2 are read back
                stream.wait_event(read[j])
            sets[j].run(kind, stream)
            computed[j].record(stream)
            rs.wait_event(computed[j])
            with torch.cuda.stream(rs):
                for host, n in zip(host_out[j], out_names):
                    host.copy_(getattr(sets[j], n), non_blocking=True)
                read[j].record(rs)
        stream.wait_stream(rs)
        stream.wait_stream(cs)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = torch.cuda.Event()
    w0.record(stream)
    run(3, w0)
    torch.cuda.synchronize()
    e0.record(stream)
    run(steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    for j in range(2):                           # the read-back results are the device's
        for host, n in zip(host_out[j], out_names):
            assert torch.equal(host, getattr(sets[j], n).cpu()), n
    nodes = int(w.n_nodes_dev.sum())
    return {"value": nodes / (ms * 1e-3), "unit": "nodes/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": steps,
            "copies": "pinned host buffers; step i+1's inputs copied on a second stream while step i computes, "
                      "results read back on a third"}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="opt30b", choices=sorted(DESCR))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other four workloads (per_config)")
    ap.add_argument("--sequence-baseline", action="store_true",
                    help="also time attention as one sequence per root-to-leaf path (SpecInfer Fig. 4 left)")
    ap.add_argument("--verify", default=None, choices=["greedy", "mss", "naive", "both"],
                    help="verifier of the step (default: the workload's)")
    ap.add_argument("--sequence-sweep", action="store_true",
                    help="tree vs sequence-based attention on the LLaMA-7B-shaped layer at batch 1, 2, 4, 8, 16")
    ap.add_argument("--paged", action="store_true", help="the KV cache in pages of 64 keys (paged calls)")
    ap.add_argument("--serial-verify", action="store_true",
                    help="verification after the attention on one stream (no overlap)")
    ap.add_argument("--eager", action="store_true", help="launch every step from the host instead of a CUDA graph")
    ap.add_argument("--scale-down", type=int, default=1,
                    help="divide the batch (and the long prefix) by N: a smaller case of the same kernels, for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
