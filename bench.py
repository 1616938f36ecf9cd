#!/usr/bin/env python3
"""Benchmark of paged grouped-query attention on GB300.

One step = one call of the hot path on one batch: pa_decode (split partials
+ combine) on the ragged continuous-batching decode batch (16 sequences,
32 q / 8 kv heads, head_dim 128, 32-token pages, bf16) unless --workload
names another.  Inputs are device-resident; consecutive calls rotate over R
disjoint sets of physical pages of one pool (and R copies of q) whose total
footprint is at least 3x the L2 size, so every call reads K/V from HBM.  The K timed steps are replays of a CUDA graph of
calls, timed with CUDA events on the launching stream.

value = algorithmic bytes per call (K+V once per kv head, Q, O as f32)
        x steps x ranks / max-over-ranks time, in GB/s.

--impl reference times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import datetime as dt
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA attention µs/call and KV HBM GB/s (fraction of GB300 peak)"
DEFAULT_WORKLOAD = "ragged_b16_32x8_d128"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-secondary", action="store_true", help="skip the other workloads")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ncu-once", action="store_true",
                    help="profiling target: warm-up calls then one call of --workload, no graphs")
    return ap.parse_args()


# --------------------------------------------------------------- helpers --

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


_TOKENS = re.compile(r'"(?:\\.|[^"\\])*"' + r"|'(?:\\.|[^'\\])*'" + r"|//[^\n]*|/\*.*?\*/", re.S)


# The translation unit each profiled kernel is compiled from.
KERNEL_FILES = {"decode_v1": "pa_decode_v1.cu", "combine_v1": "pa_decode_v1.cu",
                "prefill_tc": "pa_prefill_tc.cu", "prefill_f32": "pa_prefill_f32.cu",
                "decode_v0": "pa_tile_v0.cu", "combine_v0": "pa_tile_v0.cu"}
_INCLUDE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)


def kernel_sources(kernel: str):
    """The kernel's translation unit and every local header it includes,
    directly or not (looked up beside the includer, then in include/)."""
    csrc = os.path.join(ROOT, "paged_kv_gqa_02_gb300", "csrc")
    todo, seen = [os.path.join(csrc, KERNEL_FILES[kernel])], []
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.append(f)
        with open(f, encoding="utf-8") as fh:
            for name in _INCLUDE.findall(fh.read()):
                for d in (os.path.dirname(f), csrc, os.path.join(ROOT, "include")):
                    if os.path.exists(os.path.join(d, name)):
                        todo.append(os.path.join(d, name))
                        break
    return sorted(seen)


def src_hash(kernel: str):
    """Hash of the kernel's sources (kernel_sources) without their comments
    and with runs of white space collapsed: editing a comment, or a file the
    kernel does not include, leaves the compiled kernel, and so the ncu
    counters taken on it, as they were."""
    h = hashlib.sha256()
    for f in kernel_sources(kernel):
        with open(f, encoding="utf-8") as fh:
            text = fh.read()
        code = _TOKENS.sub(lambda m: " " if m.group(0).startswith("/") else m.group(0), text)
        h.update(os.path.basename(f).encode() + b"\0" + " ".join(code.split()).encode() + b"\0")
    return h.hexdigest()[:12]


def read_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes from a committed ncu summary line of the form
    'bench-traffic: workload=W kernel=K bytes=N src=H scale=S', or None when
    absent or taken on other sources of that kernel."""
    if kernel not in KERNEL_FILES:
        return None
    cur = src_hash(kernel)
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(f):
            if not line.startswith("bench-traffic:"):
                continue
            kv = dict(x.split("=", 1) for x in line.split()[1:] if "=" in x)
            if kv.get("workload") == workload and kv.get("kernel") == kernel and kv.get("src") == cur:
                return float(kv["bytes"]) * float(kv.get("scale", "1"))
    return None


class ClockSampler:
    """nvidia-smi samples (200 ms) of the GPU that torch uses."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower().replace("gpu-", "")
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True, bufsize=1)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if self.uuid and self.uuid not in parts[1].lower():
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 <= ts <= t1]
        use = inside or [p for ts, p in rows if t0 - 1.0 <= ts <= t1 + 1.0]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for p in use if num(p[2]) is not None]
        reasons = set()
        for p in use:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max((num(p[3]) or 0) for p in use) if use else None,
                "power_w_max": max((num(p[4]) or 0) for p in use) if use else None,
                "reasons": sorted(reasons), "samples_in_window": len(inside),
                "samples_used": len(use)}


# ------------------------------------------------------------ distributed --

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as td
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        td.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as td
        td.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as td
    dev = "cuda" if td.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- GPU arm --

class Rotation:
    """R rotation steps over one page pool of the workload's own layout.

    Step i reads its own set of physical pages, disjoint from every other
    step's and holding a copy of the problem's page data, and its own copy of
    q, so no call finds its K/V or q in L2 from an earlier call while the
    results stay the same.  The pool keeps the workload's page count unless
    R sets of used pages need more; the sets are drawn from one seeded
    Fisher-Yates shuffle of the pool (consecutive page ids when the workload's
    table is the identity)."""

    TID_ROTATION = 5  # generator stream of the rotation's page shuffle

    def __init__(self, wl, inp, R, ops, torch):
        import numpy as np
        from paged_kv_gqa_02_gb300 import inputs
        base = ops.device_inputs(inp, wl)
        bt0 = np.asarray(inp["block_tables"])
        npg0 = int(inp["num_pages"])
        used = np.unique(bt0[bt0 >= 0]).astype(np.int64)
        U = len(used)
        pool = max(npg0, R * U)
        order = (inputs.fisher_yates(pool, inputs.stream_seed(wl.seed, self.TID_ROTATION))
                 if wl.shuffle else np.arange(pool, dtype=np.int64))
        k0, v0 = base["k_cache"], base["v_cache"]
        self.k = torch.zeros((pool,) + tuple(k0.shape[1:]), dtype=k0.dtype, device="cuda")
        self.v = torch.zeros_like(self.k)
        src = torch.as_tensor(used, device="cuda")
        self.R = R
        self.pool_pages = pool
        self.q = [base["q"].clone() for _ in range(R)]
        self.bt = []
        for i in range(R):
            dst = np.asarray(order[i * U:(i + 1) * U], dtype=np.int64)
            dst_t = torch.as_tensor(dst, device="cuda")
            self.k[dst_t] = k0[src]
            self.v[dst_t] = v0[src]
            remap = np.full(npg0, -1, dtype=np.int64)
            remap[used] = dst
            t = np.where(bt0 >= 0, remap[np.clip(bt0, 0, None)], bt0).astype(np.int32)
            self.bt.append(torch.as_tensor(t, device="cuda"))
        self.cl = base["context_lens"]
        self.cu = base["cu_q_lens"]
        self.params = ops.params_for(wl, num_pages=pool)
        self.out = torch.empty((wl.total_q, wl.num_q_heads, wl.head_dim), dtype=torch.float32,
                               device="cuda")


def rotation_copies(wl, l2_bytes, cap=256):
    foot = wl.kv_bytes() + wl.q_bytes() + wl.o_bytes()
    return max(2, min(cap, math.ceil(3 * l2_bytes / foot)))


def time_graph(torch, calls, K, W, world):
    """Warm up W calls, capture a graph of len(calls) calls, replay it so that
    exactly K calls run in the timed region; returns (ms total, t0, t1)."""
    s = torch.cuda.Stream()
    R = len(calls)
    with torch.cuda.stream(s):
        for i in range(W):
            calls[i % R](s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c(s)
    rem = K % R
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=s):
            for c in calls[:rem]:
                c(s)
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(K // R):
            g.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(s)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    return e0.elapsed_time(e1), t0, t1


def decode_calls(rot, ops, torch, partial_only=False, form=0):
    """pa_decode calls over the rotation copies in decode form `form`
    (PA_FORM_AUTO, PA_FORM_PAIR or PA_FORM_COUNTED); with partial_only, the
    pair's partial kernel alone (decode_phases = 1)."""
    import copy
    p = copy.copy(rot.params)
    p.decode_phases = 1 if partial_only else 0
    p.decode_form = ops.PA_FORM_PAIR if partial_only else form
    S, _ = ops.decode_plan(p)
    nws = ops.decode_workspace_size(p)
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device="cuda")
    calls = [lambda s, i=i: ops.decode(p, rot.q[i], rot.k, rot.v, rot.bt[i], rot.cl, out=rot.out,
                                       workspace=ws if nws else None, stream=s)
             for i in range(rot.R)]
    if partial_only:
        launches = 1
    elif p.num_splits == 0 and p.kv_dtype != ops.PA_F32:
        launches = 1 if single_launch(p) else 2
    else:
        launches = 2 if S > 1 else 1
    return calls, launches, S


def single_launch(p) -> bool:
    """Whether pa_decode runs these parameters as one kernel: the counted
    form, 16-bit K/V, automatic splits, head_dim <= 128, one MMA column tile
    (query rows x q heads per kv head <= 8)."""
    from paged_kv_gqa_02_gb300 import ops
    rows = max(1, p.decode_q_rows)
    g = p.num_q_heads // p.num_kv_heads
    rb = min(rows, (8 if p.head_dim == 256 else 16) // g)
    if not (p.num_splits == 0 and p.kv_dtype != ops.PA_F32 and p.head_dim <= 128 and rb * g <= 8
            and p.decode_phases in (0, 3)):
        return False
    return p.decode_form == ops.PA_FORM_COUNTED


def append_calls(rot, wl, ops, torch):
    """pa_decode_append over the rotation: each step also writes its
    sequences' new K/V rows (the same rows every replay) into its pages."""
    from paged_kv_gqa_02_gb300 import inputs
    k_new, v_new = inputs.make_append_rows(num_seqs=wl.num_seqs, num_kv_heads=wl.num_kv_heads,
                                           head_dim=wl.head_dim, kv_dtype=wl.kv_dtype, seed=wl.seed)
    kn, vn = ops.to_device(k_new, wl.kv_dtype), ops.to_device(v_new, wl.kv_dtype)
    p = rot.params
    nws = ops.decode_workspace_size(p)
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device="cuda")
    return [lambda s, i=i: ops.decode_append(p, rot.q[i], kn, vn, rot.k, rot.v, rot.bt[i], rot.cl, out=rot.out,
                                             workspace=ws if nws else None, stream=s)
            for i in range(rot.R)]


def rows_calls(rot, wl, ops, torch, T):
    """pa_decode with T query rows per sequence (decode_q_rows) over the
    rotation; lengths below T are raised to T (the pages hold those keys)."""
    import copy
    from paged_kv_gqa_02_gb300 import inputs
    p = copy.copy(rot.params)
    p.decode_q_rows = T
    q = ops.to_device(inputs.normal_tensor(wl.seed, 8, (wl.num_seqs * T, wl.num_q_heads, wl.head_dim),
                                           wl.q_dtype), wl.q_dtype)
    cl = torch.clamp(rot.cl, min=T)
    out = torch.empty((wl.num_seqs * T, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    nws = ops.decode_workspace_size(p)
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device="cuda")
    return [lambda s, i=i: ops.decode(p, q, rot.k, rot.v, rot.bt[i], cl, out=out,
                                      workspace=ws if nws else None, stream=s)
            for i in range(rot.R)]


def window_calls(rot, wl, ops, torch, W):
    """pa_decode with a W-key sliding window over the rotation."""
    import copy
    p = copy.copy(rot.params)
    p.sliding_window = W
    nws = ops.decode_workspace_size(p)
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device="cuda")
    return [lambda s, i=i: ops.decode(p, rot.q[i], rot.k, rot.v, rot.bt[i], rot.cl, out=rot.out,
                                      workspace=ws if nws else None, stream=s)
            for i in range(rot.R)]


def prefill_calls(rot, wl, ops, torch):
    p = rot.params
    calls = [lambda s, i=i: ops.prefill_chunk(p, rot.q[i], rot.cu, wl.total_q, max(wl.q_lens), rot.k,
                                              rot.v, rot.bt[i], rot.cl, out=rot.out, stream=s)
             for i in range(rot.R)]
    return calls, 1


def e2e_decode(wl, inp, ops, torch, steps):
    """Same metric through the public API with pinned host buffers: each step
    copies the inputs host->device, runs pa_decode and copies out back."""
    import numpy as np
    host = {}
    for name in ("q", "k_cache", "v_cache", "block_tables", "context_lens"):
        dt_ = wl.q_dtype if name == "q" else (wl.kv_dtype if "cache" in name else None)
        t = ops.to_device(inp[name], dt_, device="cpu").pin_memory()
        host[name] = t
    dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}
    p = ops.params_for(wl)
    out_d = torch.empty((wl.total_q, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    out_h = torch.empty_like(out_d, device="cpu").pin_memory()
    nws = ops.decode_workspace_size(p)
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step():
        with torch.cuda.stream(s):
            for k in dev:
                dev[k].copy_(host[k], non_blocking=True)
            ops.decode(p, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                       dev["context_lens"], out=out_d, workspace=ws if nws else None, stream=s)
            out_h.copy_(out_d, non_blocking=True)
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        step()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    return ms, h2d, d2h


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def _row_block(inp, s, r0, r1):
    """Rows [r0, r1) of sequence s of a prefill batch as a problem of their
    own over the same pool: the last r1 - r0 rows of a context that ends at
    row r1 - 1, so each row sees exactly the keys it sees in the batch."""
    import numpy as np
    cu, cl = inp["cu_q_lens"], inp["context_lens"]
    T = int(cu[s + 1] - cu[s])
    out = dict(inp)
    out["q"] = inp["q"][int(cu[s]) + r0:int(cu[s]) + r1]
    out["cu_q_lens"] = np.array([0, r1 - r0], dtype=cu.dtype)
    out["context_lens"] = np.array([int(cl[s]) - T + r1], dtype=cl.dtype)
    out["block_tables"] = inp["block_tables"][s:s + 1]
    return out


def cpu_baseline(wl, inp, seconds):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload, timed twice: on one thread and on every core the process may
    use (OpenMP over rows x heads), each for about half of `seconds`.
    Decode: whole calls.  Prefill: on one thread, single (row, head)
    distributions drawn at random; on all cores, blocks of 64 consecutive
    rows of one sequence with all their heads.  `value` and `cores` are the
    all-core run's."""
    import numpy as np
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    affinity = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None
    per_key = wl.algorithmic_bytes() / (wl.visible_keys() * wl.num_q_heads)
    rng = np.random.default_rng(0)

    def run(threads, budget):
        t0 = time.perf_counter()
        n, keys = 0, 0
        while True:
            if wl.kind == "decode":
                oracle.attention(inp, wl, threads=threads)
            elif threads == 1:
                r, h = int(rng.integers(0, wl.total_q)), int(rng.integers(0, wl.num_q_heads))
                s = int(np.searchsorted(inp["cu_q_lens"], r, side="right") - 1)
                oracle.attention_rows(inp, [(r, h)], wl)
                cu, cl = inp["cu_q_lens"], inp["context_lens"]
                keys += int(cl[s] - (cu[s + 1] - cu[s]) + (r - cu[s]) + 1)
            else:
                s = n % wl.num_seqs
                T = wl.q_lens[s]
                r0 = (n // wl.num_seqs * 64) % T
                blk = _row_block(inp, s, r0, min(T, r0 + 64))
                _, k = oracle.attention(blk, wl, threads=threads, return_keys=True)
                keys += k
            n += 1
            if time.perf_counter() - t0 >= budget:
                break
        el = time.perf_counter() - t0
        # prefill: `keys` counts (row, head, key) terms, as per_key's denominator does
        return (wl.algorithmic_bytes() * n if wl.kind == "decode" else per_key * keys) / el / 1e9, n, el

    unit1, unita = ("calls", "calls") if wl.kind == "decode" else \
        ("(row, head) distributions", "64-row blocks (all heads)")
    v1, n1, e1 = run(1, seconds / 2)
    va, na, ea = run(cores, seconds / 2)
    return {"value": va, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{na} {unita} of {wl.name} on {cores} threads ({ea:.1f} s); "
                      f"{n1} {unit1} on 1 thread ({e1:.1f} s) (fp64)",
            "single_thread": {"value": v1, "unit": "GB/s", "sample": f"{n1} {unit1}"},
            "all_cores": {"value": va, "unit": "GB/s", "threads": cores, "sample": f"{na} {unita}"},
            "cpu_model": cpu_model(), "affinity_cores": affinity, "os_cpu_count": os.cpu_count()}


def measure_workload(wl, ops, torch, K, W, world, l2, hbm_peak, flop_peak, clocks=None):
    inp = wl.make_inputs()
    R = rotation_copies(wl, l2)
    rot = Rotation(wl, inp, R, ops, torch)
    res = {"workload": wl.name, "rotation_copies": R, "pool_pages": rot.pool_pages}
    if wl.kind == "decode":
        calls, launches, S = decode_calls(rot, ops, torch)
        ms, t0, t1 = time_graph(torch, calls, K, W, world)
        ms = max_over_ranks(ms, world)
        # the partial step alone (decode_phases = 1: the split partial kernel
        # of the two-kernel form)
        pcalls, _, _ = decode_calls(rot, ops, torch, partial_only=True)
        pms, _, _ = time_graph(torch, pcalls, K, W, world)
        pms = max_over_ranks(pms, world)
        per_call = ms / K
        part = pms / K
        if launches == 1:
            # one kernel per call: its average launch period is the call's,
            # and it moves every algorithmic byte (K/V, q and out)
            dom_name, dom_ms, dom_bytes = "decode (one kernel)", per_call, wl.algorithmic_bytes()
        else:
            dom_name, dom_ms, dom_bytes = "decode split partial", part, wl.kv_bytes() + wl.q_bytes()
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
        for form, key in ((ops.PA_FORM_PAIR, "pair"), (ops.PA_FORM_COUNTED, "counted")):
            fcalls, flaunches, _ = decode_calls(rot, ops, torch, form=form)
            if form == ops.PA_FORM_PAIR and launches == 2:
                continue  # the main measurement is the pair already
            if form == ops.PA_FORM_COUNTED and flaunches != 1:
                continue
            fms, _, _ = time_graph(torch, fcalls, K, W, world)
            res[f"{key}_us_per_call"] = max_over_ranks(fms, world) / K * 1e3
        ams, _, _ = time_graph(torch, append_calls(rot, wl, ops, torch), K, W, world)
        res["append_us_per_call"] = max_over_ranks(ams, world) / K * 1e3
        for T in (2, 4):
            tms, _, _ = time_graph(torch, rows_calls(rot, wl, ops, torch, T), K, W, world)
            res[f"rows{T}_us_per_call"] = max_over_ranks(tms, world) / K * 1e3
        if wl.kv_dtype != "f32":  # windows run on the split-KV kernel only
            wms, _, _ = time_graph(torch, window_calls(rot, wl, ops, torch, 1024), K, W, world)
            res["window1024_us_per_call"] = max_over_ranks(wms, world) / K * 1e3
            wbytes = sum(min(L, 1024) for L in wl.context_lens) * 2 * wl.num_kv_heads * wl.head_dim * \
                wl.elt(wl.kv_dtype) + wl.q_bytes() + wl.o_bytes()
            res["window1024_gbs"] = wbytes / (res["window1024_us_per_call"] * 1e-6) / 1e9
        res.update(num_splits=S, launches_per_call=launches, ms_total=ms, us_per_call=per_call * 1e3,
                   gbs=wl.algorithmic_bytes() / (per_call * 1e-3) / 1e9,
                   frac_of_hbm=wl.algorithmic_bytes() / (per_call * 1e-3) / 1e9 / hbm_peak,
                   partial_only_us=part * 1e3,
                   dominant={"kernel": dom_name, "us_per_launch": dom_ms * 1e3,
                             "algorithmic_bytes": dom_bytes, "achieved_gbs": achieved,
                             "frac": achieved / hbm_peak}, t0=t0, t1=t1)
    else:
        calls, launches = prefill_calls(rot, wl, ops, torch)
        ms, t0, t1 = time_graph(torch, calls, K, W, world)
        ms = max_over_ranks(ms, world)
        per_call = ms / K
        tflops = wl.flops() / (per_call * 1e-3) / 1e12
        res.update(launches_per_call=launches, ms_total=ms, us_per_call=per_call * 1e3,
                   tflops=tflops, frac_of_tensor_peak=tflops / flop_peak,
                   gbs=wl.algorithmic_bytes() / (per_call * 1e-3) / 1e9, t0=t0, t1=t1)
    return res, inp


def run_ours(args):
    import torch
    from paged_kv_gqa_02_gb300 import build, ops, workloads
    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    build.build()
    ops.load()
    hbm, bf16, bf16_sus, peak_src = peaks()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    wl = workloads.BY_NAME[args.workload]
    K, W = args.steps, max(3, args.warmup)
    if wl.kind == "prefill":
        K = min(K, 200)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    time.sleep(0.5)
    # the prefill kernel is timed alone in a short burst of calls: the burst bf16 peak applies
    main, inp = measure_workload(wl, ops, torch, K, W, world, l2, hbm, bf16)
    time.sleep(0.3)
    sampler.stop()
    clocks = sampler.summary(main.pop("t0"), main.pop("t1"))
    secondary = {}
    if not args.no_secondary:
        for other in workloads.ALL + workloads.EXTRA:
            if other.name == wl.name:
                continue
            k2 = 2000 if other.kind == "decode" else 20
            r, _ = measure_workload(other, ops, torch, k2, 10, world, l2, hbm, bf16)
            r.pop("t0"), r.pop("t1")
            secondary[other.name] = r
    e2e_ms, h2d, d2h = (None, 0, 0)
    if wl.kind == "decode":
        e2e_ms, h2d, d2h = e2e_decode(wl, inp, ops, torch, args.e2e_steps)
        e2e_ms = max_over_ranks(e2e_ms, world)
    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baseline(wl, inp, args.cpu_seconds)
    if rank != 0:
        return
    per_call_ms = main["ms_total"] / K
    value = wl.algorithmic_bytes() * K * world / (main["ms_total"] * 1e-3) / 1e9
    dom = main.get("dominant")
    if dom:
        traffic = read_traffic(wl.name, "decode_v1")
        roof = {"bound": "hbm", "achieved": round(dom["achieved_gbs"], 1), "peak": hbm,
                "unit": "GB/s", "frac": round(dom["achieved_gbs"] / hbm, 4),
                "traffic": traffic, "peak_source": f"{peak_src} (hbm_gbs, copy)",
                "kernel": dom["kernel"], "us_per_launch": round(dom["us_per_launch"], 3),
                "algorithmic_bytes_per_launch": dom["algorithmic_bytes"],
                "partial_step_alone_us": round(main["partial_only_us"], 3)}
    else:
        roof = {"bound": "tensor", "achieved": round(main["tflops"], 1), "peak": bf16,
                "unit": "TFLOP/s", "frac": round(main["tflops"] / bf16, 4),
                "traffic": read_traffic(wl.name, "prefill_tc"),
                "peak_source": f"{peak_src} (bf16_tflops, burst: the kernel is timed alone in short bursts)",
                "kernel": "prefill_tc"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(per_call_ms, 6), "us_per_call": round(per_call_ms * 1e3, 3),
        "frac_of_hbm_peak": round(per_call_ms and wl.algorithmic_bytes() / (per_call_ms * 1e-3) / 1e9 / hbm, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.kv_dtype,
        "data": "synthetic (seeded N(0,1), shuffled 4096-page pool)",
        "config": {"workload": wl.name, "kind": wl.kind, "num_seqs": wl.num_seqs,
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "page_size": wl.page_size,
                   "context_tokens": sum(wl.context_lens), "num_splits": main.get("num_splits"),
                   "algorithmic_bytes_per_call": wl.algorithmic_bytes(),
                   "l2": f"inputs larger than L2: rotation over {main['rotation_copies']} disjoint page "
                         f"sets of one {main['pool_pages']}-page pool (>= 3x the {l2 // 2**20} MiB L2)",
                   "timing": "CUDA graph replays, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "decode_append_us_per_call": round(main["append_us_per_call"], 3) if "append_us_per_call" in main else None,
        "decode_forms_us_per_call": {k: round(main[f"{k}_us_per_call"], 3) for k in ("pair", "counted")
                                     if f"{k}_us_per_call" in main},
        "decode_rows_us_per_call": {T: round(main[f"rows{T}_us_per_call"], 3) for T in (2, 4)
                                    if f"rows{T}_us_per_call" in main},
        "decode_window1024": {"us_per_call": round(main["window1024_us_per_call"], 3),
                              "gbs": round(main["window1024_gbs"], 1)} if "window1024_us_per_call" in main else None,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": None if e2e_ms is None else {
            "value": round(wl.algorithmic_bytes() / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "pinned host q, full K/V pools, tables, lengths copied every step"},
        "gpu_launches": K * main["launches_per_call"],
        "clocks": clocks,
        "workloads": secondary,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------- reference arm --

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import numpy as np
    import oracle
    from paged_kv_gqa_02_gb300 import workloads
    oracle.build()
    wl = workloads.BY_NAME[args.workload]
    inp = wl.make_inputs()
    K, W = args.steps, max(3, args.warmup)
    # each step: a bounded sample of (row, head) distributions, sized so the
    # whole run stays near a minute of CPU time
    rng = np.random.default_rng(0)
    rows = np.arange(wl.total_q)
    per_key = wl.algorithmic_bytes() / (wl.visible_keys() * wl.num_q_heads)
    cu, cl = inp["cu_q_lens"], inp["context_lens"]

    def keys_of(r):
        s = int(np.searchsorted(cu, r, side="right") - 1)
        return int(cl[s] - (cu[s + 1] - cu[s]) + (r - cu[s]) + 1)
    t = time.perf_counter()
    oracle.attention_rows(inp, [(int(rows[-1]), 0)], wl)
    one = max(time.perf_counter() - t, 1e-6)
    n_per_step = max(1, int(60.0 / (K * one)))
    picks = [(int(rng.integers(0, wl.total_q)), int(rng.integers(0, wl.num_q_heads)))
             for _ in range(n_per_step * (K + W))]
    for i in range(W):
        oracle.attention_rows(inp, picks[i * n_per_step:(i + 1) * n_per_step], wl)
    t0 = time.perf_counter()
    keys = 0
    for i in range(W, W + K):
        sel = picks[i * n_per_step:(i + 1) * n_per_step]
        oracle.attention_rows(inp, sel, wl)
        keys += sum(keys_of(r) for r, _ in sel)
    el = time.perf_counter() - t0
    value = per_key * keys / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(el / K * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), shuffled 4096-page pool)",
        "config": {"workload": wl.name, "kind": wl.kind, "parallelism": "rank 0 only"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n_per_step} random (row, head) distributions per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ncu_once(args):
    """A short, graph-free run for ncu: `warmup` calls, then one call, on a
    single copy of the inputs (ncu flushes caches between replays itself)."""
    import torch
    from paged_kv_gqa_02_gb300 import build, ops, workloads
    build.build()
    wl = workloads.BY_NAME[args.workload]
    inp = wl.make_inputs()
    d = ops.device_inputs(inp, wl)
    p = ops.params_for(wl)
    out = torch.empty((wl.total_q, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    nws = ops.decode_workspace_size(p) if wl.kind == "decode" else 0
    ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device="cuda") if nws else None  # once, not per call
    for _ in range(args.warmup + 1):
        if wl.kind == "decode":
            ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], out=out,
                       workspace=ws)
        else:
            ops.prefill_chunk(p, d["q"], d["cu_q_lens"], wl.total_q, max(wl.q_lens), d["k_cache"],
                              d["v_cache"], d["block_tables"], d["context_lens"], out=out)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_once": wl.name, "calls": args.warmup + 1}))


def main():
    args = parse_args()
    if args.ncu_once:
        run_ncu_once(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
