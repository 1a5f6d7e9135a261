#!/usr/bin/env python
"""Benchmark of tree-verify attention over a paged MLA latent pool (one GB300).

Metric: verify-attention microseconds per call, with TFLOP/s, KV GB/s and the
fraction of the roofline max(FLOPs / bf16 peak, bytes / HBM bandwidth).

One step = one full call of the hot path (status clear, split kernels, split
combine) on one batch of the headline workload, inputs resident in HBM, run
as a serving loop runs it: one call captured once in a CUDA graph and
replayed.  L2 is flushed (a 256 MiB write) before every timed replay; each
replay is timed with CUDA events around it, and the library's own phase
events, captured inside the graph, give the split and combine times.  The
line also carries the same call launched directly (cold and warm) and end to
end from pinned host buffers.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config ragged|long|mid|short|tiny] [--kernel tc|simt]

The path runs on one GPU.  More than one GPU (``--gpus N > 1`` or a torchrun
world larger than one) is refused before CUDA is touched: rank 0 prints a
JSON line with an ``unavailable`` reason, every rank exits 0, and nothing is
launched.  The tensor-core kernel's 4-CTA clusters issue TMA loads with
cluster multicast, which this library keeps to single-GPU calls.
``--impl reference`` times the CPU oracle on the host cores (rank 0 only;
other ranks exit 0 at once).
"""
from __future__ import annotations

import argparse
import copy
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-attn µs/call, TFLOP/s and KV GB/s as % of GB300 roofline (1 GPU)"
UNIT = "us/call"
HEADLINE = "ragged"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
CLOCK_HOLD_S = 1.0          # the timed replays' load is held this long for the 200 ms clock sampler
KERNEL_SOURCES = {"tc": "speculative_decode_mla_paged_gb300/csrc/verify_tc.cu",
                  "simt": "speculative_decode_mla_paged_gb300/csrc/verify_simt.cu"}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--kernel", choices=["tc", "simt"], default="tc")
    ap.add_argument("--num-splits", type=int, default=0, help="0 = per-config default")
    ap.add_argument("--no-per-config", action="store_true", help="skip the five-config table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle timings")
    ap.add_argument("--cpu-seconds", type=float, default=None,
                    help="accepted for older profile commands; the oracle is now timed on whole calls")
    ap.add_argument("--launch-only", action="store_true",
                    help="for profilers: W warm-up and K timed direct calls of the workload, nothing else")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def choose_splits(inp, d, kernel):
    """Split count for this workload and how it was chosen: the tensor-core
    path times the four best candidates of the grid simulation as cold
    CUDA-graph replays (api.tune_num_splits) and keeps the fastest; the
    CUDA-core path takes the simulation's pick."""
    from speculative_decode_mla_paged_gb300 import api, tuning
    if kernel != "tc":
        return tuning.plan_num_splits(inp.prefix_lens, inp.draft_lens, inp.num_heads, kernel), "simulated"
    cands = tuning.ranked_num_splits(inp.prefix_lens, inp.draft_lens, inp.num_heads, k=4)
    s = api.tune_num_splits(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                            d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], inp.sm_scale, d["out"],
                            inp.max_q_per_req, cands)
    return s, f"fastest of {cands} timed as graph replays (simulated ranking)"


def code_text(src: str) -> str:
    """C++/CUDA source without comments and whitespace: what the compiler sees."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] == '"':                      # string literal, kept as written
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            if not src[i].isspace():
                out.append(src[i])
            i += 1
    return "".join(out)


def kernel_hash(kernel):
    """First 12 hex digits of the SHA-1 of the kernel source's code text
    (comments and whitespace removed, so an edit to a comment keeps a
    capture valid)."""
    with open(os.path.join(ROOT, KERNEL_SOURCES[kernel]), encoding="utf-8") as f:
        return hashlib.sha1(code_text(f.read()).encode()).hexdigest()[:12]


def profiled_traffic(kernel, cfg_name):
    """DRAM bytes of the split phase of one call (all its split launches) from
    a committed ncu summary for this exact kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    if not os.path.exists(path):
        return None
    h = kernel_hash(kernel)
    for line in open(path):
        m = re.match(r"\|\s*(\w+)\s*\|\s*(\w+)\s*\|\s*([0-9a-f]{12})\s*\|\s*([0-9.e+]+)\s*\|", line)
        if m and m.group(1) == kernel and m.group(2) == cfg_name and m.group(3) == h:
            return float(m.group(4))
    return None


# Issued tensor-core work per MMA instruction of the tensor-core kernel: every
# 128-key tile of 128 rows takes 36 score MMAs (M128 N128 K16) and 16 P V
# MMAs (M128 N256 K16), always in that ratio, so FLOPs per instruction
# average out to this over any whole number of tiles.
TC_FLOP_PER_MMA_INST = (36 * 2 * 128 * 128 * 16 + 16 * 2 * 128 * 256 * 16) / 52


def profiled_tensor_pipe(kernel, cfg_name):
    """Tensor-pipe counters of the split phase of one call (all its split
    launches) from a committed ncu summary for this exact kernel source:
    {"active_cycles": sm__pipe_tensor_cycles_active.sum, "units": the number
    of instances that sum runs over, "mma_inst": sm__inst_executed_pipe_tensor.sum},
    or None."""
    path = os.path.join(ROOT, "profiles", "tensor_pipe.md")
    if not os.path.exists(path):
        return None
    h = kernel_hash(kernel)
    num = r"\s*([0-9.e+]+)\s*\|"
    for line in open(path):
        m = re.match(r"\|\s*(\w+)\s*\|\s*(\w+)\s*\|\s*([0-9a-f]{12})\s*\|" + num * 3, line)
        if m and m.group(1) == kernel and m.group(2) == cfg_name and m.group(3) == h:
            return {"active_cycles": float(m.group(4)), "units": float(m.group(5)), "mma_inst": float(m.group(6))}
    return None


def tensor_pipe_summary(counters, split_s, sm_mhz, flops):
    """What the counters say about the timed split phase: the share of the
    tensor pipes' cycles in which they were active (counter cycles over
    instances x split-phase time x the sampled SM clock), the issued MMA FLOPs
    and their ratio to the algorithmic FLOPs (the padding of partial and
    masked tiles and of rows past a request's end)."""
    if counters is None or not split_s or not sm_mhz:
        return None
    issued = counters["mma_inst"] * TC_FLOP_PER_MMA_INST
    return {"active_frac": counters["active_cycles"] / (counters["units"] * split_s * sm_mhz * 1e6),
            "issued_flops": issued, "issued_over_algorithmic": issued / flops,
            "source": "profiles/tensor_pipe.md (ncu, same kernel source)"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_index is not None:
            cmd += ["-i", str(self.gpu_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, window=None):
        """Stop sampling; summarise the samples read inside `window` = (t0, t1)
        (wall-clock seconds), or all of them when no window is given."""
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return summarise_clocks(self.lines, window)


def _clock_stats(lines):
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for _, line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1])); mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


def summarise_clocks(lines, window=None):
    """Median SM clock, max clock and throttle reasons of nvidia-smi CSV lines
    [(read time, text)].  With a load `window` = (t0, t1) only the lines read
    inside it (its end stretched by one 200 ms period) count, and `window_s`
    gives its length; if no line was read inside it (output that reached the
    pipe late), every line counts and `window_s` is null."""
    if window is not None:
        out = _clock_stats([(ts, ln) for ts, ln in lines if window[0] <= ts <= window[1] + 0.2])
        if out is not None:
            out["window_s"] = round(window[1] - window[0], 3)
            return out
    out = _clock_stats(lines)
    if out is not None and window is not None:
        out["window_s"] = None
    return out


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, world, device=None):
    """The largest of the ranks' values: the job takes as long as its slowest
    replica.  With one rank, the value itself (no process group needed)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def per_call_us(total_ms, steps, world):
    """Whole-job time per call: every rank ran `steps` calls in `total_ms`."""
    return total_ms * 1e3 / (steps * world)


# ------------------------------------------------------------------ oracle (CPU) timing

def visible_per_row(inp):
    """Visible keys of every output row (t*H + h), from the packed mask."""
    bits = np.unpackbits(inp.custom_mask, bitorder="little")
    counts = []
    for b in range(inp.batch):
        T = int(inp.draft_lens[b]); N = int(inp.prefix_lens[b]) + T
        m0 = int(inp.mask_indptr[b])
        rows = bits[m0:m0 + T * N].reshape(T, N).sum(axis=1) if T else np.zeros(0)
        counts.append(np.repeat(rows, inp.num_heads))
    return np.concatenate(counts).astype(np.int64)


def time_oracle(inp, seconds, seed=0):
    """Run the oracle on a row sample sized to ~`seconds` of CPU work and scale
    to microseconds per full call by visible (row, key) pairs."""
    import oracle
    vis = visible_per_row(inp)
    total_pairs = float(vis.sum())
    rng = np.random.default_rng(seed)
    order = rng.permutation(len(vis))
    t0 = time.perf_counter()
    oracle.run(inp, rows=order[:1])
    one = max(time.perf_counter() - t0, 1e-4)
    per_pair = one / max(vis[order[0]], 1) / max(1, oracle.num_threads())
    want_pairs = seconds / per_pair
    csum = np.cumsum(vis[order])
    n = int(min(len(vis), max(oracle.num_threads(), np.searchsorted(csum, want_pairs) + 1)))
    rows = np.sort(order[:n])
    t0 = time.perf_counter()
    oracle.run(inp, rows=rows)
    dt = time.perf_counter() - t0
    pairs = float(vis[rows].sum())
    us_per_call = dt * 1e6 * total_pairs / max(pairs, 1.0)
    return us_per_call, {"rows": int(n), "of_rows": int(len(vis)), "seconds": round(dt, 3),
                         "pairs": int(pairs), "of_pairs": int(total_pairs)}


def cpu_model() -> str:
    """The host CPU's model name (x86: /proc/cpuinfo; Arm: lscpu), or '' if unknown."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def time_oracle_call(inp, threads=None):
    """Wall seconds of one whole oracle call (every output row) on `threads`
    host threads (None: all of them)."""
    import oracle
    cores = oracle.num_threads()
    if threads is not None:
        oracle.set_num_threads(threads)
    try:
        t0 = time.perf_counter()
        oracle.run(inp)
        return time.perf_counter() - t0
    finally:
        if threads is not None:
            oracle.set_num_threads(cores)


def oracle_timings(inp, single_core_budget_s=20.0):
    """The oracle on this host for one workload: a whole call on all cores,
    and on one core either a whole call (when the all-core time x cores
    predicts at most `single_core_budget_s`) or a row sample of about 4 s
    scaled to a full call by visible (row, key) pairs, labelled as such."""
    import oracle
    cores = oracle.num_threads()
    all_s = time_oracle_call(inp)
    rec = {"all_cores_s": all_s, "cores": cores, "rows": int(inp.total_q * inp.num_heads)}
    if all_s * cores <= single_core_budget_s:
        rec["single_core_s"] = time_oracle_call(inp, threads=1)
        rec["single_core_how"] = "whole call"
    else:
        oracle.set_num_threads(1)
        try:
            us, sample = time_oracle(inp, 4.0, seed=1)
        finally:
            oracle.set_num_threads(cores)
        rec["single_core_s"] = us / 1e6
        rec["single_core_how"] = (f"row sample: {sample['rows']} of {sample['of_rows']} rows in "
                                  f"{sample['seconds']} s, scaled by visible (row, key) pairs")
    return rec


def reference_inputs(config):
    """The workload's inputs on the host (large pools are drawn on the GPU
    when one is present, as our arm draws them, then copied)."""
    from speculative_decode_mla_paged_gb300 import workloads as W
    if config in ("tiny", "short"):
        return W.make_config_inputs(config, device="cpu")
    import torch
    if torch.cuda.is_available():
        inp = W.make_config_inputs(config, device="cuda")
        inp.q, inp.kv_pool = inp.q.cpu(), inp.kv_pool.cpu()
        torch.cuda.empty_cache()
        return inp
    return W.make_config_inputs(config, device="cpu")


REFERENCE_BUDGET_S = 150.0


def run_reference(args):
    """The oracle, as it stands, on the host cores: whole calls of the
    workload (every output row), as many of the requested W + K as fit in
    about REFERENCE_BUDGET_S; the line reports the counts actually run."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    import oracle
    from speculative_decode_mla_paged_gb300 import workloads as W
    oracle.build()
    inp = reference_inputs(args.config)
    t_begin = time.perf_counter()
    warm = [time_oracle_call(inp)]          # one untimed whole call, which also sizes the run
    per_call = warm[0]
    left = REFERENCE_BUDGET_S - (time.perf_counter() - t_begin)
    steps = max(1, min(args.steps, int(left // max(per_call, 1e-6))))
    vals = [time_oracle_call(inp) for _ in range(steps)]
    value = statistics.mean(vals) * 1e6
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": len(warm), "steps_requested": args.steps, "warmup_requested": args.warmup,
        "ms_per_step": value / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.config}: {W.CONFIGS[args.config].description}", "name": args.config},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"whole calls (all {inp.total_q * inp.num_heads} output rows): {len(warm)} "
                                   f"untimed, then {steps} timed, of the {args.warmup} + {args.steps} requested "
                                   f"(whole calls bounded to about {REFERENCE_BUDGET_S:.0f} s)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def measure(inp, d, runner, steps, warmup, flush, torch):
    """Device timing of `steps` calls, each after an L2 flush.  Returns per-step
    lists of (call_ms, split_ms, combine_ms)."""
    from speculative_decode_mla_paged_gb300 import api  # noqa: F401
    out = d["out"]
    stream = torch.cuda.current_stream()

    def call(events=None):
        runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
               d["custom_mask"], d["mask_indptr"], inp.sm_scale, out, events=events)

    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for k in range(steps):
        flush.zero_()
        call(evs[k])
    torch.cuda.synchronize()
    call_ms = [e[0].elapsed_time(e[3]) for e in evs]
    split_ms = [e[1].elapsed_time(e[2]) for e in evs]
    comb_ms = [e[2].elapsed_time(e[3]) for e in evs]
    return call_ms, split_ms, comb_ms


def launches_per_call(inp, kernel):
    """Library kernels per call: the split kernel(s) and the combine.  The
    tensor-core path launches both cluster shapes (on two streams) when the
    capacity T * H exceeds one 128-row tile and H does not."""
    rows = inp.max_q_per_req * inp.num_heads
    both = kernel == "tc" and rows > 128 and inp.num_heads <= 128
    return 3 if both else 2


def measure_warm(inp, d, runner, steps, torch):
    """Device time per call of `steps` back-to-back calls with no L2 flush
    (inputs partly L2-resident from the previous call)."""
    def call():
        runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
               d["custom_mask"], d["mask_indptr"], inp.sm_scale, d["out"])

    call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


def measure_graph(inp, d, runner, steps, warmup, flush, torch, hold_s=0.0):
    """Cold replays of one call captured in a CUDA graph (how a serving loop
    runs it), each after an L2 flush outside the timed events.  The library
    records its phase events inside the graph.  After the timed replays the
    same flush + replay pairs go on, untimed and synchronised one by one,
    until the load has lasted `hold_s` seconds, so that a clock sampler with a
    200 ms period sees the GPU under this load.  Returns per-replay lists of
    (replay_ms, split_ms, combine_ms) and the load's wall-clock window."""
    inner = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in inner:                     # create the CUDA events before the capture
        e.record()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
                   d["custom_mask"], d["mask_indptr"], inp.sm_scale, d["out"], events=inner)
    torch.cuda.synchronize()
    call_ms, split_ms, comb_ms = [], [], []
    t_load = time.time()
    for k in range(warmup + steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        if k >= warmup:
            call_ms.append(e0.elapsed_time(e1))
            split_ms.append(inner[1].elapsed_time(inner[2]))
            comb_ms.append(inner[2].elapsed_time(inner[3]))
    while time.time() - t_load < hold_s:
        flush.zero_()
        g.replay()
        torch.cuda.synchronize()
    return call_ms, split_ms, comb_ms, (t_load, time.time())


def device_tensors(inp, torch, dev):
    from speculative_decode_mla_paged_gb300 import api  # noqa: F401
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).to(dev)
         for k in ("qo_indptr", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask", "mask_indptr")}
    d["q"] = inp.q.to(dev)
    d["kv_pool"] = inp.kv_pool.to(dev)
    d["out"] = torch.empty(inp.total_q, inp.num_heads, 512, dtype=torch.bfloat16, device=dev)
    return d


def run_launch_only(args):
    """W warm-up and K direct calls of one workload (L2 flushed before each),
    with no split-count timing, graph, end-to-end or oracle work around them,
    so that a profiler's launch list is just these calls: 2 or 3 library
    launches per call (the split kernel(s) and the combine)."""
    import torch

    from speculative_decode_mla_paged_gb300 import api, tuning
    from speculative_decode_mla_paged_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    api.init()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    inp = W.make_config_inputs(args.config, device=dev)
    d = device_tensors(inp, torch, dev)
    splits = args.num_splits or tuning.plan_num_splits(inp.prefix_lens, inp.draft_lens, inp.num_heads,
                                                       args.kernel)
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, splits, impl=args.kernel)
    call_ms, split_ms, _ = measure(inp, d, runner, args.steps, args.warmup, flush, torch)
    status = runner.status()
    print(json.dumps({"mode": "launch-only", "config": args.config, "kernel": args.kernel, "num_splits": splits,
                      "steps": args.steps, "warmup": args.warmup, "status": status,
                      "us_per_call": statistics.mean(call_ms) * 1e3, "split_us": statistics.mean(split_ms) * 1e3,
                      "launches_per_call": launches_per_call(inp, args.kernel)}), flush=True)
    if status != 0:
        raise SystemExit(f"device status word {status:#x}")


def run_ours(args):
    import torch

    from speculative_decode_mla_paged_gb300 import api
    from speculative_decode_mla_paged_gb300 import workloads as W

    world, rank, local = dist_setup(args)
    assert world == 1, "multi-GPU runs are refused in main() before CUDA is touched"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    api.init()
    peaks, peak_src = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    inp = W.make_config_inputs(args.config, device=dev)
    d = device_tensors(inp, torch, dev)
    splits, split_choice = (args.num_splits, "given") if args.num_splits else choose_splits(inp, d, args.kernel)
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, splits, impl=args.kernel)

    # ---- device-resident timed region
    torch.cuda.synchronize()
    gpu_index = None
    try:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        gpu_index = int(vis.split(",")[local]) if vis else local
    except ValueError:
        gpu_index = None
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    call_ms, split_ms, comb_ms, load_window = measure_graph(inp, d, runner, args.steps, args.warmup, flush, torch,
                                                           hold_s=CLOCK_HOLD_S)
    clocks = sampler.stop(load_window)
    status = runner.status()
    if status != 0:
        raise RuntimeError(f"device status word {status:#x}")
    t_total_ms = max_over_ranks(sum(call_ms), world, dev)
    value_us = per_call_us(t_total_ms, args.steps, world)

    # ---- the same call launched directly (host work between the library's
    # launches falls inside the timed events)
    d_call_ms, d_split_ms, d_comb_ms = measure(inp, d, runner, args.steps, args.warmup, flush, torch)

    # ---- end-to-end: pinned host inputs -> device, call, result -> host
    h2d_names = ("q", "qo_indptr", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask", "mask_indptr")
    host = {k: (inp.q.cpu() if k == "q" else torch.from_numpy(np.ascontiguousarray(getattr(inp, k)))).pin_memory()
            for k in h2d_names}
    host_out = torch.empty(d["out"].shape, dtype=torch.bfloat16).pin_memory()
    h2d_bytes = sum(t.numel() * t.element_size() for t in host.values())
    d2h_bytes = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for k in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for name in h2d_names:
            d[name].copy_(host[name], non_blocking=True)
        runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
               d["custom_mask"], d["mask_indptr"], inp.sm_scale, d["out"])
        host_out.copy_(d["out"], non_blocking=True)
        e1.record()
        e1.synchronize()
        if k >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_us = per_call_us(max_over_ranks(sum(e2e_ms), world, dev), args.steps, world)

    # ---- the same call warm (no flush, back-to-back direct calls)
    warm_us = measure_warm(inp, d, runner, args.steps, torch) * 1e3
    if runner.status() != 0:
        raise RuntimeError(f"device status word {runner.status():#x}")

    # ---- roofline of the dominant kernel (the split kernel)
    flops = inp.algorithmic_flops()
    nbytes = inp.algorithmic_bytes()
    split_s = statistics.mean(split_ms) / 1e3
    call_s = statistics.mean(call_ms) / 1e3
    t_f = flops / (peaks["bf16_tflops"] * 1e12)
    t_b = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_f >= t_b:
        roof = {"bound": "tensor", "achieved": flops / split_s / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": nbytes / split_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(args.kernel, args.config)
    roof["tensor_pipe"] = tensor_pipe_summary(profiled_tensor_pipe(args.kernel, args.config), split_s,
                                              (clocks or {}).get("sm_mhz"), flops)
    roof["peak_source"] = f"{peak_src} (burst; kernel timed alone)"
    roof["kernel"] = (f"{args.kernel} split phase (the split launches of one call, concurrent when both "
                      "tensor-core cluster shapes run; traffic summed over them)")
    roof["algorithmic_flops"] = flops
    roof["algorithmic_bytes"] = nbytes

    line = {
        "metric": METRIC, "value": value_us, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_total_ms / args.steps, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.config}: {W.CONFIGS[args.config].description}",
                   "kernel": args.kernel, "num_splits": splits, "num_splits_choice": split_choice,
                   "timing": "cold replays of one call captured in a CUDA graph",
                   "l2": "flushed before every timed replay (256 MiB write, excluded from timing)",
                   "parallelism": "single-gpu"},
        "tflops": flops / call_s / 1e12, "kv_gbs": nbytes / call_s / 1e9,
        "roofline_frac_call": max(t_f, t_b) / call_s,
        "split_us": statistics.mean(split_ms) * 1e3, "combine_us": statistics.mean(comb_ms) * 1e3,
        "roofline": roof,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": int(h2d_bytes),
                "d2h_bytes_per_step": int(d2h_bytes)},
        "gpu_launches": launches_per_call(inp, args.kernel) * args.steps,
        "clocks": clocks,
        "direct": {"value": statistics.mean(d_call_ms) * 1e3, "unit": UNIT,
                   "split_us": statistics.mean(d_split_ms) * 1e3, "combine_us": statistics.mean(d_comb_ms) * 1e3,
                   "what": "the same call launched directly each step (L2 flushed); host work between the "
                           "library's launches falls inside the timed events"},
        "warm": {"value": warm_us, "unit": UNIT, "l2": "not flushed (back-to-back direct calls)"},
    }

    # ---- the five workloads and the two extra ones (chain verify, decode),
    # device time per call (informational)
    headline_oracle = None
    if not args.no_cpu:
        import oracle
        oracle.build()
    if not args.no_per_config:
        table = {}
        for name in W.CONFIG_ORDER + W.EXTRA_CONFIG_ORDER:
            ci = inp if name == args.config else W.make_config_inputs(name, device=dev)
            cd = d if name == args.config else device_tensors(ci, torch, dev)
            cs = splits if name == args.config else (args.num_splits or choose_splits(ci, cd, args.kernel)[0])
            cr = runner if name == args.config else api.VerifyAttention(ci.batch, ci.max_q_per_req,
                                                                          ci.num_heads, cs, impl=args.kernel)
            gm, gs, _, _ = measure_graph(ci, cd, cr, 10, 3, flush, torch)
            cm, sm, _ = measure(ci, cd, cr, 5, 3, flush, torch)
            f, b = ci.algorithmic_flops(), ci.algorithmic_bytes()
            tg, tgs = statistics.mean(gm) / 1e3, statistics.mean(gs) / 1e3
            t_roof = max(f / (peaks["bf16_tflops"] * 1e12), b / (peaks["hbm_gbs"] * 1e9))
            table[name] = {"us_per_call": tg * 1e6, "split_us": tgs * 1e6,
                           "tflops": f / tg / 1e12, "kv_gbs": b / tg / 1e9,
                           "roofline_frac": t_roof / tg, "roofline_frac_split": t_roof / tgs,
                           "num_splits": cs,
                           "timing": "cold CUDA-graph replays (L2 flushed), 3 warm-up + 10 timed",
                           "direct_us_per_call": statistics.mean(cm) * 1e3,
                           "direct_split_us": statistics.mean(sm) * 1e3}
            if not args.no_cpu:
                host = ci if name != args.config else copy.copy(ci)
                host.q, host.kv_pool = ci.q.cpu(), ci.kv_pool.cpu()
                table[name]["cpu_oracle"] = oracle_timings(host)
                if name == args.config:
                    headline_oracle = table[name]["cpu_oracle"]
                del host
            if name != args.config:
                del cd, cr, ci
                torch.cuda.empty_cache()
        line["per_config"] = table

    # ---- CPU oracle baseline on the host cores: one whole call of the
    # headline workload on all cores (and on one core, see oracle_timings)
    if not args.no_cpu:
        if headline_oracle is None:
            host = copy.copy(inp)
            host.q, host.kv_pool = inp.q.cpu(), inp.kv_pool.cpu()
            headline_oracle = oracle_timings(host)
        line["cpu_baseline"] = {
            "value": headline_oracle["all_cores_s"] * 1e6, "unit": UNIT, "cores": headline_oracle["cores"],
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"one whole call (all {headline_oracle['rows']} output rows), timed, not scaled",
            "single_core": {"value": headline_oracle["single_core_s"] * 1e6, "unit": UNIT, "cores": 1,
                            "sample": headline_oracle["single_core_how"]}}
    print(json.dumps(line), flush=True)


MULTI_GPU_REFUSAL = ("single-GPU path: the tensor-core kernel's 4-CTA clusters use cluster-multicast TMA "
                     "loads, which this library runs on single-GPU calls only; no launch was made")


def refuse_multi_gpu(args):
    """True (after rank 0 printed the refusal line) when the run asks for more
    than one GPU.  Called before anything touches CUDA."""
    world, rank, _ = dist_setup(args)
    if world <= 1 and args.gpus <= 1:
        return False
    if rank == 0:
        print(json.dumps({"metric": METRIC, "n_gpus": max(world, args.gpus), "unit": UNIT,
                          "unavailable": MULTI_GPU_REFUSAL}), flush=True)
    return True


def main():
    args = parse_args()
    if args.impl != "reference" and refuse_multi_gpu(args):
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.launch_only:
        run_launch_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
