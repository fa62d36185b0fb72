#!/usr/bin/env python
"""GDN prefill benchmark on GB300: tokens/s and TFLOP/s through the C ABI.

One step = one gdn_extend_chunkwise call over the whole workload (every chunk of
every sequence and head: schedule, intra-chunk WY factors, inter-chunk scan with
the output epilogue). Default workload: the long-prefill configuration
(B=1, T=65536, H=HV=16, K=V=128, chunk_size=64, bf16, zero initial state), seeded
synthetic inputs resident in HBM when the timed region starts.

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle on
the host cores instead (the reference arm of this benchmark).

Multi-GPU (torchrun, N ranks): every rank runs its own replica of the workload on
its own GPU (the path needs no exchange between GPUs); value = tokens of all
ranks / the slowest rank's time ("weak" scaling).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s and TFLOP/s (% of GB300 bf16 peak), 1 GPU"
METRIC_DECODE = "GDN single-token step (decode) tokens/s and state GB/s (% of GB300 HBM), 1 GPU"
METRIC_BACKWARD = "GDN chunkwise backward tokens/s and gradient GB/s (% of GB300 HBM), 1 GPU"
DEC_KEYS = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state_pool", "cache_indices")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KEYS = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state_pool", "cache_indices", "cu_seqlens")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="long",
                    help="workload name (tiny, varlen, long, throughput, wide; decode: the single-token step; "
                         "backward: the backward pass on the long workload)")
    ap.add_argument("--backward-of", default="long",
                    help="with --config backward: the workload whose backward is timed (default: long)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time of the CPU baseline")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) with host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", device_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def wait_first(self, timeout_s: float = 5.0):
        """Waits until nvidia-smi has delivered a sample (it takes a moment to start)."""
        t_end = time.time() + timeout_s
        while self.proc and not self.samples and time.time() < t_end:
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "sampled during the timed region"
        if not inside:
            after = [p for (t, p) in self.samples if t > t1]
            inside = after[:1]
            note = "timed region shorter than the sampling period: first sample after it"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def device_uuid(torch, dev) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


# ----------------------------------------------------------------------------- roofline

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_accounting(w, lengths):
    """Algorithmic bytes and FLOPs per launch of each kernel: what the method must move (q, k, v, a, b
    read once, o written once, each touched state read and written once) and compute (triangular
    products at their true size), not what a kernel happens to execute."""
    from gated_deltanet_chunkwise_gdn_gb300 import accounting as acc
    T = sum(lengths)
    H, HV, K, V, C = w.H, w.HV, w.K, w.V, w.chunk_size
    B = len(lengths)
    e = 2  # bf16
    qk = T * H * K * e * 2
    intra_bytes = qk + T * HV * V * e
    gates_bytes = T * HV * 8 * 2  # a, b read; g, beta written
    scan_bytes = qk + T * HV * V * e + B * HV * V * K * 4 * 2
    intra_flops = scan_flops = 0.0
    for n in lengths:
        for s in range(0, n, C):
            L = min(C, n - s)
            intra_flops += HV * ((H / HV) * (L * (L - 1) * K + L * (L + 1) * K) + L ** 3 / 3.0 + L * (L + 1) * (K + V))
            scan_flops += HV * (6.0 * L * K * V + L * (L + 1) * V)
    path = {"bytes": acc.min_hbm_bytes(lengths, H, HV, K, V), "flops": acc.flop_count(lengths, H, HV, K, V, C)}
    if w.name == "decode":  # one kernel does the whole step
        return {"decode": dict(path), "path": path}
    return {
        "gates": {"bytes": gates_bytes, "flops": 0.0},
        "intra": {"bytes": intra_bytes, "flops": intra_flops},
        "scan": {"bytes": scan_bytes, "flops": scan_flops},
        "path": path,
    }


def _code_only(src: str) -> str:
    """C/CUDA source with comments and whitespace removed (string literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            i = src.find("*/", i + 2)
            i = n if i < 0 else i + 2
        elif c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (not the comments) of a kernel's sources and the shared headers."""
    files = {"gates": ["gdn_gates.cu"], "intra": ["gdn_intra.cu", "gdn_inverse.cuh"],
             "scan": ["gdn_scan.cu", "gdn_scan_affine.cu"],
             "schedule": ["gdn_schedule.cu"], "decode": ["gdn_decode.cu", "gdn_decode.cuh"],
             "backward": ["gdn_backward.cu", "gdn_backward.cuh", "gdn_mma.cuh", "gdn_inverse.cuh",
                          "gdn_gates.cu", "gdn_schedule.cu"]}
    csrc = os.path.join(ROOT, "gated_deltanet_chunkwise_gdn_gb300", "csrc")
    h = hashlib.sha256()
    for f in files.get(kernel, []) + ["gdn_common.cuh", "gdn_tc.cuh"]:
        p = os.path.join(csrc, f)
        if os.path.exists(p):
            h.update(_code_only(open(p, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        tab = json.load(open(path))
        ent = tab.get(workload, {}).get(kernel)
        if ent and ent.get("source_hash") == kernel_source_hash(kernel):
            return ent.get("dram_bytes_per_launch")
    except (ValueError, OSError):
        pass
    return None


def roofline_entry(name, acct, ms_avg, peaks, peak_kind, workload):
    bw = float(peaks["hbm_gbs"])
    tf = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    intensity = acct["flops"] / max(acct["bytes"], 1.0)
    ridge = tf * 1e12 / (bw * 1e9)
    if intensity < ridge:
        achieved = acct["bytes"] / (ms_avg * 1e-3) / 1e9
        ent = {"bound": "hbm", "achieved": round(achieved, 1), "peak": bw, "unit": "GB/s"}
    else:
        achieved = acct["flops"] / (ms_avg * 1e-3) / 1e12
        ent = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tf, "unit": "TFLOP/s"}
    ent["frac"] = round(ent["achieved"] / ent["peak"], 4)
    ent["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback"
    ent["kernel"] = name
    ent["ms_per_launch"] = round(ms_avg, 4)
    ent["algorithmic_bytes_per_launch"] = acct["bytes"]
    ent["algorithmic_flops_per_launch"] = acct["flops"]
    ent["traffic"] = measured_traffic(name, workload)
    return ent


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(d: dict, w, target_s: float):
    """Runs the oracle on the first S tokens of the first sequence (all value heads),
    S sized so the run takes about target_s seconds. Returns (tokens, seconds, threads, S)."""
    import oracle
    import torch
    cu = d["cu_seqlens"]
    L0 = int(cu[1] - cu[0])

    def run(S):
        sub = dict(d)
        for k in ("q", "k", "v", "a", "b"):
            sub[k] = d[k][:S]
        sub["cu_seqlens"] = torch.tensor([0, S], dtype=torch.int64)
        sub["cache_indices"] = d["cache_indices"][:1]
        t = time.perf_counter()
        res = oracle.gdn_forward(*[sub[k] for k in KEYS])
        return time.perf_counter() - t, res.threads

    probe = min(L0, 512)
    dt, _ = run(probe)
    S = max(1, min(L0, int(probe * target_s / max(dt, 1e-6))))
    dt, threads = run(S)
    return S, dt, threads


# ----------------------------------------------------------------------------- arms

def run_reference(args, dist):
    """The reference arm: the fp64 CPU oracle timed on the host cores (rank 0 only)."""
    if dist.rank != 0:
        return
    import oracle
    from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl
    oracle.build()
    w = wl.BY_NAME[args.config]
    d = wl.make_inputs(w)
    per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    import torch
    if w.name == "decode":  # the whole single-token batch is a small sample already
        sub, S = d, int(d["cache_indices"].numel())
        sample = f"the whole batch ({S} sequences x {w.HV} value heads), per step"
    else:
        S, _, _ = oracle_sample(d, w, per_step)
        sub = dict(d)
        for k in ("q", "k", "v", "a", "b"):
            sub[k] = d[k][:S]
        sub["cu_seqlens"] = torch.tensor([0, S], dtype=torch.int64)
        sub["cache_indices"] = d["cache_indices"][:1]
        sample = f"first {S} tokens of sequence 0, all {w.HV} value heads, per step"
    for _ in range(args.warmup):
        oracle.gdn_forward(*[sub[k] for k in KEYS])
    t = time.perf_counter()
    threads = 1
    for _ in range(args.steps):
        threads = oracle.gdn_forward(*[sub[k] for k in KEYS]).threads
    el = time.perf_counter() - t
    tok_s = S * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC_DECODE if w.name == "decode" else METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.note}", "sample": sample},
        "cpu_baseline": {"value": round(tok_s, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(tok_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def oracle_sample_decode(d: dict, target_s: float):
    """Runs the oracle on the whole single-token batch, repeated until about target_s seconds.
    Returns (tokens, seconds, threads, repeats)."""
    import oracle
    t = time.perf_counter()
    res = oracle.gdn_forward(*[d[k] for k in KEYS])
    one = time.perf_counter() - t
    reps = max(1, int(target_s / max(one, 1e-6)))
    t = time.perf_counter()
    for _ in range(reps):
        res = oracle.gdn_forward(*[d[k] for k in KEYS])
    dt = time.perf_counter() - t
    return int(d["cache_indices"].numel()) * reps, dt, res.threads, reps


def run_ours(args, dist):
    import torch
    import gated_deltanet_chunkwise_gdn_gb300 as gdn
    from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl

    dev = torch.device("cuda", dist.local_rank if dist.world > 1 else 0)
    torch.cuda.set_device(dev)
    w = wl.BY_NAME[args.config]
    decode = w.name == "decode"
    d = wl.make_inputs(w)
    lengths = wl.sequence_lengths(w)
    T = sum(lengths)
    g = {k: d[k].to(dev) for k in KEYS}
    out = torch.empty((T, w.HV, w.V), dtype=w.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(bufs, o, check=False):
        if decode:  # one token per sequence: q, k, v, a, b are [B, ...]
            gdn.gdn_decode_step(*[bufs[k] for k in DEC_KEYS], out=o, check=check)
        else:
            gdn.gdn_extend_chunkwise(*[bufs[k] for k in KEYS], chunk_size=w.chunk_size, out=o, check=check)

    def step():
        call(g, out)

    call(g, out, check=True)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    # ---- timed region: kernels only, inputs resident in HBM. The library's per-kernel events
    # would sit between the kernels of a call (and stop each kernel from being scheduled while
    # the previous one finishes), so the step time is taken without them; the per-kernel
    # durations come from a second pass over the same steps with the events on.
    sampler = ClockSampler(device_uuid(torch, dev))
    sampler.wait_first()
    for _ in range(max(3, args.warmup)):  # the GPU is busy again when the timed region starts
        step()
    dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = gdn.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    dist.barrier()
    launches = gdn.launch_count() - n0
    time.sleep(0.1)
    sampler.stop()
    ms = e0.elapsed_time(e1)
    ms_max = dist.max(ms)
    clocks = sampler.summary(t_host0, t_host1)
    prof = gdn.KernelProfile(max_launches=8 * args.steps + 64)
    prof.start()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    kernels = prof.stop()

    # ---- e2e: host buffers through the public API, copies inside the timed region. Every step
    # copies its inputs host->device and its output device->host; as a serving loop would, the
    # copies of neighbouring steps overlap the call (two device buffer sets, copy streams
    # ordered by events). The state pool is shared, so the calls stay in order on one stream.
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    in_keys = ("q", "k", "v", "a", "b", "cache_indices") + (() if decode else ("cu_seqlens",))
    host_in = {k: d[k].pin_memory() for k in in_keys}
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    bufs = [dict(g)] + [dict(g, **{k: torch.empty_like(g[k]) for k in in_keys})]
    outs = [out, torch.empty_like(out)]
    n_in = 1  # upload streams (splitting the inputs over 4 concurrent copies measured slower)
    s_ins = [torch.cuda.Stream(dev) for _ in range(n_in)]
    s_out = torch.cuda.Stream(dev)
    ev_in = [[torch.cuda.Event() for _ in range(n_in)] for _ in range(2)]  # inputs of set i landed
    ev_done = [torch.cuda.Event() for _ in range(2)]   # call on buffer set i finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # output of set i copied to the host

    def e2e_run(n):
        for i in range(n):
            b = i % 2
            for j, sj in enumerate(s_ins):  # inputs of step i, once step i-2 is done with the set
                with torch.cuda.stream(sj):
                    sj.wait_event(ev_done[b])
                    for k, t in host_in.items():  # piece j of every input, split along tokens
                        n = t.shape[0]
                        lo, hi = n * j // n_in, n * (j + 1) // n_in
                        if hi > lo:
                            bufs[b][k][lo:hi].copy_(t[lo:hi], non_blocking=True)
                    ev_in[b][j].record(sj)
            for e in ev_in[b]:
                stream.wait_event(e)
            stream.wait_event(ev_out[b])  # the output buffer of step i-2 has been read back
            call(bufs[b], outs[b])
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                host_out[b].copy_(outs[b], non_blocking=True)
                ev_out[b].record(s_out)

    for e in ev_done + ev_out:
        e.record(stream)
    e2e_run(2)
    torch.cuda.synchronize(dev)
    dist.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for sj in s_ins:
        sj.wait_stream(stream)  # the first copies start after f0
    e2e_run(e2e_steps)
    stream.wait_stream(s_out)  # f1 after the last output copy
    f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = dist.max(f0.elapsed_time(f1))

    if dist.rank != 0:
        return
    acct = kernel_accounting(w, lengths)
    peaks, peak_kind = load_peaks()
    per_kernel = {}
    for name, (tot, n) in kernels.items():
        if n:
            per_kernel[name] = {"ms_per_launch": round(tot / n, 4), "launches": n,
                                "share": round(tot / max(sum(v[0] for v in kernels.values()), 1e-9), 4)}
    dominant = max((k for k in kernels if k in acct and kernels[k][1]), key=lambda k: kernels[k][0])
    roof = roofline_entry(dominant, acct[dominant], kernels[dominant][0] / kernels[dominant][1], peaks, peak_kind,
                          w.name)
    step_ms = ms / args.steps
    path = roofline_entry("path", acct["path"], step_ms, peaks, peak_kind, w.name)
    path.pop("traffic", None)
    tokens = T * args.steps * dist.world
    value = tokens / (ms_max * 1e-3)
    tflops = acct["path"]["flops"] * args.steps * dist.world / (ms_max * 1e-3) / 1e12
    if decode:
        l2 = "inputs larger than L2 (state slots %.0f MB read and written > 129 MB), no flush" % (
            len(lengths) * w.HV * w.V * w.K * 4 / 1e6)
    else:
        l2 = "inputs larger than L2 (q,k,v %.0f MB > 129 MB), no flush" % (3 * T * w.H * w.K * 2 / 1e6)
    line = {
        "metric": METRIC_DECODE if decode else METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.note}", "global_batch": len(lengths) * dist.world, "seq_len": max(lengths),
                   "total_tokens_per_gpu": T, "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU",
                   "l2": l2},
        "tflops": round(tflops, 2),
        "frac_bf16_peak": round(tflops / float(peaks["bf16_tflops"]), 4),
        "roofline": roof,
        "path_roofline": path,
        "kernels": per_kernel,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": {"value": round(T * e2e_steps * dist.world / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": round(e2e_ms / e2e_steps, 4)},
    }
    if dist.world == 1 and not args.no_cpu_baseline and decode:
        n, dt, threads, reps = oracle_sample_decode(d, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(n / dt, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": f"the whole batch ({len(lengths)} sequences x {w.HV} value heads), "
                                          f"{reps} times ({dt:.1f} s)"}
    elif dist.world == 1 and not args.no_cpu_baseline:
        S, dt, threads = oracle_sample(d, w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(S / dt, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {S} tokens of sequence 0, all {w.HV} value heads ({dt:.1f} s)"}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- backward

def backward_inputs(w):
    """The long workload's inputs plus seeded gradients from above (d_out like v, d_state like the pool)."""
    import torch
    from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl
    d = wl.make_inputs(w)
    gen = torch.Generator().manual_seed(1000 + w.seed)
    d["d_out"] = torch.randn(d["v"].shape, generator=gen).to(w.dtype)
    d["d_state"] = 0.1 * torch.randn(d["state_pool"].shape, generator=gen)
    return d


def backward_accounting(w, lengths):
    """Algorithmic bytes of one backward call: q, k, v, d_out, a, b read once; dq, dk, dv (fp32), da, db
    written once; each touched initial state and final-state gradient read once and the initial state's
    gradient written once. FLOPs: twice the forward's algorithmic count (an estimate: the backward runs
    about two forward-sized sets of products)."""
    from gated_deltanet_chunkwise_gdn_gb300 import accounting as acc
    T, B = sum(lengths), len(lengths)
    H, HV, K, V = w.H, w.HV, w.K, w.V
    nbytes = (T * H * K * 2 * 2 + T * HV * V * 2 * 2 + T * HV * 4 * 2 + T * H * K * 4 * 2 + T * HV * V * 4
              + T * HV * 4 * 2 + B * HV * V * K * 4 * 3 + HV * 4 * 4)
    return {"bytes": nbytes, "flops": 2.0 * acc.flop_count(lengths, H, HV, K, V, w.chunk_size)}


def oracle_backward_sample(d, S):
    """The gradient oracle (chain rule on the token recurrence, fp64 numpy) on the first S tokens of
    sequence 0, all value heads. Returns seconds."""
    import torch
    from oracle import backward as bw
    sub = {k: d[k][:S] for k in ("q", "k", "v", "a", "b", "d_out")}
    idx = d["cache_indices"][:1]
    t = time.perf_counter()
    bw.gdn_backward(sub["q"], sub["k"], sub["v"], sub["a"], sub["b"], d["A_log"], d["dt_bias"], d["state_pool"],
                    idx, torch.tensor([0, S], dtype=torch.int64), sub["d_out"].double(),
                    d["d_state"].double().numpy()[idx.numpy()])
    return time.perf_counter() - t


def backward_cpu_sample(d, target_s):
    L0 = int(d["cu_seqlens"][1] - d["cu_seqlens"][0])
    probe = min(L0, 64)
    dt = oracle_backward_sample(d, probe)
    S = max(1, min(L0, int(probe * target_s / max(dt, 1e-6))))
    return S, oracle_backward_sample(d, S)


def run_backward(args, dist):
    import torch
    import gated_deltanet_chunkwise_gdn_gb300 as gdn
    from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl

    w = wl.BY_NAME[args.backward_of]
    if w.K not in (64, 128) or w.K != w.V:
        raise SystemExit(f"the backward is built for K = V in {{64, 128}}; {w.name} has K={w.K}, V={w.V}")
    if args.impl == "reference":
        if dist.rank != 0:
            return
        d = backward_inputs(w)
        per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))
        S, _ = backward_cpu_sample(d, per_step)
        for _ in range(args.warmup):
            oracle_backward_sample(d, S)
        el = sum(oracle_backward_sample(d, S) for _ in range(args.steps))
        tok_s = S * args.steps / el
        sample = f"first {S} tokens of sequence 0, all {w.HV} value heads, per step"
        print(json.dumps({
            "impl": "reference", "metric": METRIC_BACKWARD, "value": round(tok_s, 1), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"backward of {w.name}: {w.note}", "sample": sample},
            "cpu_baseline": {"value": round(tok_s, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(tok_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    dev = torch.device("cuda", dist.local_rank if dist.world > 1 else 0)
    torch.cuda.set_device(dev)
    d = backward_inputs(w)
    lengths = wl.sequence_lengths(w)
    T = sum(lengths)
    keys = KEYS + ("d_out", "d_state")
    g = {k: d[k].to(dev) for k in keys}
    need = gdn.gdn_backward_workspace_size(T, len(lengths), w.H, w.HV, w.K, w.V, w.chunk_size)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    grads = gdn.GdnGrads(torch.empty((T, w.H, w.K), **f32), torch.empty((T, w.H, w.K), **f32),
                         torch.empty((T, w.HV, w.V), **f32), torch.empty((T, w.HV), **f32),
                         torch.empty((T, w.HV), **f32), torch.empty((w.HV,), **f32), torch.empty((w.HV,), **f32),
                         torch.zeros_like(g["state_pool"]))
    stream = torch.cuda.current_stream(dev)

    def call(b, check=False):
        gdn.gdn_chunkwise_backward(*[b[k] for k in KEYS], b["d_out"], b["d_state"], chunk_size=w.chunk_size,
                                   workspace=ws, grads=grads, check=check)

    call(g, check=True)
    for _ in range(max(3, args.warmup)):
        call(g)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(device_uuid(torch, dev))
    sampler.wait_first()
    for _ in range(max(3, args.warmup)):
        call(g)
    dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = gdn.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        call(g)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    dist.barrier()
    launches = gdn.launch_count() - n0
    time.sleep(0.1)
    sampler.stop()
    ms = e0.elapsed_time(e1)
    ms_max = dist.max(ms)
    clocks = sampler.summary(t_host0, t_host1)
    prof = gdn.KernelProfile(max_launches=4 * args.steps + 64)
    prof.start()
    for _ in range(args.steps):
        call(g)
    torch.cuda.synchronize(dev)
    kernels = prof.stop()

    # e2e: host buffers through the public API; every step uploads its inputs and the gradients
    # from above, and reads every gradient back (the initial states stay resident)
    e2e_steps = max(1, min(args.e2e_steps, args.steps, 10))
    in_keys = ("q", "k", "v", "a", "b", "cache_indices", "cu_seqlens", "d_out", "d_state")
    host_in = {k: d[k].pin_memory() for k in in_keys}
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in grads]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    dbuf = dict(g, **{k: torch.empty_like(g[k]) for k in in_keys})

    def e2e_step():
        for k, t in host_in.items():
            dbuf[k].copy_(t, non_blocking=True)
        call(dbuf)
        for h, t in zip(host_out, grads):
            h.copy_(t, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    dist.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = dist.max(f0.elapsed_time(f1))

    if dist.rank != 0:
        return
    peaks, peak_kind = load_peaks()
    acct = backward_accounting(w, lengths)
    tot_all = max(sum(v[0] for v in kernels.values()), 1e-9)
    per_kernel = {name: {"ms_per_launch": round(tot / n, 4), "launches": n, "share": round(tot / tot_all, 4)}
                  for name, (tot, n) in kernels.items() if n}
    bt, bn = kernels["backward"]
    roof = roofline_entry("backward", acct, bt / bn, peaks, peak_kind, w.name)
    step_ms = ms_max / args.steps
    path = roofline_entry("path", acct, step_ms, peaks, peak_kind, w.name)
    path.pop("traffic", None)
    tokens = T * args.steps * dist.world
    line = {
        "metric": METRIC_BACKWARD, "value": round(tokens / (ms_max * 1e-3), 1), "unit": "tokens/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"backward of {w.name}: {w.note}; d_out ~ N(0,1), d_state ~ N(0, 0.1^2)",
                   "global_batch": len(lengths) * dist.world, "seq_len": max(lengths), "total_tokens_per_gpu": T,
                   "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (q,k,v,d_out %.0f MB > 129 MB), no flush" % (4 * T * w.H * w.K * 2 / 1e6)},
        "tflops": round(acct["flops"] * args.steps * dist.world / (ms_max * 1e-3) / 1e12, 2),
        "roofline": roof,
        "path_roofline": path,
        "kernels": per_kernel,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": {"value": round(T * e2e_steps * dist.world / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": round(e2e_ms / e2e_steps, 4)},
    }
    if dist.world == 1 and not args.no_cpu_baseline:
        S, dt = backward_cpu_sample(d, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(S / dt, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"first {S} tokens of sequence 0, all {w.HV} value heads ({dt:.1f} s)"}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    dist = Dist()
    try:
        if args.config == "backward":
            run_backward(args, dist)
        elif args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
