#!/usr/bin/env python
"""Benchmark of the chunked gated-delta-rule prefill forward on one GB300.

One step = one gdn_chunk_fwd call (chunk-table builder, intra-chunk kernel,
inter-chunk scan) over the Qwen3.5-9B-shaped GQA prefill: one sequence of
T=4096 tokens, H=16 key heads, Hv=32 value heads, dk=dv=128, bf16 q/k/v and
output, fp32 g/beta/initial and final state. Inputs are seeded synthetic
tensors already resident in HBM; a 512 MiB buffer is written between timed
steps so that every step starts with a cold L2 (129 MB).

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle
(fp64 token recurrence in C) on the host cores instead, on a bounded sample of
the same workload. Under torchrun (N > 1) every rank runs an independent
replica (the path has no exchange step); the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN chunk-prefill tokens/s at T=4096 H16/Hv32 bf16; % of roofline"
CHUNK = 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--clocks-file", default=None)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (smaller cases for profiling)")
    ap.add_argument("--backward", action="store_true",
                    help="time gdn_chunk_bwd (the backward pass) on the workload instead")
    return ap.parse_args(argv)


# --------------------------------------------------------------------- workload arithmetic
def n_chunks(lengths):
    return sum(-(-int(x) // CHUNK) for x in lengths)


def algorithmic_bytes(x, out_bytes=2):
    """Compulsory HBM bytes of one call: q, k, v, out, g, beta, initial and final states."""
    esz = 2 if x["dtype"] == "bf16" else 4
    T, H, Hv, dk, dv, N = x["n_tokens"], x["H"], x["Hv"], x["dk"], x["dv"], x["N"]
    g_b = T * Hv * (dk if x.get("channel_gates") else 1) * 4
    b = 2 * T * H * dk * esz + T * Hv * dv * esz + T * Hv * dv * out_bytes + g_b + T * Hv * 4
    states = N * Hv * dk * dv * 4
    b += states * (2 if x["initial_state"] is not None else 1)
    return b


def algorithmic_flops(x):
    """FLOPs of the chunked method (q.k^T and k.k^T once per key head per chunk; with
    per-channel gates the decay sits inside those products, so once per value head)."""
    NT = n_chunks(x["lengths"])
    C, dk, dv = CHUNK, x["dk"], x["dv"]
    per_h = 2 * 2 * C * C * dk
    per_hv = C ** 3 / 3 + 2 * C * C * dk + 2 * C * C * dv + 3 * 2 * C * dk * dv + 2 * C * C * dv
    heads_qk = x["Hv"] if x.get("channel_gates") else x["H"]
    return NT * heads_qk * per_h + NT * x["Hv"] * per_hv


def gdn_metric(workload: int) -> str:
    from gated_delta_rule_chunk_gb300.inputs import HEADLINE, WORKLOADS
    if workload == HEADLINE:
        return METRIC
    return f"GDN chunk-prefill tokens/s, {WORKLOADS[workload].name}; % of roofline"


def stage_flops(x):
    """FLOPs of the intra kernel (A and M products, triangular inverse, w and u) and of
    the scan (w S, q S, M v_new and the state update), counted as in algorithmic_flops."""
    NT = n_chunks(x["lengths"])
    C, dk, dv = CHUNK, x["dk"], x["dv"]
    heads_qk = x["Hv"] if x.get("channel_gates") else x["H"]
    intra = NT * heads_qk * 2 * 2 * C * C * dk + NT * x["Hv"] * (C ** 3 / 3 + 2 * C * C * (dk + dv))
    inter = NT * x["Hv"] * (3 * 2 * C * dk * dv + 2 * C * C * dv)
    return {"chunk_table": 0.0, "intra": intra, "inter": inter}


# fp32 FMA peak of the SIMT kernels: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (max SM clock)
SIMT_FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def uses_tc_path(x):
    """bf16 inputs run on the tensor-core kernels (d = 64 zero-padded to 128; per-channel
    gates through their own intra kernel and the scan's per-channel mode); fp32 inputs on
    the SIMT kernels."""
    return x["dtype"] == "bf16"


def method_stage_bytes(x, out_bytes=2):
    """Algorithmic bytes of each stage as the method defines its boundary: the intra
    stage reads q, k, v, g and beta and writes w and u (bf16) and the in-chunk gate sums
    G; the scan reads q, k, w, u, G and the initial state and writes out and the final
    state. (This implementation's own bridge is larger; see stage_bytes.)"""
    esz = 2 if x["dtype"] == "bf16" else 4
    T, H, Hv, dk, dv, N = x["n_tokens"], x["H"], x["Hv"], x["dk"], x["dv"], x["N"]
    NT = n_chunks(x["lengths"])
    qk = 2 * T * H * dk * esz
    g_b = T * Hv * (dk if x.get("channel_gates") else 1) * 4
    wu = NT * Hv * CHUNK * (dk + dv) * 2
    G = NT * Hv * CHUNK * 4
    states = N * Hv * dk * dv * 4
    s_in = states if x["initial_state"] is not None else 0
    intra = qk + T * Hv * dv * esz + g_b + T * Hv * 4 + wu + G
    inter = qk + wu + G + s_in + states + T * Hv * dv * out_bytes
    return {"chunk_table": 8 * (x["N"] + 1 + x["nt_max"]), "intra": intra, "inter": inter}


def stage_bytes(x, out_bytes=2):
    """Bytes each kernel must move given the intra/inter bridge it exchanges
    (per chunk and value head: w bf16, u fp32, decay-masked q.k as a bf16 hi/lo
    pair, G fp32; per chunk and key head on the bf16 path: an fp16 copy of k,
    which the inter kernel reads in place of k)."""
    esz = 2 if x["dtype"] == "bf16" else 4
    T, H, Hv, dk, dv, N = x["n_tokens"], x["H"], x["Hv"], x["dk"], x["dv"], x["N"]
    NT = n_chunks(x["lengths"])
    q = T * H * dk * esz
    k = T * H * dk * esz
    states = N * Hv * dk * dv * 4
    s_in = states if x["initial_state"] is not None else 0
    g_b = T * Hv * (dk if x.get("channel_gates") else 1) * 4
    if uses_tc_path(x) and x.get("channel_gates"):
        # per chunk and value head: w (bf16), u (fp32), M (hi/lo), the decayed k (fp16),
        # the decayed q (bf16 hi/lo) and exp(G_L) per channel
        bridge = NT * Hv * (16384 + 32768 + 16384 + 16384 + 32768 + 512)
        intra = q + k + T * Hv * dv * esz + g_b + T * Hv * 4 + bridge
        inter = bridge + s_in + states + T * Hv * dv * out_bytes
    elif uses_tc_path(x):
        # the bridge is 128 wide (a head of 64 runs zero-padded to 128)
        bridge = NT * Hv * (CHUNK * 128 * 2 + CHUNK * 128 * 4 + CHUNK * CHUNK * 4 + CHUNK * 4)
        k16 = NT * H * CHUNK * 128 * 2
        intra = q + k + T * Hv * dv * esz + g_b + T * Hv * 4 + bridge + k16
        inter = q + k16 + bridge + s_in + states + T * Hv * dv * out_bytes
    else:
        # per chunk and value head, fp32: w^T, u, M^T, exp(G) q, exp(G_L - G) k, exp(G_L)
        bridge = NT * Hv * (4 * CHUNK * dk * 4 + CHUNK * CHUNK * 4 + dk * 4)
        intra = q + k + T * Hv * dv * esz + g_b + T * Hv * 4 + bridge
        inter = bridge + s_in + states + T * Hv * dv * out_bytes
    return {"chunk_table": 8 * (x["N"] + 1 + x["nt_max"]), "intra": intra, "inter": inter}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of each
# kernel on the T=4096 H=16 Hv=32 workload, from the ncu capture summarised in the
# named profile, together with the SHA-1 of the kernel's source at capture time:
# when the source has changed since, the figure no longer applies and is not reported.
NCU_TRAFFIC = {
    "inter": {"source": "gated_delta_rule_chunk_gb300/csrc/k_scan.cu",
              "sha1": "5ca9466ac1045ce7ec35eeb70ae6c304d02d02df", "bytes": 191374592,
              "profile": "profiles/scan_kernel_T4096_H16_Hv32.md"},
    "intra": {"source": "gated_delta_rule_chunk_gb300/csrc/k_tc_intra.cu",
              "sha1": "26a91d063b343c011e5188e356d94ef0321f8ced", "bytes": 181576192,
              "profile": "profiles/tc_intra_kernel_T4096_H16_Hv32.md"},
}
NCU_WORKLOAD = 2


def ncu_traffic(stage: str, workload: int):
    """Captured DRAM bytes per launch of `stage`, or None when no capture applies."""
    import hashlib
    e = NCU_TRAFFIC.get(stage)
    if e is None or workload != NCU_WORKLOAD:
        return None, None
    try:
        with open(os.path.join(ROOT, e["source"]), "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != e["sha1"]:
                return None, "kernel source changed since the capture"
    except OSError:
        return None, None
    return e["bytes"], e["profile"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path=None):
        self.path = path or os.path.join(tempfile.gettempdir(), f"gdn_clocks_{os.getpid()}.csv")
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------- CPU oracle
def cpu_model() -> str:
    """The host CPU's name (x86 model name, or the Arm implementer/part of the cores)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    arm_parts = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1"}
    part = fields.get("CPU part")
    if part:
        return f"{arm_parts.get(part, 'Arm core')} (implementer {fields.get('CPU implementer', '?')}, part {part})"
    return "unknown"


def oracle_rate(x, seconds: float, max_tokens=None, nthreads: int = 0):
    """Time the CPU oracle on the first T_s tokens of the workload (all heads).
    T_s is sized from a short probe so the timed sample takes about `seconds`.
    nthreads: 0 = every core the process may use, else that many threads."""
    import oracle
    import torch

    def run(ts):
        cu = torch.tensor([0, ts], dtype=torch.int32)
        sl = slice(0, ts)
        s0 = x["initial_state"][:1] if x["initial_state"] is not None else None
        t = time.perf_counter()
        oracle.recurrent_forward(x["q"][sl], x["k"][sl], x["v"][sl], x["g"][sl], x["beta"][sl],
                                 x["scale"], s0, cu, nthreads=nthreads)
        return time.perf_counter() - t

    oracle.build()
    probe = min(64, x["n_tokens"])
    dt = run(probe)
    limit = max_tokens or x["n_tokens"]
    ts = int(max(16, min(limit, probe * seconds / max(dt, 1e-6))))
    ts = max(16, ts // 16 * 16)
    dt = run(ts)
    reps = 1
    while dt < 0.8 * seconds and ts == limit:  # the whole workload is shorter: repeat it
        dt += run(ts)
        reps += 1
    return reps * ts / dt, ts, dt, (nthreads or oracle.max_threads()), reps


# --------------------------------------------------------------------- distributed plumbing
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(val: float, ws: int) -> float:
    if ws == 1:
        return val
    import torch
    import torch.distributed as dist
    t = torch.tensor([val], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------- arms
def run_reference(args, ws, rank):
    from gated_delta_rule_chunk_gb300.inputs import WORKLOADS, make_inputs
    if rank != 0:
        return None
    x = make_inputs(args.workload, T=args.tokens)
    budget = 150.0 / max(1, args.steps + args.warmup)   # whole run within a few minutes
    rate0, ts, dt, cores, _ = oracle_rate(x, min(budget, args.cpu_seconds))
    import oracle
    import torch
    cu = torch.tensor([0, ts], dtype=torch.int32)
    sl = slice(0, ts)
    s0 = x["initial_state"][:1] if x["initial_state"] is not None else None
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        oracle.recurrent_forward(x["q"][sl], x["k"][sl], x["v"][sl], x["g"][sl], x["beta"][sl],
                                 x["scale"], s0, cu)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    ms = 1000.0 * statistics.mean(times)
    value = ts / (ms / 1000.0)
    sample = (f"first {ts} tokens of the {WORKLOADS[args.workload].name} workload, all "
              f"{x['Hv']} value heads, per step")
    return {
        "impl": "reference", "metric": gdn_metric(args.workload), "value": value,
        "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload].name, "T": x["T"], "H": x["H"],
                   "Hv": x["Hv"], "dk": x["dk"], "dv": x["dv"], "chunk": CHUNK,
                   "oracle": "fp64 token-by-token recurrence in C, OpenMP over (seq, head)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def recurrent_bytes(x, out_bytes=2):
    """Bytes the token-serial kernel must move: each sequence's state read and written
    once (fp32 [Hv, dv, dk]), q, k, v, g, beta read and out written per token."""
    esz = 2 if x["dtype"] == "bf16" else 4
    T, H, Hv, dk, dv, N = x["n_tokens"], x["H"], x["Hv"], x["dk"], x["dv"], x["N"]
    states = N * Hv * dk * dv * 4
    s_in = states if x["initial_state"] is not None else 0
    return (s_in + states + 2 * T * H * dk * esz + T * Hv * dv * esz + 2 * T * Hv * 4
            + T * Hv * dv * out_bytes)


def run_recurrent(args, ws, rank, local):
    """Decode / speculative-verify workloads through gdn_recurrent_fwd."""
    import torch
    from gated_delta_rule_chunk_gb300 import binding as B
    from gated_delta_rule_chunk_gb300.build import build
    from gated_delta_rule_chunk_gb300.inputs import WORKLOADS, make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    x = make_inputs(args.workload, T=args.tokens)
    d = {k: (x[k].to(dev) if x.get(k) is not None else None)
         for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")}
    out = torch.empty(x["T"], x["Hv"], 128, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(x["N"], x["Hv"], 128, 128, dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        B.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                            d["initial_state"], d["cu_seqlens"], out=out, final_state=fin)

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(args.warmup):
        flush.fill_(i & 255)
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, args.clocks_file)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_((i + 1) & 255)
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    ms = statistics.mean(r[0].elapsed_time(r[1]) for r in evs)
    ms_max = max_over_ranks(ms, ws)
    tokens = x["n_tokens"]
    value = ws * tokens / (ms_max / 1000.0)

    # e2e: the step's tokens come from pinned host memory and the output goes back; the
    # recurrent state stays resident on the device, as in a decode loop
    host = {k: x[k].pin_memory() for k in ("q", "k", "v", "g", "beta", "cu_seqlens")}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    e2e_ms = []
    for i in range(3 + args.e2e_steps if args.e2e_steps > 0 else 0):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for key, t in host.items():
            d[key].copy_(t, non_blocking=True)
        call()
        out_h.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(b))
    e2e_val = (ws * tokens / (max_over_ranks(statistics.mean(e2e_ms), ws) / 1000.0)
               if e2e_ms else None)
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    nbytes = recurrent_bytes(x)
    gbs = nbytes / (ms / 1000.0) / 1e9
    res = {
        "metric": "GDN token-serial decode/verify tokens/s (H16/Hv32 bf16, fp32 state)",
        "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload].name, "N": x["N"],
                   "tokens_per_sequence": x["lengths"][0], "H": x["H"], "Hv": x["Hv"],
                   "dk": 128, "dv": 128, "qkv_dtype": "bf16", "out_dtype": "bf16",
                   "initial_state": x["initial_state"] is not None,
                   "l2": "512 MiB buffer written between timed steps (L2 is 129 MB)",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "inputs": "resident in HBM"},
        "roofline": {"bound": "hbm", "kernel": "recurrent", "achieved": gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": nbytes, "traffic": None},
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "ms_per_step": statistics.mean(e2e_ms) if e2e_ms else None},
        "gpu_launches": K,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        rate, ts, dt, cores, reps = oracle_rate(x, args.cpu_seconds)
        res["cpu_baseline"] = {
            "value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"first {ts} tokens as one sequence, all {x['Hv']} value heads, "
                      f"run {reps} times ({dt:.1f} s of fp64 C on the host cores)"}
    return res


def conv_bytes(c):
    """Bytes the front end must move: x read, q/k/v written (same size), the taps,
    the conv state read and written."""
    esz = 2 if c["dtype"] == "bf16" else 4
    T, C, d, N = c["T"], c["C"], c["d_conv"], c["N"]
    states = N * C * (d - 1) * 4
    return 2 * T * C * esz + C * d * 4 + 2 * states


def run_conv(args, ws, rank, local):
    """The front end (gdn_conv_front) on the Qwen3.5-9B-shaped prefill."""
    import torch
    from gated_delta_rule_chunk_gb300 import binding as B
    from gated_delta_rule_chunk_gb300.build import build
    from gated_delta_rule_chunk_gb300.inputs import WORKLOADS, make_conv_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    wl = WORKLOADS[args.workload]
    c = make_conv_inputs(seed=1000 + args.workload, T=wl.T, H=wl.H, Hv=wl.Hv, d_conv=4)
    x, w, s0 = c["x"].to(dev), c["w"].to(dev), c["state"].to(dev)
    T, C = x.shape
    q = torch.empty(T, wl.H, 128, dtype=x.dtype, device=dev)
    k = torch.empty_like(q)
    v = torch.empty(T, wl.Hv, 128, dtype=x.dtype, device=dev)
    s1 = torch.empty_like(s0)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        B.gdn_conv_front(x, w, wl.H, wl.Hv, s0, None, conv_state_out=s1, q=q, k=k, v=v)

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(args.warmup):
        flush.fill_(i & 255)
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, args.clocks_file)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_((i + 1) & 255)
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    ms = statistics.mean(r[0].elapsed_time(r[1]) for r in evs)
    ms_max = max_over_ranks(ms, ws)
    value = ws * T / (ms_max / 1000.0)
    # e2e: x from pinned host memory, q/k/v back; the conv state stays resident
    x_h = c["x"].pin_memory()
    outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (q, k, v)]
    h2d = x_h.numel() * x_h.element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    e2e_ms = []
    for i in range(3 + args.e2e_steps if args.e2e_steps > 0 else 0):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x.copy_(x_h, non_blocking=True)
        call()
        for hh, dd in zip(outs_h, (q, k, v)):
            hh.copy_(dd, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(b))
    e2e_val = (ws * T / (max_over_ranks(statistics.mean(e2e_ms), ws) / 1000.0)
               if e2e_ms else None)
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    nbytes = conv_bytes(c)
    gbs = nbytes / (ms / 1000.0) / 1e9
    res = {
        "metric": "GDN front end (conv1d d=4 + SiLU over the qkv projection) tokens/s",
        "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "T": T, "channels": C, "d_conv": 4, "H": wl.H,
                   "Hv": wl.Hv, "qkv_dtype": "bf16", "conv_state": True,
                   "l2": "512 MiB buffer written between timed steps (L2 is 129 MB)",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "inputs": "resident in HBM"},
        "roofline": {"bound": "hbm", "kernel": "conv", "achieved": gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": nbytes, "traffic": None},
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "ms_per_step": statistics.mean(e2e_ms) if e2e_ms else None},
        "gpu_launches": 2 * K,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        from oracle.conv_front import conv_front
        ts = min(T, 256)
        t1 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t1 < min(args.cpu_seconds, 5.0) or reps == 0:
            conv_front(c["x"][:ts], c["w"], wl.H, wl.Hv, conv_state=c["state"])
            reps += 1
        dt = time.perf_counter() - t1
        res["cpu_baseline"] = {"value": reps * ts / dt, "unit": "tokens/s", "cores": 1,
                               "kind": "oracle",
                               "sample": f"first {ts} rows, all {C} channels, run {reps} times "
                                         f"({dt:.1f} s of fp64 NumPy on one core)"}
    return res


def timing_variants(call, flush, stream, n):
    """Medians (us) of the same call with L2 left warm between calls, and of the call
    captured once in a CUDA graph and replayed, with and without the L2 flush. Reported
    beside the headline (which flushes L2 and launches eagerly), not instead of it."""
    import torch

    def timed(fn, do_flush):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for i in range(3):
            if do_flush:
                flush.fill_(i & 255)
            fn()
        torch.cuda.synchronize()
        for i in range(n):
            if do_flush:
                flush.fill_((i + 7) & 255)
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return 1000.0 * statistics.median(a.elapsed_time(b) for a, b in evs)

    res = {"warm_l2_us_median": timed(call, False)}
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        call()
        with torch.cuda.graph(graph, stream=side):
            call()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    res["graph_replay_us_median"] = timed(graph.replay, True)
    res["graph_replay_warm_l2_us_median"] = timed(graph.replay, False)
    res["calls_per_variant"] = n
    return res


def run_gdn(args, ws, rank, local):
    import torch
    from gated_delta_rule_chunk_gb300 import binding as B
    from gated_delta_rule_chunk_gb300.build import build
    from gated_delta_rule_chunk_gb300.inputs import WORKLOADS, make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    x = make_inputs(args.workload, T=args.tokens)
    d = {k: (x[k].to(dev) if x.get(k) is not None else None)
         for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")}
    D = x["dk"]
    out = torch.empty(x["T"], x["Hv"], D, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(x["N"], x["Hv"], D, D, dtype=torch.float32, device=dev)
    desc = B.make_desc(x["T"], x["N"], x["H"], x["Hv"], d["q"].dtype, torch.bfloat16, dk=D, dv=D,
                       flags=B.GDN_FLAG_CHANNEL_GATES if x.get("channel_gates") else 0)
    wsp = B.alloc_workspace(desc, dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call(evs=None):
        B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                        d["initial_state"], d["cu_seqlens"], out=out, final_state=fin,
                        workspace=wsp, stage_events=evs)

    # The headline pass brackets each call with two events only: events recorded
    # between the three kernels would keep each launch from overlapping the tail of
    # the one before it. A second pass records the library's stage events for the
    # per-kernel breakdown and the roofline of the dominant kernel.
    K = args.steps

    def make_events(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n)] for _ in range(K)]
        for row in evs:
            for e in row:
                e.record()      # creates the event; recorded again in the timed loop
        return evs

    evs, sevs = make_events(2), make_events(5)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        flush.fill_(i & 255)
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, args.clocks_file)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_((i + 1) & 255)
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    for i in range(K):
        flush.fill_((i + 1) & 255)
        sevs[i][0].record(stream)
        call([e.cuda_event for e in sevs[i][1:]])
    torch.cuda.synchronize()
    step_ms = [r[0].elapsed_time(r[1]) for r in evs]
    st = {"chunk_table": [r[1].elapsed_time(r[2]) for r in sevs],
          "intra": [r[2].elapsed_time(r[3]) for r in sevs],
          "inter": [r[3].elapsed_time(r[4]) for r in sevs]}
    staged_ms = statistics.mean(r[0].elapsed_time(r[4]) for r in sevs)
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, ws)
    tokens = x["n_tokens"]
    value = ws * tokens / (ms_max / 1000.0)
    variants = timing_variants(call, flush, stream, min(K, 200))
    variants["us_median"] = 1000.0 * statistics.median(step_ms)

    # ---------------------------------------------------------------- e2e through host buffers
    host = {k: (x[k].pin_memory() if x.get(k) is not None else None)
            for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    fin_h = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * fin_h.element_size()
    # (1) one step at a time: copy in, call, copy out, wait
    e2e_ms = []
    for i in range(3 + args.e2e_steps if args.e2e_steps > 0 else 0):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for key, t in host.items():
            if t is not None:
                d[key].copy_(t, non_blocking=True)
        call()
        out_h.copy_(out, non_blocking=True)
        fin_h.copy_(fin, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(b))
    # (2) steps in flight, as a prefill server runs them: the inputs of step i + 1 are
    # copied in while step i computes and step i - 1's results are copied out (three
    # streams, two device buffer sets); every step still copies all of its inputs in and
    # its output and final state out, and the time spans all the steps
    e2e_pipe_ms = None
    if args.e2e_steps > 0:
        sets = [(d, out, fin),
                ({k: (torch.empty_like(v) if v is not None else None) for k, v in d.items()},
                 torch.empty_like(out), torch.empty_like(fin))]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def pipelined(n):
            in_ev, comp_ev, out_ev = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
            start = torch.cuda.Event(enable_timing=True)
            stop = torch.cuda.Event(enable_timing=True)
            s_in.wait_stream(stream)
            start.record(s_in)
            for i in range(n):
                di, oi, fi = sets[i & 1]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(comp_ev[i - 2])  # buffer set i & 1 read by step i - 2
                    for key, t in host.items():
                        if t is not None:
                            di[key].copy_(t, non_blocking=True)
                    in_ev[i].record(s_in)
                stream.wait_event(in_ev[i])
                if i >= 2:
                    stream.wait_event(out_ev[i - 2])  # its output and state copied out
                B.gdn_chunk_fwd(di["q"], di["k"], di["v"], di["g"], di["beta"], x["scale"],
                                di["initial_state"], di["cu_seqlens"], out=oi, final_state=fi,
                                workspace=wsp)
                comp_ev[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_ev[i])
                    out_h.copy_(oi, non_blocking=True)
                    fin_h.copy_(fi, non_blocking=True)
                    out_ev[i].record(s_out)
            stop.record(s_out)
            stop.synchronize()
            stream.wait_stream(s_out)
            return start.elapsed_time(stop) / n

        pipelined(3)  # warm-up
        e2e_pipe_ms = pipelined(args.e2e_steps)
    e2e_serial_ms = statistics.mean(e2e_ms) if e2e_ms else None
    e2e_step_ms = e2e_pipe_ms if e2e_pipe_ms is not None else e2e_serial_ms
    e2e_val = (ws * tokens / (max_over_ranks(e2e_step_ms, ws) / 1000.0)
               if e2e_step_ms else None)

    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    sb = stage_bytes(x)
    stage_mean = {k: statistics.mean(v) for k, v in st.items()}
    dom = max(("intra", "inter"), key=stage_mean.get)  # the two kernels that move the bytes
    dom_gbs = sb[dom] / (stage_mean[dom] / 1000.0) / 1e9
    traffic, traffic_src = ncu_traffic(dom, args.workload)
    alg_b, alg_f = algorithmic_bytes(x), algorithmic_flops(x)
    t_hbm = alg_b / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg_f / (peaks["bf16_tflops"] * 1e12)
    t_ns_hbm = alg_b / 8.0e12   # the 8 TB/s reading of the target
    path_roof = {
        "bound": "hbm" if t_hbm >= t_tc else "tensor",
        "algorithmic_bytes": alg_b, "algorithmic_flops": alg_f,
        "roofline_us_measured_peaks": 1e6 * max(t_hbm, t_tc),
        "roofline_us_8tbs": 1e6 * max(t_ns_hbm, alg_f / (peaks["bf16_tflops"] * 1e12)),
        "us_per_call": 1000.0 * ms,
        "frac_of_measured": max(t_hbm, t_tc) / (ms / 1000.0),
        "frac_of_8tbs": max(t_ns_hbm, t_tc) / (ms / 1000.0),
    }
    tc = uses_tc_path(x)
    if tc:
        # The headline roofline is the whole call's: its compulsory bytes (q, k, v, out, g,
        # beta and the states: 25.9 KB per token at the headline shape) over the call's time,
        # against the measured HBM peak (and the 8 TB/s reading beside it). Each kernel's
        # own fraction uses the bytes the method's stage boundary implies (w and u in bf16
        # between the stages); this implementation's bridge-level bytes and the ncu DRAM
        # count stand beside them.
        ssb = method_stage_bytes(x)
        call_gbs = alg_b / (ms / 1000.0) / 1e9
        kernels = {}
        for k in ("intra", "inter"):
            kb = ssb[k] / (stage_mean[k] / 1000.0) / 1e9
            tr, tsrc = ncu_traffic(k, args.workload)
            kernels[k] = {"us": 1000.0 * stage_mean[k], "algorithmic_bytes_per_launch": ssb[k],
                          "achieved_gbs": kb, "frac": kb / peaks["hbm_gbs"],
                          "bridge_bytes_per_launch": sb[k], "traffic": tr,
                          "traffic_over_algorithmic": (tr / ssb[k]) if tr else None,
                          "traffic_source": tsrc}
        tr_all = [kernels[k]["traffic"] for k in ("intra", "inter")]
        roof = {"bound": "hbm", "kernel": "whole call (chunk table, intra, scan)",
                "achieved": call_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": call_gbs / peaks["hbm_gbs"], "frac_of_8tbs": call_gbs / 8000.0,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": alg_b,
                "traffic": (sum(tr_all) if all(t is not None for t in tr_all) else None),
                "dominant_kernel": dom, "kernel_frac": kernels[dom]["frac"],
                "kernels": kernels}
    else:
        # the fp32 SIMT kernels: FMA-pipe bound; peak from the unit counts and clock
        sf = stage_flops(x)
        achieved = sf[dom] / (stage_mean[dom] / 1000.0) / 1e12
        roof = {"bound": "alu", "kernel": dom, "achieved": achieved, "peak": SIMT_FP32_TFLOPS,
                "unit": "TFLOP/s", "frac": achieved / SIMT_FP32_TFLOPS,
                "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 FLOP x 2.07 GHz",
                "algorithmic_flops_per_launch": sf[dom],
                "hbm_frac": dom_gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": sb[dom],
                "traffic": traffic, "traffic_source": traffic_src}
    metric = gdn_metric(args.workload)
    res = {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if tc else "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload].name, "T": x["T"], "N": x["N"],
                   "H": x["H"], "Hv": x["Hv"], "dk": x["dk"], "dv": x["dv"], "chunk": CHUNK,
                   "gates": "per key channel" if x.get("channel_gates") else "per token",
                   "kernels": "tensor-core (tcgen05) intra + scan" if tc else "fp32 SIMT intra + scan",
                   "qkv_dtype": "bf16", "out_dtype": "bf16", "g_beta_state_dtype": "fp32",
                   "initial_state": x["initial_state"] is not None,
                   "l2": "512 MiB buffer written between timed steps (L2 is 129 MB)",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "inputs": "resident in HBM"},
        "roofline": roof,
        "path_roofline": path_roof,
        "stages_us": {k: 1000.0 * v for k, v in stage_mean.items()},
        "us_per_call_with_stage_events": 1000.0 * staged_ms,
        "timing_variants": variants,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step_ms,
                "mode": "pipelined: step i+1's inputs copied in while step i computes and "
                        "step i-1's results are copied out (3 streams, 2 device buffer sets)",
                "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": 3 * K,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        rate, ts, dt, cores, reps = oracle_rate(x, args.cpu_seconds)
        what = (f"the whole workload ({ts} tokens), all {x['Hv']} value heads, run {reps} times"
                if reps > 1 else f"first {ts} tokens of the workload, all {x['Hv']} value heads")
        # the same oracle on one thread, on a shorter sample
        rate1, ts1, dt1, _, _ = oracle_rate(x, max(1.0, args.cpu_seconds / 4), nthreads=1)
        res["cpu_baseline"] = {
            "value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{what} ({dt:.1f} s of fp64 C on the host cores)",
            "cpu_model": cpu_model(),
            "value_1thread": rate1,
            "sample_1thread": f"first {ts1} tokens, all {x['Hv']} value heads, one thread "
                              f"({dt1:.1f} s)"}
    return res


def bwd_bytes(x):
    """Compulsory HBM bytes of one backward call: q, k, v, g, beta, the initial state and
    the upstream gradients in; dq, dk, dv, dg, dbeta and the initial-state gradient out."""
    esz = 2 if x["dtype"] == "bf16" else 4
    T, H, Hv, D, N = x["n_tokens"], x["H"], x["Hv"], x["dk"], x["N"]
    st = N * Hv * D * D * 4
    ins = 2 * T * H * D * esz + T * Hv * D * esz + 2 * T * Hv * 4 + st + T * Hv * D * 4 + st
    outs = 2 * T * H * D * 4 + T * Hv * D * 4 + 2 * T * Hv * 4 + st
    return ins + outs


def bwd_stage_flops(x):
    """FLOPs of the backward's four stages (64 x 64 and 64 x d products counted in full):
    the forward recompute (intra kernel, and w S plus the state update of the scan), the
    reverse scan (Kt dS, M^T dO, Qt^T dO, w^T dv_new), the three contractions with the
    stored states (dO S^T, dv_new S^T, v_new dS^T) and the per-chunk kernels (K K^T, Q K^T,
    the inverse, dP, Z, T^T dv_new, T^T dw, T^T Z T^T and the dq / dk products)."""
    NT = n_chunks(x["lengths"])
    C, D, Hv = CHUNK, x["dk"], x["Hv"]
    intra = stage_flops(x)["intra"]
    recompute = intra + NT * Hv * (2 * 2 * C * D * D)
    scan = NT * Hv * (6 * C * D * D + 2 * C * C * D)
    state = NT * Hv * (6 * C * D * D)
    chunk = NT * Hv * (20 * C * C * D + 4 * C ** 3 + C ** 3 / 3)
    return {"recompute": recompute, "reverse_scan": scan, "state_products": state,
            "chunk_grads": chunk}


def bwd_state_bytes(x):
    """Algorithmic bytes of the state contractions per call: per (chunk, value head) the
    chunk-start state and its gradient (fp32 D x D each), v_new and dv_new (fp32 64 x D),
    dO (64 x D) in; dO S^T, dw and v_new dS^T (fp32 64 x D) out."""
    NT = n_chunks(x["lengths"])
    D, Hv = x["dk"], x["Hv"]
    return NT * Hv * (2 * D * D * 4 + 2 * 64 * D * 4 + 64 * D * 4 + 3 * 64 * D * 4)


def run_gdn_bwd(args, ws, rank, local):
    import torch
    from gated_delta_rule_chunk_gb300 import binding as B
    from gated_delta_rule_chunk_gb300.build import build
    from gated_delta_rule_chunk_gb300.inputs import WORKLOADS, make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    x = make_inputs(args.workload, T=args.tokens)
    if x.get("channel_gates"):
        raise SystemExit("the backward pass takes scalar gates")
    gen = torch.Generator().manual_seed(77)
    D = x["dk"]
    do_h = torch.randn(x["T"], x["Hv"], D, generator=gen, dtype=torch.float64).float()
    dfin_h = torch.randn(x["N"], x["Hv"], D, D, generator=gen, dtype=torch.float64).float()
    d = {k: (x[k].to(dev) if x.get(k) is not None else None)
         for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")}
    do, dfin = do_h.to(dev), dfin_h.to(dev)
    f32 = torch.float32
    T, H, Hv, N = x["T"], x["H"], x["Hv"], x["N"]
    grads = dict(dq=torch.zeros(T, H, D, dtype=f32, device=dev),
                 dk=torch.zeros(T, H, D, dtype=f32, device=dev),
                 dv=torch.zeros(T, Hv, D, dtype=f32, device=dev),
                 dg=torch.zeros(T, Hv, dtype=f32, device=dev),
                 dbeta=torch.zeros(T, Hv, dtype=f32, device=dev),
                 d_initial_state=torch.zeros(N, Hv, D, D, dtype=f32, device=dev))
    desc = B.make_desc(T, N, H, Hv, d["q"].dtype, f32, dk=D, dv=D)
    wsp = torch.empty(int(B.load_library().gdn_bwd_workspace_size(__import__("ctypes").byref(desc))),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call(evs=None):
        B.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do, x["scale"],
                        d["initial_state"], d["cu_seqlens"], dfin, workspace=wsp, grads=grads,
                        stage_events=evs)

    K = args.steps
    mk = lambda n: [[torch.cuda.Event(enable_timing=True) for _ in range(n)] for _ in range(K)]
    evs, sevs = mk(2), mk(6)
    for row in evs + sevs:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(args.warmup):
        flush.fill_(i & 255)
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, args.clocks_file)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_((i + 1) & 255)
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    for i in range(K):
        flush.fill_((i + 1) & 255)
        sevs[i][0].record(stream)
        call([e.cuda_event for e in sevs[i][1:]])
    torch.cuda.synchronize()
    ms = statistics.mean(r[0].elapsed_time(r[1]) for r in evs)
    names = ("recompute", "reverse_scan", "state_products", "chunk_grads")
    st = {nm: statistics.mean(r[j + 1].elapsed_time(r[j + 2]) for r in sevs)
          for j, nm in enumerate(names)}
    ms_max = max_over_ranks(ms, ws)
    tokens = x["n_tokens"]
    value = ws * tokens / (ms_max / 1000.0)

    # end to end through host buffers: inputs and upstream gradients in, gradients out
    host = {k: (x[k].pin_memory() if x.get(k) is not None else None)
            for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")}
    do_p, dfin_p = do_h.pin_memory(), dfin_h.pin_memory()
    outs_h = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in grads.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    h2d += do_p.numel() * 4 + dfin_p.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in outs_h.values())
    e2e_ms = []
    for i in range(3 + args.e2e_steps if args.e2e_steps > 0 else 0):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for key, t in host.items():
            if t is not None:
                d[key].copy_(t, non_blocking=True)
        do.copy_(do_p, non_blocking=True)
        dfin.copy_(dfin_p, non_blocking=True)
        call()
        for key, t in outs_h.items():
            t.copy_(grads[key], non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(b))
    e2e_val = (ws * tokens / (max_over_ranks(statistics.mean(e2e_ms), ws) / 1000.0)
               if e2e_ms else None)
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    sf = bwd_stage_flops(x)
    dom = max(st, key=st.get)
    achieved = sf[dom] / (st[dom] / 1000.0) / 1e12
    alg_b, alg_f = bwd_bytes(x), sum(sf.values())
    t_hbm = alg_b / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg_f / (peaks["bf16_tflops"] * 1e12)
    tensor_stage = x["dtype"] == "bf16" or dom in ("state_products", "chunk_grads")
    if dom == "state_products":  # warp-MMA contractions: bound by HBM
        sb = bwd_state_bytes(x)
        gbs = sb / (st[dom] / 1000.0) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": gbs, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": sb, "traffic": None, "traffic_source": None}
    elif tensor_stage:
        # fp32 products run as three bf16 warp MMAs (hi*hi + hi*lo + lo*hi): the peak is a
        # third of the measured bf16 tensor rate
        peak3 = peaks["bf16_tflops"] / 3.0
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak3,
                "unit": "TFLOP/s", "frac": achieved / peak3,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops) / 3: fp32 "
                               "products as three bf16 MMAs",
                "algorithmic_flops_per_launch": sf[dom], "traffic": None,
                "traffic_source": None, "fp32_fma_frac": achieved / SIMT_FP32_TFLOPS}
    else:
        roof = {"bound": "alu", "kernel": dom, "achieved": achieved,
                "peak": SIMT_FP32_TFLOPS, "unit": "TFLOP/s",
                "frac": achieved / SIMT_FP32_TFLOPS,
                "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 FLOP x 2.07 GHz",
                "algorithmic_flops_per_launch": sf[dom], "traffic": None,
                "traffic_source": None}
    if x["dtype"] == "bf16":
        kinds = ("tensor-core recompute and reverse scan" if D == 128 else
                 "tensor-core recompute, fp32 SIMT reverse scan")
    else:
        kinds = "fp32 SIMT recompute and reverse scan"
    kinds += ", warp-MMA state contractions and per-chunk gradients"
    res = {
        "metric": f"GDN chunk backward tokens/s, {WORKLOADS[args.workload].name}; % of roofline",
        "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload].name, "pass": "backward",
                   "T": T, "N": N, "H": H, "Hv": Hv, "dk": D, "dv": D, "chunk": CHUNK,
                   "qkv_dtype": x["dtype"], "grad_dtype": "fp32", "d_out_dtype": "fp32",
                   "kernels": kinds,
                   "l2": "512 MiB buffer written between timed steps (L2 is 129 MB)",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "inputs": "resident in HBM"},
        "roofline": roof,
        "path_roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor",
                          "algorithmic_bytes": alg_b, "algorithmic_flops": alg_f,
                          "roofline_us_measured_peaks": 1e6 * max(t_hbm, t_tc),
                          "us_per_call": 1000.0 * ms,
                          "frac_of_measured": max(t_hbm, t_tc) / (ms / 1000.0),
                          "simt_alu_us": 1e6 * alg_f / (SIMT_FP32_TFLOPS * 1e12)},
        "stages_us": {k: 1000.0 * v for k, v in st.items()},
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "ms_per_step": statistics.mean(e2e_ms) if e2e_ms else None},
        "gpu_launches": 7 * K,   # chunk table, intra, scan, reverse scan, 3 chunk kernels
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        rate, ts, dt, cores = oracle_bwd_rate(x, do_h, dfin_h, args.cpu_seconds)
        res["cpu_baseline"] = {
            "value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {ts} tokens of the workload, all {Hv} value heads, backward "
                      f"({dt:.1f} s of fp64 C on the host cores)"}
    return res


def oracle_bwd_rate(x, do, dfin, seconds):
    """Time the oracle's backward on the first T_s tokens (all heads), T_s sized from a probe."""
    import oracle
    import torch

    def run(ts):
        cu = torch.tensor([0, ts], dtype=torch.int32)
        sl = slice(0, ts)
        s0 = x["initial_state"][:1] if x["initial_state"] is not None else None
        t = time.perf_counter()
        oracle.recurrent_backward(x["q"][sl], x["k"][sl], x["v"][sl], x["g"][sl],
                                  x["beta"][sl], x["scale"], s0, cu, do[sl], dfin[:1])
        return time.perf_counter() - t

    oracle.build()
    probe = min(64, x["n_tokens"])
    dt = run(probe)
    ts = int(max(16, min(x["n_tokens"], probe * seconds / max(dt, 1e-6))))
    ts = max(16, ts // 16 * 16)
    dt = run(ts)
    return ts / dt, ts, dt, oracle.max_threads()


def main(argv=None):
    args = parse_args(argv)
    ws, rank, local = dist_env()
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "gdn" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            res = run_reference(args, ws, rank)
        else:
            from gated_delta_rule_chunk_gb300.inputs import WORKLOADS
            if WORKLOADS[args.workload].kind == "fixed":
                res = run_recurrent(args, ws, rank, local)
            elif WORKLOADS[args.workload].kind == "conv":
                res = run_conv(args, ws, rank, local)
            elif args.backward:
                res = run_gdn_bwd(args, ws, rank, local)
            else:
                res = run_gdn(args, ws, rank, local)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
