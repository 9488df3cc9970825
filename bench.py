#!/usr/bin/env python
"""Benchmark of the Simple GLA hot path on GB300.

Step = one chunked prefill (``sala_gla_chunk_fwd``) of the MiniCPM-SALA lightning-layer
workload: B=1, T=8192, H=32, d=128, bf16 q/k/v with RMS-normalised q/k, fixed per-head
log-decay g_h = -2^(-8(h+1)/32), h0 = 0, returning o and the final state. Inputs are synthetic
and seeded, resident in HBM before the timed region; two input sets alternate between steps
and each set (201 MB of q/k/v plus 67 MB of o) is larger than the 126 MB L2.

Prints ONE JSON line (rank 0). Beside the headline prefill number it reports: the roofline
of the dominant kernel (per-kernel CUDA-event time measured inside the timed region by the
library's timing instrumentation), the end-to-end rate through the C ABI with host buffers
(host->device copies of q/k/v/g and device->host copies of o/hT inside the timed region), the
fp64 CPU oracle timed on the host cores on a bounded sample, the SM clocks sampled during the
run, and the batched recurrent decode workload (256 sequences x 32 heads, 1000 consecutive
steps on a 512 MB fp32 state updated in place) in GB/s against the HBM roofline.

``--impl reference`` times the fp64 oracle instead (the reference arm of this benchmark).
Multi-GPU (torchrun): every rank runs its own copy of the workload (weak scaling; prefill units
are independent, no data-path collective); the timing is the max over ranks.
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

METRIC = "prefill tokens/s (H=32,d=128) and decode HBM GB/s, as % of GB300 roofline"
D = 128


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sala_layer")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other prefill workloads (tiny, varlen, long)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="decode steps to run (default: the workload's 1000; fewer for profiling)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


# ---------------------------------------------------------------------------------------
# distributed plumbing (timing only: barriers and a max over ranks)


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------------------
# clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            self.t0 = time.time()
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), max=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                     active=parts[4], hw=parts[5], hwt=parts[6], swt=parts[7],
                                     pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        return rows


def summarise_clocks(rows):
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    # samples under load: the upper half by power draw
    pw = sorted(r["power"] for r in rows)
    cut = pw[len(pw) // 2] if pw else 0.0
    loaded = [r for r in rows if r["power"] >= cut] or rows
    reasons = set()
    for r in loaded:
        if r["hw"] == "Active":
            reasons.add("hw_slowdown")
        if r["hwt"] == "Active":
            reasons.add("hw_thermal_slowdown")
        if r["swt"] == "Active":
            reasons.add("sw_thermal_slowdown")
        if r["pcap"] == "Active":
            reasons.add("sw_power_cap")
    return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
            "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
            "samples": len(loaded), "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------------------
# byte / flop accounting (algorithmic: each input read once, each output written once)


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture of
# one launch of each kernel as it stands (-k <kernel> -c 1), on the workload the bench times;
# retaken whenever a kernel changes (None: not measured since the last change).
MEASURED_TRAFFIC = {"prefill_fused": 251_700_000, "prefill_fused_varlen": 2_615_000_000,
                    "prefill_fused_long": 5_140_000_000, "prefill_pair_long": 6_122_000_000,
                    "prefill_pair_varlen": 3_113_000_000, "recurrent_step": 1_021_800_000,
                    "recurrent_step_indexed": 486_100_000, "output_norm_gate": 160_700_000,
                    "qk_prologue": 211_300_000, "gdn_step": 1_022_200_000,
                    "gdn_fwd": 775_600_000}


def prefill_bytes(T, H, nseq, has_h0, has_hT):
    per_token = H * (3 * D * 2 + 4 + D * 2)      # q, k, v bf16 + g fp32 + o bf16
    state = nseq * H * D * D * 4
    return T * per_token + (state if has_h0 else 0) + (state if has_hT else 0)


def prefill_flops(T, H):
    # causal intra-chunk QK^T and PV (2 d (C+1) per token), Q S and K^T V (2 d^2 each)
    return T * H * (2 * D * (64 + 1) + 4 * D * D)


def decode_bytes(N, H):
    return N * H * (2 * D * D * 4 + 3 * D * 2 + 4 + D * 2)


def decode_pool_bytes(N, H, state_bytes):
    # the N addressed states read and written, q, k, v, g read, o written, the slot indices
    return N * H * (2 * D * D * state_bytes + 3 * D * 2 + 4 + D * 2) + N * 4


# ---------------------------------------------------------------------------------------
# the oracle on the host cores (reference arm and CPU baseline)


def oracle_sample_rate(x, tokens, reps=1):
    """tokens/s of the fp64 oracle on the first `tokens` tokens (all heads) of workload x."""
    import oracle
    q, k, v, g = (x[n][:, :tokens] for n in ("q", "k", "v", "g"))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.recurrent(q, k, v, g, x["scale"], h0=None)
    dt = time.perf_counter() - t0
    return tokens * reps / dt, dt


def cpu_baseline(x, target_s):
    """The oracle on a bounded sample of the workload: a prefix of the tokens (all heads),
    repeated whole passes if the full workload takes less than the target time."""
    import oracle
    T = x["q"].shape[1]
    probe = min(T, 256)
    _, dt = oracle_sample_rate(x, probe)
    want = probe * target_s / max(dt, 1e-6)          # tokens the target time would cover
    tokens = int(min(T, max(probe, want)))
    tokens = max(64, (tokens // 64) * 64) if T >= 64 else T
    reps = max(1, int(round(want / tokens))) if tokens == T else 1
    rate, dt = oracle_sample_rate(x, tokens, reps)
    return {"value": rate, "unit": "tokens/s", "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": f"fp64 recurrence over the first {tokens} of {T} tokens x all "
                      f"{x['q'].shape[2]} heads of the same workload, {reps} pass(es), "
                      f"{dt:.1f} s"}


def run_reference(args, dist):
    from gated_linear_attention_gb300 import inputs
    import oracle
    oracle.build()
    if dist.rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    x = inputs.make_prefill(w)
    tokens = min(w.T, 1024)
    for _ in range(args.warmup):
        oracle_sample_rate(x, tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_rate(x, tokens)
    dt = time.perf_counter() - t0
    value = tokens * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": 1, "T": w.T, "H": w.H, "d": D, "chunk": 64,
                   "description": w.description},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.default_threads(),
                         "kind": "oracle",
                         "sample": f"each step: fp64 recurrence over the first {tokens} of "
                                   f"{w.T} tokens x all {w.H} heads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# our arm


def run_ours(args, dist):
    import torch
    torch.cuda.set_device(dist.local)
    dist.init("nccl")
    from gated_linear_attention_gb300 import build as libbuild
    if dist.rank == 0:
        libbuild.build()
    dist.barrier()
    from gated_linear_attention_gb300 import inputs, sala_gla
    sala_gla.load()
    peaks = load_peaks()
    dev = torch.device("cuda", dist.local)
    w = inputs.WORKLOADS[args.workload]
    assert w.kind == "prefill"

    # two input sets (the second with another seed), resident in HBM
    host = inputs.make_prefill(w, seed=w.seed + 1000 * dist.rank)
    alt = inputs.make_prefill(w, seed=w.seed + 1000 * dist.rank + 500)
    sets = []
    for x in (host, alt):
        sets.append({n: (x[n].to(dev) if x[n] is not None else None)
                     for n in ("q", "k", "v", "g", "h0", "cu_seqlens")})
    T_total = host["q"].shape[0] * host["q"].shape[1] if host["q"].dim() == 4 else host["q"].shape[0]
    nseq = len(w.seqlens)
    outs = [(torch.empty_like(s["q"]), torch.empty((nseq, w.H, D, D), device=dev))
            for s in sets]
    scale = host["scale"]

    def step(i):
        s, (o, hT) = sets[i % 2], outs[i % 2]
        sala_gla.chunk_fwd(s["q"], s["k"], s["v"], s["g"], scale, h0=s["h0"],
                           cu_seqlens=s["cu_seqlens"], o=o, hT=hT)

    clocks = ClockSampler(dist.local)
    clocks.start()
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    assert sala_gla.get_device_status() == 0

    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ms = ev0.elapsed_time(ev1)
    # per-kernel CUDA events on the launching stream, in a second timed pass of the same K
    # steps: recording them adds host work between launches, so the step time above is taken
    # without them
    sala_gla.timing_enable(True)
    for i in range(args.steps):
        step(i)
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()
    step_pct = call_percentiles(stream, step, args.steps)
    ms_max = dist.max(ms)
    tokens_all = dist.sum(T_total * args.steps)
    value = tokens_all / (ms_max / 1e3)
    launches = sum(n for _, n in kern.values())

    # dominant kernel and its roofline (algorithmic bytes per launch / mean launch time)
    top = max(kern.items(), key=lambda kv: kv[1][0])
    top_name, (top_ms, top_n) = top
    # the fused prefill kernel moves the whole step's algorithmic bytes: q, k, v, g read
    # once, o written once, h0 read and hT written once per (sequence, head)
    bytes_per_kernel = {
        "prefill_fused": prefill_bytes(T_total, w.H, nseq, host["h0"] is not None, True),
        "prefill_pair": prefill_bytes(T_total, w.H, nseq, host["h0"] is not None, True),
    }
    if top_name in bytes_per_kernel and top_n:
        ach = bytes_per_kernel[top_name] / (top_ms / top_n / 1e3) / 1e9
        traffic = MEASURED_TRAFFIC.get(top_name) if w.name == "sala_layer" else None
        roof = {"kernel": top_name, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": peaks["source"], "mean_launch_us": 1e3 * top_ms / top_n}
    else:
        roof = {"kernel": top_name, "bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": None, "traffic": None}
    step_bytes = prefill_bytes(T_total, w.H, nseq, host["h0"] is not None, True)
    step_roof_rate = T_total / (step_bytes / (peaks["hbm_gbs"] * 1e9))
    kernels = {k: {"ms_total": v[0], "launches": v[1],
                   "us_per_launch": (1e3 * v[0] / v[1]) if v[1] else None}
               for k, v in kern.items() if v[1]}

    # end to end through the C ABI with host buffers: every step copies its q, k, v, g from
    # pinned host memory, runs the prefill and reads o and hT back. Steps are pipelined over
    # three streams with two buffer sets, as a serving loop would run them: the copy in of
    # step i + 1 and the copy out of step i - 1 overlap the prefill of step i (one more copy
    # stream for the copy in measured the same: the host link is the limit).
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hg = (host[n].pin_memory() for n in ("q", "k", "v", "g"))
        hos = [torch.empty(host["q"].shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        hhs = [torch.empty((nseq, w.H, D, D), dtype=torch.float32).pin_memory() for _ in range(2)]
        dbufs = []
        for _ in range(2):
            dq, dk, dv, dg = (torch.empty_like(t, device=dev) for t in (hq, hk, hv, hg))
            dbufs.append((dq, dk, dv, dg, torch.empty_like(dq), torch.empty((nseq, w.H, D, D), device=dev)))
        s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_done, run_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        for e_ in run_done + out_done:
            e_.record(stream)

        def e2e_step(i):
            b = i % 2
            dq, dk, dv, dg, do, dh = dbufs[b]
            s_in.wait_event(run_done[b])            # step i - 2 has read these inputs
            with torch.cuda.stream(s_in):
                for d_, h_ in ((dq, hq), (dk, hk), (dv, hv), (dg, hg)):
                    d_.copy_(h_, non_blocking=True)
                in_done[b].record(s_in)
            s_run.wait_event(in_done[b])
            s_run.wait_event(out_done[b])           # step i - 2's outputs have been read back
            sala_gla.chunk_fwd(dq, dk, dv, dg, scale, o=do, hT=dh, stream=s_run)
            run_done[b].record(s_run)
            s_out.wait_event(run_done[b])
            with torch.cuda.stream(s_out):
                hos[b].copy_(do, non_blocking=True)
                hhs[b].copy_(dh, non_blocking=True)
                out_done[b].record(s_out)

        for i in range(max(3, args.warmup)):
            e2e_step(i)
        dist.barrier()
        torch.cuda.synchronize()
        ev0.record(s_in)
        for i in range(args.steps):
            e2e_step(i)
        for b in range(2):
            s_out.wait_event(out_done[b])
        ev1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = dist.max(ev0.elapsed_time(ev1))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg))
        d2h = hos[0].numel() * 2 + hhs[0].numel() * 4
        e2e = {"value": tokens_all / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "pipeline": "copy-in, prefill and copy-out on three streams, two buffer sets"}
        del dbufs

    # batched recurrent decode: 1000 consecutive steps, state updated in place
    decode = None
    if not args.no_decode:
        decode = run_decode(args, dist, dev, peaks, sala_gla, inputs)
        launches_decode = decode.pop("_launches")
        launches_decode += decode["pooled"].pop("_launches")
        launches_decode += decode["gdn"].pop("_launches")
    else:
        launches_decode = 0

    # the layer's output RMSNorm and sigmoid gate on the prefill's output shape, and its q/k
    # prologue (RMSNorm + RoPE) on the prefill's q and k
    gate = prologue = gdn_prefill = None
    if not args.no_decode:
        gate = run_output_gate(args, dist, dev, peaks, sala_gla, inputs, T_total, w.H)
        launches_decode += gate.pop("_launches")
        prologue = run_qk_prologue(args, dist, dev, peaks, sala_gla, inputs, T_total, w.H)
        launches_decode += prologue.pop("_launches")
        gdn_prefill = run_gdn_prefill(args, dist, dev, peaks, sala_gla, inputs)
        launches_decode += gdn_prefill.pop("_launches")
        launches_decode += gdn_prefill["chunked"].pop("_launches")

    # the other prefill workloads: varlen (8 packed sequences, 66,560 tokens, h0), long
    # (131,072 tokens, h0) and tiny (256 tokens, 4 heads)
    configs = None
    if not args.no_configs:
        configs = {}
        for name in ("varlen", "long", "tiny"):
            configs[name] = run_prefill_config(args, dist, dev, peaks, sala_gla, inputs, name)
            launches_decode += configs[name].pop("_launches")

    rows = clocks.stop()

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(host, args.cpu_seconds)

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": 1, "T": w.T, "H": w.H, "d": D, "chunk": 64,
                       "parallelism": f"replica x{dist.world} (independent prefills)",
                       "l2": "inputs larger than L2 (201 MB q/k/v per set), two sets alternated",
                       "description": w.description},
            "roofline": roof,
            "step_roofline": {"bytes_per_step": step_bytes,
                              "roofline_tokens_per_s": step_roof_rate,
                              "frac": (value / dist.world) / step_roof_rate},
            "step_us_percentiles": step_pct,
            "kernels": kernels,
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": summarise_clocks(rows),
            "decode": decode,
            "output_gate": gate,
            "qk_prologue": prologue,
            "gdn_prefill": gdn_prefill,
            "prefill_configs": configs,
            "gpu_launches_decode": launches_decode,
        }
        print(json.dumps(line), flush=True)
    dist.close()


def run_prefill_config(args, dist, dev, peaks, sala_gla, inputs, name):
    """One more prefill workload, timed like the headline one: inputs resident in HBM, W
    warm-up calls, K timed calls between CUDA events on the launching stream (max over
    ranks), then a second pass of K calls with the library's per-kernel events for the
    dominant kernel's roofline. One input set: varlen (1.6 GB of q, k, v) and long (3.2 GB)
    are far larger than L2 on their own; tiny (1 MB) stays in L2 and is a latency figure."""
    import torch
    w = inputs.WORKLOADS[name]
    x = inputs.make_prefill(w, seed=w.seed + 1000 * dist.rank)
    s = {n: (x[n].to(dev) if x[n] is not None else None)
         for n in ("q", "k", "v", "g", "h0", "cu_seqlens")}
    T_total = x["q"].shape[0] * x["q"].shape[1] if x["q"].dim() == 4 else x["q"].shape[0]
    nseq = len(w.seqlens)
    o = torch.empty_like(s["q"])
    hT = torch.empty((nseq, w.H, D, D), device=dev)

    def step():
        sala_gla.chunk_fwd(s["q"], s["k"], s["v"], s["g"], x["scale"], h0=s["h0"],
                           cu_seqlens=s["cu_seqlens"], o=o, hT=hT)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert sala_gla.get_device_status() == 0
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(ev0.elapsed_time(ev1))
    sala_gla.timing_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()
    step_pct = call_percentiles(stream, lambda i: step(), args.steps)
    assert sala_gla.get_device_status() == 0
    has_h0 = x["h0"] is not None
    nbytes = prefill_bytes(T_total, w.H, nseq, has_h0, True)
    # the per-call choice of sala_gla_chunk_fwd: the two-CTA kernel on many-wave workloads
    kname = "prefill_pair" if kern.get("prefill_pair", (0.0, 0))[1] else "prefill_fused"
    k_ms, k_n = kern[kname]
    k_ach = nbytes / (k_ms / k_n / 1e3) / 1e9
    value = dist.sum(T_total * args.steps) / (ms / 1e3)
    step_rate = T_total / (nbytes / (peaks["hbm_gbs"] * 1e9))
    del s, o, hT
    torch.cuda.empty_cache()
    return {
        "metric": "prefill tokens/s", "value": value, "unit": "tokens/s",
        "ms_per_step": ms / args.steps,
        "config": {"workload": w.name, "T": T_total, "H": w.H, "d": D, "sequences": nseq,
                   "h0": has_h0, "bytes_per_step": nbytes,
                   "l2": "L2-resident (latency)" if nbytes < 64e6 else "inputs larger than L2",
                   "description": w.description},
        "roofline": {"kernel": kname, "bound": "hbm", "achieved": k_ach,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": k_ach / peaks["hbm_gbs"],
                     "traffic": MEASURED_TRAFFIC.get(kname + "_" + w.name),
                     "peak_source": peaks["source"], "mean_launch_us": 1e3 * k_ms / k_n},
        "step_roofline": {"bytes_per_step": nbytes, "roofline_tokens_per_s": step_rate,
                          "frac": (value / dist.world) / step_rate},
        "step_us_percentiles": step_pct,
        "kernels": {k: {"ms_total": v[0], "launches": v[1],
                        "us_per_launch": (1e3 * v[0] / v[1]) if v[1] else None}
                    for k, v in kern.items() if v[1]},
        "_launches": sum(n for _, n in kern.values()),
    }


def run_decode(args, dist, dev, peaks, sala_gla, inputs):
    import torch
    w = inputs.WORKLOADS["decode"]
    if args.decode_steps is not None:
        import dataclasses
        w = dataclasses.replace(w, steps=max(args.decode_steps, max(3, args.warmup)))
    x = inputs.make_decode_steps(w)
    S0 = inputs.make_decode_state(w)
    q, k, v, g = (x[n].to(dev) for n in ("q", "k", "v", "g"))
    S = S0.to(dev)
    o = torch.empty_like(q[0])
    scale = x["scale"]
    # warm-up on a scratch copy of the state, then restore it
    Sw = S.clone()
    for s in range(max(3, args.warmup)):
        sala_gla.recurrent_step(q[s], k[s], v[s], g[s], scale, Sw, o=o)
    torch.cuda.synchronize()
    del Sw
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sala_gla.timing_enable(True)
    ev0.record(stream)
    for s in range(w.steps):
        sala_gla.recurrent_step(q[s], k[s], v[s], g[s], scale, S, o=o)
    ev1.record(stream)
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()["recurrent_step"]
    ms = dist.max(ev0.elapsed_time(ev1))
    per_step = decode_bytes(w.nseq, w.H)
    gbs = per_step * w.steps / (ms / 1e3) / 1e9 * dist.world
    k_ach = per_step / (kern[0] / kern[1] / 1e3) / 1e9
    pooled = run_decode_pool(args, dist, peaks, sala_gla, inputs, w, q, k, v, g, o, scale)
    gdn = run_gdn_decode(args, dist, peaks, sala_gla, inputs, w, q, k, v, g, o, scale, S0)
    return {
        "pooled": pooled,
        "gdn": gdn,
        "metric": "decode HBM GB/s", "value": gbs, "unit": "GB/s",
        "ms_per_step": ms / w.steps, "tokens_per_s": w.nseq * w.steps / (ms / 1e3) * dist.world,
        "config": {"workload": w.name, "N": w.nseq, "H": w.H, "d": D, "steps": w.steps,
                   "state_bytes": w.nseq * w.H * D * D * 4, "bytes_per_step": per_step},
        "roofline": {"kernel": "recurrent_step", "bound": "hbm", "achieved": k_ach,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": k_ach / peaks["hbm_gbs"],
                     "traffic": MEASURED_TRAFFIC["recurrent_step"] if w.nseq == 256 else None,
                     "peak_source": peaks["source"], "mean_launch_us": 1e3 * kern[0] / kern[1]},
        "_launches": kern[1],
    }


def run_gdn_decode(args, dist, peaks, sala_gla, inputs, wd, q, k, v, g, o, scale, S0):
    """The same decode steps under the gated delta rule (sala_gla_gdn_recurrent_step): the
    decode workload's tokens and initial states, write strengths beta = sigmoid(N(0, 1)) of
    the gdn_decode workload; the state flows step to step."""
    import torch
    w = inputs.WORKLOADS["gdn_decode"]
    beta = inputs.make_gdn_beta(w, 0, wd.steps, nseq=wd.nseq, H=wd.H).to(q.device)
    S = S0.to(q.device)
    Sw = S.clone()
    for s in range(max(3, args.warmup)):
        sala_gla.gdn_recurrent_step(q[s], k[s], v[s], g[s], beta[s], scale, Sw, o=o)
    torch.cuda.synchronize()
    del Sw
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    sala_gla.timing_enable(True)
    ev0.record(stream)
    for s in range(wd.steps):
        sala_gla.gdn_recurrent_step(q[s], k[s], v[s], g[s], beta[s], scale, S, o=o)
    ev1.record(stream)
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()["gdn_step"]
    assert sala_gla.get_device_status() == 0
    ms = dist.max(ev0.elapsed_time(ev1))
    per_step = decode_bytes(wd.nseq, wd.H) + wd.nseq * wd.H * 4     # + beta
    k_ach = per_step / (kern[0] / kern[1] / 1e3) / 1e9
    return {
        "metric": "gated-delta-rule decode HBM GB/s", "value": per_step * wd.steps / (ms / 1e3) / 1e9 * dist.world,
        "unit": "GB/s", "ms_per_step": ms / wd.steps,
        "tokens_per_s": wd.nseq * wd.steps / (ms / 1e3) * dist.world,
        "config": {"workload": w.name, "N": wd.nseq, "H": wd.H, "d": D, "steps": wd.steps,
                   "bytes_per_step": per_step,
                   "tokens": "the decode workload's q, k, v, g and initial states; beta of gdn_decode"},
        "roofline": {"kernel": "gdn_step", "bound": "hbm", "achieved": k_ach,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": k_ach / peaks["hbm_gbs"],
                     "traffic": MEASURED_TRAFFIC["gdn_step"] if (wd.nseq, wd.H) == (256, 32) else None,
                     "peak_source": peaks["source"], "mean_launch_us": 1e3 * kern[0] / kern[1]},
        "_launches": kern[1],
    }


def run_decode_pool(args, dist, peaks, sala_gla, inputs, wd, q, k, v, g, o, scale):
    """The same decode steps on states kept in a pool of 512 slots stored in bf16 and
    addressed through a slot permutation (sala_gla_recurrent_step_indexed). The per-step
    tokens are the decode workload's, already resident."""
    import dataclasses
    import torch
    w = dataclasses.replace(inputs.WORKLOADS["decode_pool"], steps=wd.steps)
    p = inputs.make_decode_pool(w)
    dev = q.device
    pool, idx = p["pool"].to(dev), p["indices"].to(dev)
    for s in range(max(3, args.warmup)):
        sala_gla.recurrent_step_indexed(q[s], k[s], v[s], g[s], scale, pool, idx, o=o)
    torch.cuda.synchronize()
    pool.copy_(p["pool"])
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for s in range(w.steps):
        sala_gla.recurrent_step_indexed(q[s], k[s], v[s], g[s], scale, pool, idx, o=o)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(ev0.elapsed_time(ev1))
    # per-kernel events in a second pass of the same steps
    sala_gla.timing_enable(True)
    for s in range(w.steps):
        sala_gla.recurrent_step_indexed(q[s], k[s], v[s], g[s], scale, pool, idx, o=o)
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()["recurrent_step_indexed"]
    assert sala_gla.get_device_status() == 0
    # the same steps with the q/k prologue fused (RMSNorm + RoPE on the token's q and k;
    # positions 4096 + step)
    gen = torch.Generator().manual_seed(10)
    qw = (1 + 0.1 * torch.randn(D, generator=gen)).to(torch.bfloat16).to(dev)
    kw = (1 + 0.1 * torch.randn(D, generator=gen)).to(torch.bfloat16).to(dev)
    pos = [torch.full((w.nseq,), 4096 + s, dtype=torch.int64, device=dev) for s in range(w.steps)]
    pool.copy_(p["pool"])
    torch.cuda.synchronize()
    ev0.record(stream)
    for s in range(w.steps):
        sala_gla.recurrent_step_indexed(q[s], k[s], v[s], g[s], scale, pool, idx, o=o,
                                        prologue=(qw, kw, 1e-6, 10000.0), positions=pos[s])
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_pro = dist.max(ev0.elapsed_time(ev1))
    per_step = decode_pool_bytes(w.nseq, w.H, 2 if w.storage == "bf16" else 4)
    gbs = per_step * w.steps / (ms / 1e3) / 1e9 * dist.world
    k_ach = per_step / (kern[0] / kern[1] / 1e3) / 1e9
    return {
        "metric": "pooled decode HBM GB/s", "value": gbs, "unit": "GB/s",
        "ms_per_step": ms / w.steps, "tokens_per_s": w.nseq * w.steps / (ms / 1e3) * dist.world,
        "ms_per_step_with_qk_prologue": ms_pro / w.steps,
        "config": {"workload": w.name, "N": w.nseq, "H": w.H, "d": D, "steps": w.steps,
                   "pool_slots": w.pool, "state_storage": w.storage,
                   "pool_bytes": w.pool * w.H * D * D * (2 if w.storage == "bf16" else 4),
                   "bytes_per_step": per_step,
                   "tokens": "the decode workload's per-step q, k, v, g"},
        "roofline": {"kernel": "recurrent_step_indexed", "bound": "hbm", "achieved": k_ach,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": k_ach / peaks["hbm_gbs"],
                     "traffic": MEASURED_TRAFFIC["recurrent_step_indexed"]
                     if (w.nseq, w.H, w.pool, w.storage) == (256, 32, 512, "bf16") else None,
                     "peak_source": peaks["source"], "mean_launch_us": 1e3 * kern[0] / kern[1]},
        "_launches": kern[1],
    }


def run_gdn_prefill(args, dist, dev, peaks, sala_gla, inputs):
    """The gated delta rule over a batch of short sequences (64 x 256 tokens, 32 heads), in its
    recurrent form (sala_gla_gdn_fwd, the form the GDN/KDA page uses for short prefills) and in
    its chunked form (sala_gla_gdn_chunk_fwd, sub-object "chunked"). The recurrent kernel is
    bound by fp32 FMA throughput, not by memory: the recurrence's 4 d^2 = 65,536 multiply-adds
    per token and head (the kernel executes 3 d^2, keeping the decay as a scalar), against the
    CUDA cores' 152 SMs x 128 FMA per cycle at the 2.07 GHz clock. The chunked call is
    reported against the HBM roofline of its algorithmic bytes."""
    import torch
    lens = (256,) * 64
    H = 32
    x = inputs.make_prefill("varlen", seqlens=lens, H=H, seed=13)
    gen = torch.Generator().manual_seed(13)
    beta = torch.sigmoid(torch.randn(x["g"].shape, generator=gen))
    q, k, v, g, h0, cu = (x[n].to(dev) for n in ("q", "k", "v", "g", "h0", "cu_seqlens"))
    b = beta.to(dev)
    o = torch.empty_like(q)
    hT = torch.empty_like(h0)

    def call():
        sala_gla.gdn_fwd(q, k, v, g, b, x["scale"], h0=h0, cu_seqlens=cu, o=o, hT=hT)

    for _ in range(max(3, args.warmup)):
        call()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(3, min(args.steps, 10))
    dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        call()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(ev0.elapsed_time(ev1))
    sala_gla.timing_enable(True)
    for _ in range(steps):
        call()
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()["gdn_fwd"]
    T = sum(lens)
    flops = 2.0 * 4 * D * D * T * H
    peak_tflops = 152 * 128 * 2 * 2.07e9 / 1e12
    k_ach = flops / (kern[0] / kern[1] / 1e3) / 1e12
    # the chunked form (sala_gla_gdn_chunk_fwd): the new_v pass on the tensor cores, then the
    # chunked Simple GLA prefill; HBM-bound by its algorithmic bytes (q, k, v, g, beta read
    # once, o written once, h0 read and hT written once per (sequence, head))
    def call_chunked():
        sala_gla.gdn_fwd(q, k, v, g, b, x["scale"], h0=h0, cu_seqlens=cu, o=o, hT=hT, chunked=True)

    for _ in range(max(3, args.warmup)):
        call_chunked()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        call_chunked()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_c = dist.max(ev0.elapsed_time(ev1))
    sala_gla.timing_enable(True)
    for _ in range(steps):
        call_chunked()
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kc = sala_gla.timing_read()
    assert sala_gla.get_device_status() == 0
    nseq = len(lens)
    gdn_bytes = T * H * (4 * D * 2 + 2 * 4) + 2 * nseq * H * D * D * 4
    c_kernels = {n: {"us_per_launch": 1e3 * v[0] / v[1], "launches": v[1]} for n, v in kc.items() if v[1]}
    c_launch_us = sum(1e3 * v[0] / v[1] for v in kc.values() if v[1])
    c_ach = gdn_bytes / (ms_c / steps / 1e3) / 1e9
    chunked = {
        "metric": "gated-delta-rule chunked prefill tokens/s", "value": T * steps / (ms_c / 1e3) * dist.world,
        "unit": "tokens/s", "ms_per_call": ms_c / steps, "kernels": c_kernels,
        "speedup_vs_recurrent": (ms / steps) / (ms_c / steps),
        "roofline": {"kernel": "gdn_newv + seg_table + prefill_fused (whole call)", "bound": "hbm",
                     "achieved": c_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": c_ach / peaks["hbm_gbs"], "traffic": None,
                     "bytes_per_call": gdn_bytes, "peak_source": peaks["source"],
                     "mean_call_us_from_kernels": c_launch_us},
        "_launches": sum(v[1] for v in kc.values()),
    }
    return {
        "chunked": chunked,
        "metric": "gated-delta-rule recurrent prefill tokens/s", "value": T * steps / (ms / 1e3) * dist.world,
        "unit": "tokens/s", "ms_per_call": ms / steps,
        "config": {"workload": "gdn_prefill", "seqlens": "64 x 256", "T": T, "H": H, "d": D,
                   "inputs": "varlen recipe (q, k L2, g logsigmoid, h0 N(0, 0.02)), beta = sigmoid(N(0,1))"},
        "roofline": {"kernel": "gdn_fwd", "bound": "alu", "achieved": k_ach, "peak": peak_tflops,
                     "unit": "TFLOP/s", "frac": k_ach / peak_tflops, "traffic": MEASURED_TRAFFIC["gdn_fwd"],
                     "peak_source": "derived: 152 SMs x 128 fp32 FMA/cycle x 2 flop x 2.07 GHz",
                     "mean_launch_us": 1e3 * kern[0] / kern[1]},
        "_launches": kern[1],
    }


SIDE_LAUNCHES = 40


def call_percentiles(stream, call, n):
    """p10 / p50 / p90 of n single calls, CUDA events around each on the launching stream (a
    pass of its own: the events add host work between launches)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(evs):
        a.record(stream)
        call(i)
        b.record(stream)
    torch.cuda.synchronize()
    us = sorted(1e3 * a.elapsed_time(b) for a, b in evs)
    at = lambda q: us[int(round(q * (len(us) - 1)))]
    return {"calls": n, "p10_us": at(0.1), "p50_us": at(0.5), "p90_us": at(0.9)}


def side_loop_us(stream, call):
    """Mean duration of one launch of a single-kernel call, from CUDA events on the launching
    stream around SIDE_LAUNCHES back-to-back calls (nothing else runs in between; the inputs
    alternate between two sets larger than L2 together). Events around every launch would
    add their own record gap to each one, a few percent of a 35-50 us kernel."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(SIDE_LAUNCHES):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return 1e3 * e0.elapsed_time(e1) / SIDE_LAUNCHES


def run_qk_prologue(args, dist, dev, peaks, sala_gla, inputs, T, H):
    """sala_gla_qk_prologue in place on q and k [T, H, 128] (the prefill's shape), one sequence
    from position 0, two input sets alternated (each 2 x 67 MB at T = 8192, H = 32). Every call
    rewrites its inputs, which is what it is timed on (the values stay normalised)."""
    import torch
    sets = []
    for sd in (8, 9):
        x = inputs.make_qk_prologue(T, H, seed=sd)
        sets.append((x["q"].to(dev), x["k"].to(dev), x["q_weight"].to(dev), x["k_weight"].to(dev)))
    cu = torch.tensor([0, T], dtype=torch.int64, device=dev)

    def call(i):
        q, k, qw, kw = sets[i % 2]
        sala_gla.qk_prologue(q, k, qw, kw, 1e-6, 10000.0, cu_seqlens=cu)

    for i in range(max(3, args.warmup)):
        call(i)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        call(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(ev0.elapsed_time(ev1))
    us_loop = side_loop_us(stream, call)
    sala_gla.timing_enable(True)
    for i in range(args.steps):
        call(i)
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()["qk_prologue"]
    per_call = 2 * 2 * T * H * D * 2 + 2 * D * 2
    k_ach = per_call / (us_loop / 1e6) / 1e9
    return {
        "metric": "q/k prologue HBM GB/s", "value": per_call * args.steps / (ms / 1e3) / 1e9 * dist.world,
        "unit": "GB/s", "us_per_call": 1e3 * ms / args.steps,
        "tokens_per_s": T * args.steps / (ms / 1e3) * dist.world,
        "config": {"workload": "qk_prologue", "T": T, "H": H, "bytes_per_call": per_call,
                   "inputs": "raw q, k ~ 3 N(0,1) bf16, weights 1 + 0.1 N(0,1); theta 10000; in place"},
        "roofline": {"kernel": "qk_prologue", "bound": "hbm", "achieved": k_ach,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": k_ach / peaks["hbm_gbs"],
                     "traffic": MEASURED_TRAFFIC["qk_prologue"] if (T, H) == (8192, 32) else None,
                     "peak_source": peaks["source"],
                     "mean_launch_us": us_loop, "launches_timed": SIDE_LAUNCHES,
                     "mean_launch_us_bracketed": 1e3 * kern[0] / kern[1]},
        "_launches": kern[1],
    }


def run_output_gate(args, dist, dev, peaks, sala_gla, inputs, T, H):
    """sala_gla_output_norm_gate on [T, H * 128] (the prefill's output shape), two input sets
    alternated (each 3 x 67 MB at T = 8192, H = 32: larger than L2 together)."""
    import torch
    sets = []
    for sd in (6, 7):
        x = inputs.make_output_gate(T, H, seed=sd)
        sets.append((x["o"].to(dev), x["z"].to(dev), x["w"].to(dev), torch.empty_like(x["o"], device=dev)))
    eps = 1e-6
    for i in range(max(3, args.warmup)):
        o, z, wt, out = sets[i % 2]
        sala_gla.output_norm_gate(o, z, wt, eps, out=out)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        o, z, wt, out = sets[i % 2]
        sala_gla.output_norm_gate(o, z, wt, eps, out=out)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(ev0.elapsed_time(ev1))

    def call(i):
        o, z, wt, out = sets[i % 2]
        sala_gla.output_norm_gate(o, z, wt, eps, out=out)

    us_loop = side_loop_us(stream, call)
    sala_gla.timing_enable(True)
    for i in range(args.steps):
        call(i)
    torch.cuda.synchronize()
    sala_gla.timing_enable(False)
    kern = sala_gla.timing_read()["output_norm_gate"]
    F = H * D
    per_call = 3 * T * F * 2 + F * 2
    k_ach = per_call / (us_loop / 1e6) / 1e9
    return {
        "metric": "output norm+gate HBM GB/s", "value": per_call * args.steps / (ms / 1e3) / 1e9 * dist.world,
        "unit": "GB/s", "us_per_call": 1e3 * ms / args.steps,
        "tokens_per_s": T * args.steps / (ms / 1e3) * dist.world,
        "config": {"workload": "output_gate", "T": T, "H": H, "features": F, "bytes_per_call": per_call,
                   "inputs": "o ~ N(0,1), z ~ N(0,4) bf16, w = 1 + 0.1 N(0,1) bf16; two sets alternated"},
        "roofline": {"kernel": "output_norm_gate", "bound": "hbm", "achieved": k_ach,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": k_ach / peaks["hbm_gbs"],
                     "traffic": MEASURED_TRAFFIC["output_norm_gate"] if (T, H) == (8192, 32) else None,
                     "peak_source": peaks["source"],
                     "mean_launch_us": us_loop, "launches_timed": SIDE_LAUNCHES,
                     "mean_launch_us_bracketed": 1e3 * kern[0] / kern[1]},
        "_launches": kern[1],
    }


def main():
    args = parse_args()
    dist = Dist()
    if args.impl == "reference":
        if dist.rank != 0:
            return
        run_reference(args, dist)
        return
    run_ours(args, dist)


if __name__ == "__main__":
    main()
