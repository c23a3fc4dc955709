#!/usr/bin/env python3
"""KDA benchmark on GB300: prefill tokens/s and decode state GB/s.

Default workload (one "step" = one pass of the whole hot path):
  kda_prefill on B=1, H=32, T=4096, d_k=d_v=128 (bf16 q/k/v/z/beta, fp32 A,
  zero initial state) returning the fp32 final state, then one kda_decode_step
  for each of the 32 heads from that final state (the decode handoff).
The headline `value` is prefill tokens/s (B*T / step time).  The `decode`
object times the decode workload B=256, H=96, d=128 (fp32 state ~1.6 GB resident
in HBM, bf16 per-step inputs) over 64 consecutive steps, as state GB/s.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kda|reference]
Under torchrun each rank runs an independent replica (the path needs no
collective); rank 0 prints one JSON line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (% tensor peak); decode state GB/s (% HBM peak), 1 GB300"
PREFILL_SHAPE = dict(B=1, H=32, T=4096, d=128)
DECODE_SHAPE = dict(B=256, H=96, d=128, steps=64)
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured (MEASURED_PEAKS.json)")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


def prefill_algorithmic(B, H, T, d, C=64):
    """Algorithmic bytes and flops of one prefill call (d_k = d_v = d, bf16 I/O).

    bytes: q, k, v, z, o at 2 B per element, beta at 2 B per head-token, the fp32
    final state once (zero initial state is not read).
    flops: 6 d^2 per head-token for the three state contractions plus
    (C+1)(3d+2d) - d for the causal halves of the intra-chunk products."""
    ht = B * T * H
    byts = ht * (5 * d * 2 + 2) + B * H * d * d * 4
    flops = ht * (6 * d * d + (C + 1) * 5 * d - d)
    return byts, flops


# Sources of the chunked prefill kernels; a profile summary records their
# digest so that its DRAM traffic is only reported for the kernel it measured.
PREFILL_SOURCES = ("kda_prefill_sm103.cu", "kda_chunk_phases.cuh", "sm103_ptx.cuh",
                   "kda_chunked.h")


def prefill_source_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in PREFILL_SOURCES:
        with open(os.path.join(ROOT, "kimi_delta_attention_12_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """dram bytes read + written per launch of `kernel` from its committed ncu
    summary, or None when there is none for the current sources."""
    prof = os.path.join(ROOT, "profiles", f"{kernel}_b1_h32_t4096.md")
    if not os.path.exists(prof):
        return None
    rows = {}
    for line in open(prof):
        cells = [c.strip() for c in line.split("|")]
        if len(cells) >= 4 and cells[0] == "":
            rows[cells[1]] = cells[2]
    if rows.get("source_digest") != prefill_source_digest():
        return None
    try:
        return int(rows["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def decode_algorithmic(B, H, d):
    """Bytes of one decode step: fp32 state read + write, bf16 q,k,v,z in, o out, beta."""
    return B * H * (2 * d * d * 4 + 5 * d * 2 + 2)


def conv_algorithmic(N, H, T, d, W):
    """Bytes of one kda_short_conv call (d_k = d_v = d, bf16): q, k, v read and
    their convolved copies written, conv states read and written, fp32 taps."""
    Cc = 3 * d
    return 2 * N * T * H * Cc * 2 + 2 * N * H * (W - 1) * Cc * 2 + H * Cc * W * 4


def conv_decode_extra(B, H, d, W):
    """Bytes a decode step with short convolutions moves on top of
    decode_algorithmic: the bf16 conv state read and written, the fp32 taps
    (the convolved token passes through a scratch buffer, not counted)."""
    Cc = 3 * d
    return 2 * B * H * (W - 1) * Cc * 2 + H * Cc * W * 4


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def _barrier(pg):
    if pg is not None:
        pg.barrier()


def _max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle arm
def run_oracle_sample(T_sample: int, H: int, d: int, seed: int = 0):
    """Time the fp64 CPU oracle on the first T_sample tokens of the prefill
    workload (all heads).  Returns (tokens/s, seconds, threads)."""
    import torch
    import oracle
    from kimi_delta_attention_12_gb300 import inputs
    x = inputs.make_prefill_inputs([T_sample], H, d, d, torch.bfloat16, seed=seed)
    oracle.build()
    t0 = time.perf_counter()
    _, _, threads = oracle.kda_reference(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens)
    dt = time.perf_counter() - t0
    return T_sample / dt, dt, threads


def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo, else the platform)."""
    import platform
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
        with open("/proc/cpuinfo") as fh:   # Arm: implementer / part numbers
            fields = {}
            for line in fh:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
            if "CPU part" in fields:
                return (f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} "
                        f"part {fields['CPU part']}")
    except OSError:
        pass
    return platform.machine() or "unknown"


def cpu_baseline(H: int, T: int, d: int, cpu_seconds: float = 12.0):
    """The oracle on the whole prefill workload, repeated until about
    cpu_seconds of CPU work (wall time x threads) are spent."""
    runs, wall, threads = 0, 0.0, 1
    while runs == 0 or wall * threads < cpu_seconds:
        _, dt, threads = run_oracle_sample(T, H, d)
        runs += 1
        wall += dt
    value = runs * T / wall
    sample = (f"whole prefill workload (B=1 T={T}, all {H} heads) x {runs} runs, "
              f"{wall:.1f} s wall on {threads} threads, fp64 C oracle")
    return value, threads, sample


def row_cpu_baselines(H: int, T: int, d: int, dec_B: int, dec_H: int):
    """The oracle timed on each further row's workload (or a stated sample of
    it), beside the GPU figure of that row.  Returns {row: cpu_baseline}."""
    import numpy as np
    import torch
    import oracle
    from kimi_delta_attention_12_gb300 import inputs
    oracle.build()
    x = inputs.make_prefill_inputs([T], H, d, d, torch.bfloat16, seed=0)
    rows = {}

    t0 = time.perf_counter()
    _, _, threads = oracle.kda_reference(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens,
                                         softplus_gate=True)
    dt = time.perf_counter() - t0
    rows["softplus_gate"] = {
        "value": T / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
        "sample": f"whole softplus-gate prefill (B=1 T={T}, all {H} heads), fp64 C oracle, "
                  f"{dt:.2f} s"}

    w, cs0 = inputs.make_conv_params(1, H, d, d, CONV_WIDTH, torch.bfloat16, seed=11)
    t0 = time.perf_counter()
    oracle.short_conv_qkv(x.q, x.k, x.v, w, x.cu_seqlens, cs0, True)
    dt = time.perf_counter() - t0
    byts = conv_algorithmic(1, H, T, d, CONV_WIDTH)
    rows["short_conv"] = {
        "value": byts / dt / 1e9, "unit": "GB/s", "ms": dt * 1e3, "cores": 1, "kind": "oracle",
        "sample": f"whole conv workload (T={T}, {H} heads, width {CONV_WIDTH}, SiLU, states in "
                  f"and out; inputs converted to fp64 inside the timed call), fp64 C oracle"}

    Tb = min(T, 1024)
    xb = inputs.make_prefill_inputs([Tb], H, d, d, torch.bfloat16, seed=0)
    dO, dSf = inputs.make_upstream_grads(Tb, 1, H, d, d, torch.bfloat16, seed=21)
    t0 = time.perf_counter()
    g = oracle.kda_reference_backward(xb.q, xb.k, xb.v, xb.z, xb.beta, xb.A, None,
                                      xb.cu_seqlens, dO, dSf)
    dt = time.perf_counter() - t0
    rows["backward"] = {
        "value": Tb / dt, "unit": "tokens/s", "cores": g["threads"], "kind": "oracle",
        "sample": f"backward on the first {Tb} tokens of the workload (all {H} heads), "
                  f"fp64 C oracle, {dt:.2f} s"}

    Bs = 16
    A, S0 = inputs.make_decode_state(Bs, dec_H, d, d, seed=5)
    st = inputs.make_decode_step(Bs, dec_H, d, d, torch.bfloat16, seed=5, step=0)
    cu = np.arange(Bs + 1, dtype=np.int64)
    t0 = time.perf_counter()
    _, _, threads = oracle.kda_reference(st.q, st.k, st.v, st.z, st.beta, A, S0, cu)
    dt = time.perf_counter() - t0
    rows["decode"] = {
        "value": decode_algorithmic(Bs, dec_H, d) / dt / 1e9, "unit": "GB/s",
        "ms_per_step": dt * 1e3 * dec_B / Bs, "cores": threads, "kind": "oracle",
        "sample": f"one decode step of {Bs} of the {dec_B} sequences ({dec_H} heads; state "
                  f"converted to fp64 inside the timed call), fp64 C oracle; ms_per_step "
                  f"scaled to the full batch"}
    return rows


def reference_arm(args, world, rank, pg):
    if rank != 0:
        return
    P = PREFILL_SHAPE
    T_sample = P["T"]
    # one warm-up and K timed steps; each step is the whole prefill workload
    # (B=1, T=4096, all 32 heads)
    for _ in range(max(0, min(args.warmup, 1))):
        run_oracle_sample(256, P["H"], P["d"])
    vals, secs, threads = [], 0.0, 1
    for _ in range(args.steps):
        v, dt, threads = run_oracle_sample(T_sample, P["H"], P["d"])
        vals.append(v)
        secs += dt
    value = statistics.median(vals)
    sample = (f"whole workload B=1 T={T_sample} d=128, all 32 heads, per step; "
              f"{args.steps} steps, fp64 C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded torch CPU generator)",
        "config": {"workload": "prefill B=1 H=32 T=4096 d_k=d_v=128 bf16 inputs", "B": 1,
                   "H": 32, "T": 4096, "d": 128},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU arm
def kda_arm(args, world, rank, local, pg):
    import torch
    import kimi_delta_attention_12_gb300 as kda
    from kimi_delta_attention_12_gb300 import inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.lib()
    stream = torch.cuda.current_stream()
    peaks = _peaks()
    if args.only == "decode":
        return decode_only(args, rank, local, dev, stream, peaks)
    P = PREFILL_SHAPE
    B, H, T, d = P["B"], P["H"], P["T"], P["d"]
    byts, flops = prefill_algorithmic(B, H, T, d)

    # rotating input sets so that each step's inputs are not L2-resident
    x_host = inputs.make_prefill_inputs([T] * B, H, d, d, torch.bfloat16, seed=rank)
    set_bytes = byts
    nsets = max(2, -(-3 * L2_BYTES // set_bytes))
    sets = []
    for i in range(nsets):
        xi = x_host.to(dev) if i == 0 else inputs.PrefillInputs(
            *(t.clone() if t is not None else None for t in
              (sets[0].q, sets[0].k, sets[0].v, sets[0].z, sets[0].beta, sets[0].A,
               sets[0].initial_state, sets[0].cu_seqlens)))
        sets.append(xi)
    o = torch.empty(B * T, H, d, dtype=torch.bfloat16, device=dev)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=dev)
    ws = kda.alloc_workspace(B, B * T, H, d, d, torch.bfloat16, dev)
    # the library asks for more than the minimal workspace (256 B header + one
    # int32 per sequence-head, rounded to 256 B) exactly when it runs the split kernel
    minimal_ws = 256 + -(-4 * B * H // 256) * 256
    kernel_name = "kda_split_kernel" if ws.numel() > minimal_ws else "kda_chunked_kernel"
    o_dec = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    cu_host = sets[0].cu_seqlens.cpu()

    def step(i, ev=None):
        x = sets[i % nsets]
        if ev is not None:
            ev[0].record(stream)
        kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens,
                        cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        # decode handoff: the next token of each head continues from S
        kda.kda_decode_step(x.q[:B], x.k[:B], x.v[:B], x.z[:B], x.beta[:B], x.A, S, o=o_dec)

    launches_per_step = 2
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert kda.workspace_status(ws) == kda.KDA_OK, "prefill kernel reported a timeout"

    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    _barrier(pg)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i, kev[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    _barrier(pg)
    ms_total = t_start.elapsed_time(t_end)
    ms_total = _max_over_ranks(pg, ms_total)
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    ms_per_step = ms_total / args.steps
    value = world * B * T / (ms_per_step / 1e3)
    achieved_gbs = byts / (kernel_ms / 1e3) / 1e9
    achieved_tf = flops / (kernel_ms / 1e3) / 1e12
    if args.only == "softplus":
        sp = measure_softplus(sets, ws, o, S, cu_host, args, stream)
        if rank == 0:
            print(json.dumps(dict(sp, only="softplus",
                                  tokens_per_s=B * T / (sp["kernel_ms"] / 1e3))), flush=True)
        return
    if args.only == "backward":
        bw = measure_backward(sets, B, H, T, d, args, stream)
        if rank == 0:
            print(json.dumps(dict(bw, only="backward",
                                  frac=bw["achieved_gbs"] / peaks["hbm_gbs"])), flush=True)
        return
    if args.only == "conv":
        conv = measure_conv(sets, ws, o, S, cu_host, B, H, T, d, args, stream)
        if rank == 0:
            print(json.dumps(dict(conv, only="conv",
                                  frac=conv["achieved_gbs"] / peaks["hbm_gbs"])), flush=True)
        return
    if args.only == "prefill":
        if rank == 0:
            print(json.dumps({"only": "prefill", "value": value, "unit": "tokens/s",
                              "kernel_ms": kernel_ms, "achieved_gbs": achieved_gbs,
                              "tensor_tflops": achieved_tf}), flush=True)
        return
    ckpt = measure_checkpointed(sets, ws, o, S, cu_host, B, H, T, d, args, stream)
    softplus = measure_softplus(sets, ws, o, S, cu_host, args, stream)
    softplus["tokens_per_s"] = B * T / (softplus["kernel_ms"] / 1e3)
    extras = {"prefill_checkpointed": dict(ckpt, kernel_ms_plain=kernel_ms),
              "softplus_gate": softplus,
              "short_conv": measure_conv(sets, ws, o, S, cu_host, B, H, T, d, args, stream),
              "backward": measure_backward(sets, B, H, T, d, args, stream)}

    return finish(args, world, rank, local, dev, stream, peaks, B, H, T, d, byts, flops, nsets,
                  set_bytes, x_host, o, S, ws, cu_host, value, ms_per_step, kernel_ms,
                  achieved_gbs, achieved_tf, clk, launches_per_step, kernel_name, pg, extras)


def measure_checkpointed(sets, ws, o, S, cu_host, B, H, T, d, args, stream, interval=1024):
    """The same prefill with a state checkpoint every `interval` tokens
    (kda_prefill_checkpointed): kernel time and the checkpoint bytes written."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    count = kda.checkpoint_count(cu_host, B, B * T, interval)
    pool = torch.empty(count, H, d, d, dtype=torch.float32, device=o.device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        x = sets[i % len(sets)]
        if i >= args.warmup:
            ev[i - args.warmup][0].record(stream)
        kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens,
                        cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws,
                        ckpt_interval=interval, ckpt_pool=pool)
        if i >= args.warmup:
            ev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return {"interval": interval, "checkpoints": count,
            "checkpoint_bytes": count * H * d * d * 4, "kernel_ms": ms}


CONV_WIDTH = 4


def backward_algorithmic(B, H, T, d):
    """Bytes of one kda_backward call (d_k = d_v = d, bf16 inputs): q, k, v, z,
    dO and beta read; fp32 dq, dk, dv, dz, dbeta, dS0 and dA written."""
    ht = B * T * H
    return ht * (5 * d * 2 + 2) + ht * (4 * d * 4 + 4) + B * H * d * d * 4 + H * 4


def measure_backward(sets, B, H, T, d, args, stream):
    """kda_backward on the prefill workload with seeded upstream gradients:
    the call's time (its checkpointed forward prefill, the backward and the
    finalize kernels) and bandwidth on its algorithmic bytes."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    from kimi_delta_attention_12_gb300 import inputs
    x0 = sets[0]
    dO, dSf = inputs.make_upstream_grads(B * T, B, H, d, d, torch.bfloat16, seed=21)
    dO, dSf = dO.to(x0.q.device), dSf.to(x0.q.device)
    ws = torch.empty(kda.backward_workspace_bytes(B, B * T, H, d, d, torch.bfloat16),
                     dtype=torch.uint8, device=x0.q.device)
    n = min(args.steps, 3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for i in range(1 + n):
        x = sets[i % len(sets)]
        if i >= 1:
            ev[i - 1][0].record(stream)
        kda.kda_backward(x.q, x.k, x.v, x.z, x.beta, x.A, dO, None, x.cu_seqlens,
                         dS_final=dSf, workspace=ws)
        if i >= 1:
            ev[i - 1][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    byts = backward_algorithmic(B, H, T, d)
    return {"kernel": "kda_backward_kernel", "form": "recurrent, fp32", "kernel_ms": ms,
            "steps": n, "tokens_per_s": B * T / (ms / 1e3), "algorithmic_bytes": byts,
            "achieved_gbs": byts / (ms / 1e3) / 1e9}


def measure_conv(sets, ws, o, S, cu_host, B, H, T, d, args, stream):
    """The short convolutions (width 4, SiLU, conv states in and out) on the
    prefill workload: kda_short_conv kernel time and bandwidth, and the time
    of kda_short_conv followed by kda_prefill on its outputs."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    from kimi_delta_attention_12_gb300 import inputs
    dev = o.device
    W = CONV_WIDTH
    w, cs0 = inputs.make_conv_params(B, H, d, d, W, torch.bfloat16, seed=11)
    w, cs_in = w.to(dev), cs0.to(dev)
    cs_out = torch.empty_like(cs_in)
    outs = tuple(torch.empty(B * T, H, d, dtype=torch.bfloat16, device=dev) for _ in range(3))
    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(args.warmup + n):
        x = sets[i % len(sets)]
        e = ev[i - args.warmup] if i >= args.warmup else None
        if e:
            e[0].record(stream)
        qc, kc, vc = kda.kda_short_conv(x.q, x.k, x.v, w, cs_in, cs_out, x.cu_seqlens, cu_host,
                                        silu=True, outputs=outs)
        if e:
            e[1].record(stream)
        kda.kda_prefill(qc, kc, vc, x.z, x.beta, x.A, None, x.cu_seqlens,
                        cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws)
        if e:
            e[2].record(stream)
    torch.cuda.synchronize()
    conv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    both_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    byts = conv_algorithmic(B, H, T, d, W)
    return {"kernel": "short_conv_kernel", "width": W, "silu": True, "kernel_ms": conv_ms,
            "algorithmic_bytes": byts, "achieved_gbs": byts / (conv_ms / 1e3) / 1e9,
            "conv_then_prefill_ms": both_ms,
            "conv_then_prefill_tokens_per_s": B * T / (both_ms / 1e3)}


def measure_softplus(sets, ws, o, S, cu_host, args, stream):
    """The same prefill with the softplus-decay gate (KDA_FLAG_SOFTPLUS_GATE), which
    runs on the fp32 recurrent kernel: its kernel time."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    n = min(args.steps, 5)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for i in range(args.warmup + n):
        x = sets[i % len(sets)]
        if i >= args.warmup:
            ev[i - args.warmup][0].record(stream)
        kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens,
                        cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws,
                        softplus_gate=True)
        if i >= args.warmup:
            ev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    return {"kernel": "kda_recurrent_kernel",
            "kernel_ms": statistics.mean(a.elapsed_time(b) for a, b in ev), "steps": n}


def run_decode(dev, rank, local, stream, batch=None, softplus_gate=False, conv=False):
    """64 consecutive decode steps on a resident B=256, H=96, d=128 fp32 state
    (with conv: each step preceded by the token's short convolutions, width 4
    and SiLU, on a resident bf16 conv state: kda_decode_step_conv)."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    D = DECODE_SHAPE
    g = torch.Generator(device=dev).manual_seed(1000 + rank)
    Bd, Hd, dd = batch or D["B"], D["H"], D["d"]
    state = 0.02 * torch.randn(Bd, Hd, dd, dd, device=dev, generator=g)
    Adec = 0.5 * torch.randn(Hd, device=dev, generator=g)
    unit = lambda t: t / t.norm(dim=-1, keepdim=True)
    dsteps = []
    for s in range(D["steps"]):
        dsteps.append((unit(torch.randn(Bd, Hd, dd, device=dev, generator=g)).bfloat16(),
                       unit(torch.randn(Bd, Hd, dd, device=dev, generator=g)).bfloat16(),
                       torch.randn(Bd, Hd, dd, device=dev, generator=g).bfloat16(),
                       torch.randn(Bd, Hd, dd, device=dev, generator=g).bfloat16(),
                       torch.sigmoid(torch.randn(Bd, Hd, device=dev, generator=g)).bfloat16()))
    od = torch.empty(Bd, Hd, dd, dtype=torch.bfloat16, device=dev)
    if conv:
        from kimi_delta_attention_12_gb300 import inputs
        cw, cst = inputs.make_conv_params(Bd, Hd, dd, dd, CONV_WIDTH, torch.bfloat16,
                                          seed=1000 + rank)
        cw, cst = cw.to(dev), cst.to(dev)
        cws = torch.empty(kda.decode_conv_workspace_bytes(Bd, Hd, dd, dd, torch.bfloat16),
                          dtype=torch.uint8, device=dev)

    def one(s):
        q_, k_, v_, z_, b_ = dsteps[s]
        if conv:
            kda.kda_decode_step_conv(q_, k_, v_, z_, b_, Adec, state, cw, cst, o=od, silu=True,
                                     softplus_gate=softplus_gate, workspace=cws)
        else:
            kda.kda_decode_step(q_, k_, v_, z_, b_, Adec, state, o=od,
                                softplus_gate=softplus_gate)
    for s in range(3):
        one(s)
    torch.cuda.synchronize()
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(D["steps"])]
    with ClockSampler(local) as dclk:
        for s in range(D["steps"]):
            dev_ev[s][0].record(stream)
            one(s)
            dev_ev[s][1].record(stream)
        torch.cuda.synchronize()
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
    dec_bytes = decode_algorithmic(Bd, Hd, dd)
    if conv:
        dec_bytes += conv_decode_extra(Bd, Hd, dd, CONV_WIDTH)
    return dec_ms, dec_bytes, dec_bytes / (dec_ms / 1e3) / 1e9, dclk.summary()


def decode_only(args, rank, local, dev, stream, peaks):
    dec_ms, dec_bytes, dec_gbs, clk = run_decode(dev, rank, local, stream, args.decode_batch,
                                                 conv=args.decode_conv)
    if rank == 0:
        print(json.dumps({"only": "decode", "batch": args.decode_batch,
                          "conv": args.decode_conv, "value": dec_gbs,
                          "unit": "GB/s", "ms_per_step": dec_ms,
                          "frac": dec_gbs / peaks["hbm_gbs"], "clocks": clk}), flush=True)


def finish(args, world, rank, local, dev, stream, peaks, B, H, T, d, byts, flops, nsets,
           set_bytes, x_host, o, S, ws, cu_host, value, ms_per_step, kernel_ms, achieved_gbs,
           achieved_tf, clk, launches_per_step, kernel_name, pg, extras):
    import torch
    import kimi_delta_attention_12_gb300 as kda
    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs from pinned host memory, runs kda_prefill
    # and reads o and the final state back into pinned host memory.  Steps are
    # pipelined the way a stream of requests would be: copy-in, prefill and
    # copy-out run on three streams with two device buffer sets, so that the
    # copy-in of step i + 1 overlaps the prefill of step i and the copy-out of
    # step i - 1 (host-to-device copies run at ~210 GB/s and bound the step).
    pin = lambda t: t.pin_memory()
    hq, hk, hv, hz, hb = (pin(t) for t in (x_host.q, x_host.k, x_host.v, x_host.z, x_host.beta))
    hA, hcu = pin(x_host.A), pin(x_host.cu_seqlens)
    ho = torch.empty(B * T, H, d, dtype=torch.bfloat16).pin_memory()
    hS = torch.empty(B, H, d, d, dtype=torch.float32).pin_memory()
    hosts = (hq, hk, hv, hz, hb, hA, hcu)
    dbufs = [tuple(torch.empty_like(t, device=dev) for t in hosts) for _ in range(2)]
    douts = [(o, S), (torch.empty_like(o), torch.empty_like(S))]
    h2d = sum(t.numel() * t.element_size() for t in hosts)
    d2h = ho.numel() * ho.element_size() + hS.numel() * hS.element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        dq, dk_, dv_, dz, db, dA, dcu = dbufs[b]
        ob, Sb = douts[b]
        s_in.wait_event(ev_cmp[b])      # buffer set b's last prefill has read its inputs
        with torch.cuda.stream(s_in):
            for dst, src in zip(dbufs[b], hosts):
                dst.copy_(src, non_blocking=True)
        ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        s_cmp.wait_event(ev_out[b])     # and its last outputs have been read out
        kda.kda_prefill(dq, dk_, dv_, dz, db, dA, None, dcu, cu_seqlens_host=cu_host,
                        o=ob, final_state=Sb, workspace=ws, stream=s_cmp)
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            ho.copy_(ob, non_blocking=True)
            hS.copy_(Sb, non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    _barrier(pg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    s_out.wait_event(ev_cmp[(args.steps - 1) % 2])
    e1.record(s_out)
    torch.cuda.synchronize()
    _barrier(pg)
    e2e_ms = _max_over_ranks(pg, e0.elapsed_time(e1)) / args.steps
    e2e_value = world * B * T / (e2e_ms / 1e3)

    # ---- decode workload: 64 consecutive steps on a resident 1.6 GB state ----
    D = DECODE_SHAPE
    dec_ms, dec_bytes, dec_gbs, dclk_summary = run_decode(dev, rank, local, stream)
    sp_ms, _, sp_gbs, _ = run_decode(dev, rank, local, stream, softplus_gate=True)
    extras["softplus_gate"].update({"decode_ms_per_step": sp_ms, "decode_gbs": sp_gbs,
                                    "decode_frac": sp_gbs / peaks["hbm_gbs"]})
    cv_ms, cv_bytes, cv_gbs, _ = run_decode(dev, rank, local, stream, conv=True)
    conv = extras["short_conv"]
    conv["frac"] = conv["achieved_gbs"] / peaks["hbm_gbs"]
    extras["backward"]["frac"] = extras["backward"]["achieved_gbs"] / peaks["hbm_gbs"]
    conv.update({"decode_kernels": "short_conv_decode_kernel + kda_recurrent_kernel",
                 "decode_ms_per_step": cv_ms, "decode_bytes_per_step": cv_bytes,
                 "decode_gbs": cv_gbs, "decode_frac": cv_gbs / peaks["hbm_gbs"]})

    if rank != 0:
        return
    # CPU baseline: the oracle on the same workload
    cpu_tps, cpu_threads, cpu_sample = cpu_baseline(H, T, d)
    row_cpu = row_cpu_baselines(H, T, d, D["B"], D["H"])
    for key in ("softplus_gate", "short_conv", "backward"):
        if key in extras:
            extras[key]["cpu_baseline"] = row_cpu[key]
    traffic = profiled_traffic(kernel_name)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generators; inputs rotated over "
                f"{nsets} sets of {set_bytes / 1e6:.0f} MB > L2)",
        "config": {"workload": "prefill B=1 H=32 T=4096 d_k=d_v=128 bf16 + decode handoff",
                   "B": B, "H": H, "T": T, "d": d, "chunk": 64,
                   "l2": "inputs larger than L2 (rotating sets)", "parallelism": "replicas"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                     "traffic": traffic, "kernel": kernel_name, "kernel_ms": kernel_ms,
                     "algorithmic_bytes": byts, "peak_source": peaks["source"],
                     "tensor_tflops": achieved_tf,
                     "tensor_frac": achieved_tf / peaks["bf16_tflops"]},
        "decode": {"metric": "decode state GB/s", "value": dec_gbs, "unit": "GB/s",
                   "ms_per_step": dec_ms, "bytes_per_step": dec_bytes,
                   "config": {"workload": "decode B=256 H=96 d=128 fp32 state, bf16 inputs",
                              "steps": D["steps"]},
                   "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"]},
                   "clocks": dclk_summary, "cpu_baseline": row_cpu["decode"]},
        **extras,
        "cpu_baseline": {"value": cpu_tps, "unit": "tokens/s", "cores": cpu_threads,
                         "kind": "oracle", "sample": cpu_sample, "cpu_model": cpu_model()},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelining": "copy-in, prefill and copy-out of consecutive steps overlap "
                              "(three streams, two device buffer sets)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "conv", "backward", "softplus"],
                    default="all",
                    help="run one part only (for profiler captures); the default runs all")
    ap.add_argument("--decode-batch", type=int, default=DECODE_SHAPE["B"],
                    help="decode batch for --only decode (smaller cases for profiler captures)")
    ap.add_argument("--decode-conv", action="store_true",
                    help="--only decode: each step preceded by the short convolutions")
    args = ap.parse_args()
    world, rank, local, pg = _dist_setup(args)
    try:
        if args.impl == "reference":
            reference_arm(args, world, rank, pg)
        else:
            kda_arm(args, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    main()
