#!/usr/bin/env python3
"""KDA benchmark on GB300: prefill tokens/s and decode state GB/s.

Default workload (one "step" = one pass of the whole hot path):
  kda_prefill on the long-prefill workload B=1, H=96, T=65,536, d_k=d_v=128
  (bf16 q/k/v/z/beta, fp32 A, zero initial state) returning the fp32 final
  state, then one kda_decode_step for each of the 96 heads from that final
  state (the decode handoff).  This is the largest single-GPU prefill
  configuration; the headline `value` is its prefill tokens/s (B*T / step
  time).  Further keys: the 4K prefill (B=1, H=32, T=4096) and the varlen
  workload (16 packed sequences, H=64, nonzero initial states), each with its
  roofline; the further rows (checkpoints, softplus gate, short
  convolutions, backward) on the 4K workload; and the decode workload
  B=256, H=96, d=128 (fp32 state ~1.6 GB resident in HBM) over 64
  consecutive steps, as state GB/s.

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
# the headline: the long prefill with its decode handoff (largest single-GPU config)
PREFILL_SHAPE = dict(B=1, H=96, T=65536, d=128)
PREFILL_4K_SHAPE = dict(B=1, H=32, T=4096, d=128)
# heads of the headline workload the oracle runs for the CPU baseline (the
# figure is extrapolated to all heads; heads are independent)
ORACLE_SAMPLE_HEADS = 16
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


def prefill_algorithmic(B, H, T, d, C=64, read_state=False, N=None):
    """Algorithmic bytes and flops of one prefill call over B*T packed tokens
    in N sequences (default B; d_k = d_v = d, bf16 I/O).

    bytes: q, k, v, z, o at 2 B per element, beta at 2 B per head-token, the
    fp32 final state once per (sequence, head), and the initial state once
    more when it is read (a zero initial state is not).
    flops: 6 d^2 per head-token for the three state contractions plus
    (C+1)(3d+2d) - d for the causal halves of the intra-chunk products."""
    N = B if N is None else N
    ht = B * T * H
    byts = ht * (5 * d * 2 + 2) + (2 if read_state else 1) * N * H * d * d * 4
    flops = ht * (6 * d * d + (C + 1) * 5 * d - d)
    return byts, flops


# Sources of the chunked prefill kernels; a profile summary records their
# digest so that its DRAM traffic is only reported for the kernel it measured.
PREFILL_SOURCES = ("kda_prefill_sm103.cu", "kda_chunk_phases.cuh", "kda_split_phases.cuh",
                   "sm103_ptx.cuh", "kda_chunked.h", "kda_seqlens.cuh")


def prefill_source_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in PREFILL_SOURCES:
        with open(os.path.join(ROOT, "kimi_delta_attention_12_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile: str, units: int):
    """DRAM bytes read + written per launch from the committed ncu summary
    profiles/<profile>.md, scaled from the profiled launch's (token, head)
    units to `units` (the kernel's traffic grows in proportion to them), or
    None when there is no summary for the current sources."""
    prof = os.path.join(ROOT, "profiles", f"{profile}.md")
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
        per = int(rows["traffic_bytes_per_launch"])
        prof_units = int(rows.get("head_token_units", "0")) or units
    except (KeyError, ValueError):
        return None
    return per * units / prof_units


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
    """Time the fp64 CPU oracle on one sequence of T_sample tokens and H heads
    (the prefill recipe's inputs).  Returns (head-tokens/s, seconds, threads)."""
    import torch
    import oracle
    from kimi_delta_attention_12_gb300 import inputs
    x = inputs.make_prefill_inputs([T_sample], H, d, d, torch.bfloat16, seed=seed)
    oracle.build()
    t0 = time.perf_counter()
    _, _, threads = oracle.kda_reference(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens)
    dt = time.perf_counter() - t0
    return T_sample * H / dt, dt, threads


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
    """The oracle on the whole prefill workload (B=1, T tokens, H heads),
    repeated until about cpu_seconds of CPU work (wall time x threads) are
    spent.  Returns (tokens/s, threads, sample)."""
    runs, wall, threads = 0, 0.0, 1
    while runs == 0 or wall * threads < cpu_seconds:
        _, dt, threads = run_oracle_sample(T, H, d)
        runs += 1
        wall += dt
    value = runs * T / wall
    sample = (f"whole prefill workload (B=1 T={T}, all {H} heads) x {runs} runs, "
              f"{wall:.1f} s wall on {threads} threads, fp64 C oracle")
    return value, threads, sample


def headline_cpu_baseline(H: int, T: int, d: int, H_sample: int = ORACLE_SAMPLE_HEADS):
    """The oracle on H_sample of the H heads of the long-prefill workload, all
    T tokens (heads are independent, so the whole workload takes H / H_sample
    times as long): tokens/s of the whole workload, extrapolated.  Returns
    (tokens/s, threads, sample)."""
    hts, dt, threads = run_oracle_sample(T, H_sample, d)
    value = T / (dt * H / H_sample)
    sample = (f"{H_sample} of the {H} heads of the workload, all {T} tokens (B=1), "
              f"{dt:.1f} s wall on {threads} threads, fp64 C oracle; tokens/s extrapolated "
              f"to all {H} heads")
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
    """The oracle arm: each step runs the fp64 oracle on a bounded sample of
    the headline workload (ORACLE_SAMPLE_HEADS of its heads, its first
    T_sample tokens) and reports the whole workload's tokens/s extrapolated
    from it (heads are independent, and the oracle's cost per token does not
    depend on the position)."""
    if rank != 0:
        return
    P = PREFILL_SHAPE
    Hs, T_sample = ORACLE_SAMPLE_HEADS, 8192
    for _ in range(max(0, min(args.warmup, 1))):
        run_oracle_sample(256, Hs, P["d"])
    vals, secs, threads = [], 0.0, 1
    for _ in range(args.steps):
        _, dt, threads = run_oracle_sample(T_sample, Hs, P["d"])
        vals.append(T_sample / (dt * P["H"] / Hs))
        secs += dt
    value = statistics.median(vals)
    sample = (f"per step {Hs} of the {P['H']} heads x the first {T_sample} of the "
              f"{P['T']} tokens of the workload; tokens/s extrapolated to the whole "
              f"workload; {args.steps} steps, fp64 C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / max(args.steps, 1),
        "ms_per_workload_extrapolated": 1000.0 * P["T"] / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded torch CPU generator)",
        "config": headline_config(),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def headline_config():
    P = PREFILL_SHAPE
    return {"workload": f"long prefill B={P['B']} H={P['H']} T={P['T']} d_k=d_v={P['d']} "
                        "bf16 + final state handed to one decode step",
            "B": P["B"], "H": P["H"], "T": P["T"], "d": P["d"], "chunk": 64,
            "l2": "inputs larger than L2 (6.4 GB per step)", "parallelism": "replicas"}


# ------------------------------------------------------------------- GPU arm
def device_prefill_inputs(seq_lens, H: int, d: int, seed: int, dev, nonzero_state=False):
    """The prefill recipe's distributions drawn on the device with a seeded
    CUDA generator (the benchmark's large workloads; their values are not
    compared with the oracle -- the parity tests draw on the host)."""
    import torch
    from kimi_delta_attention_12_gb300 import inputs
    g = torch.Generator(device=dev).manual_seed(seed)
    T = int(sum(seq_lens))
    unit = lambda t: t / t.norm(dim=-1, keepdim=True)
    q = unit(torch.randn(T, H, d, device=dev, generator=g)).bfloat16()
    k = unit(torch.randn(T, H, d, device=dev, generator=g)).bfloat16()
    v = torch.randn(T, H, d, device=dev, generator=g).bfloat16()
    z = torch.randn(T, H, d, device=dev, generator=g).bfloat16()
    beta = torch.sigmoid(torch.randn(T, H, device=dev, generator=g)).bfloat16()
    A = 0.5 * torch.randn(H, device=dev, generator=g)
    S0 = None
    if nonzero_state:
        S0 = 0.02 * torch.randn(len(seq_lens), H, d, d, device=dev, generator=g)
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int64), 0).to(torch.int32)
    return inputs.PrefillInputs(q, k, v, z, beta, A, S0, cu.to(dev))


def check_status(kda, ws, what):
    st = kda.workspace_status(ws)
    assert st == kda.KDA_OK, f"{what}: prefill kernel reported {kda.status_string(st)}"


def time_prefill(kda, sets, ws, o, S, cu_host, steps, warmup, stream, what, **kw):
    """Mean CUDA-event time (ms) of kda_prefill over `steps` calls after
    `warmup`, inputs rotating over `sets`; the status word is checked after
    the warm-up and after the timed calls."""
    import torch
    for i in range(warmup):
        x = sets[i % len(sets)]
        kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, x.initial_state, x.cu_seqlens,
                        cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws, **kw)
    check_status(kda, ws, what + " (warm-up)")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        x = sets[(warmup + i) % len(sets)]
        ev[i][0].record(stream)
        kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, x.initial_state, x.cu_seqlens,
                        cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws, **kw)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    check_status(kda, ws, what)
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def roofline(byts, flops, ms, peaks, traffic=None, kernel=None):
    gbs = byts / (ms / 1e3) / 1e9
    tf = flops / (ms / 1e3) / 1e12
    r = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": gbs / peaks["hbm_gbs"], "traffic": traffic, "kernel_ms": ms,
         "algorithmic_bytes": byts, "algorithmic_flops": flops,
         "peak_source": peaks["source"] + ", of measured copy peak",
         "tensor_tflops": tf, "tensor_frac": tf / peaks["bf16_tflops"]}
    if kernel:
        r["kernel"] = kernel
    return r


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
    if args.only in ("softplus", "backward", "conv", "prefill4k"):
        return four_k_only(args, rank, dev, stream, peaks)

    # ---- the headline: long prefill B=1, H=96, T=65536 + decode handoff ----
    P = PREFILL_SHAPE
    B, H, T, d = P["B"], args.prefill_heads or P["H"], args.prefill_tokens or P["T"], P["d"]
    byts, flops = prefill_algorithmic(B, H, T, d)
    x = device_prefill_inputs([T] * B, H, d, seed=100 + rank, dev=dev)
    cu_host = x.cu_seqlens.cpu()
    o = torch.empty(B * T, H, d, dtype=torch.bfloat16, device=dev)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=dev)
    ws = kda.alloc_workspace(B, B * T, H, d, d, torch.bfloat16, dev)
    minimal_ws = 256 + -(-4 * B * H // 256) * 256
    kernel_name = "kda_split_kernel" if ws.numel() > minimal_ws else "kda_chunked_kernel"
    o_dec = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens,
                        cu_seqlens_host=cu_host, o=o, final_state=S, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        # decode handoff: the next token of each head continues from S
        kda.kda_decode_step(x.q[:B], x.k[:B], x.v[:B], x.z[:B], x.beta[:B], x.A, S, o=o_dec)

    launches_per_step = 2
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    check_status(kda, ws, "headline prefill (warm-up)")
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    _barrier(pg)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            step(kev[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    _barrier(pg)
    check_status(kda, ws, "headline prefill")
    ms_total = _max_over_ranks(pg, t_start.elapsed_time(t_end))
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    ms_per_step = ms_total / args.steps
    value = world * B * T / (ms_per_step / 1e3)
    if args.only == "prefill":
        if rank == 0:
            r = roofline(byts, flops, kernel_ms, peaks, kernel=kernel_name)
            print(json.dumps({"only": "prefill", "H": H, "T": T, "value": value,
                              "unit": "tokens/s", "kernel_ms": kernel_ms,
                              "achieved_gbs": r["achieved"], "frac": r["frac"],
                              "tensor_tflops": r["tensor_tflops"], "clocks": clk.summary()}),
                  flush=True)
        return
    head = {"value": value, "ms_per_step": ms_per_step, "kernel_ms": kernel_ms,
            "kernel": kernel_name, "byts": byts, "flops": flops, "clk": clk,
            "launches_per_step": launches_per_step}
    headline = (x, o, S, ws, cu_host)

    # ---- the 4K prefill and the further rows on it ----
    four_k = measure_4k(args, dev, stream, peaks, rank)
    # ---- the varlen workload ----
    varlen = measure_varlen(args, dev, stream, peaks)
    return finish(args, world, rank, local, dev, stream, peaks, B, H, T, d, head, headline,
                  four_k, varlen, pg)


def four_k_sets(dev, rank):
    """Rotating copies of the 4K workload's inputs (host recipe), enough that
    each step's inputs are not L2-resident."""
    import torch
    from kimi_delta_attention_12_gb300 import inputs
    P = PREFILL_4K_SHAPE
    x_host = inputs.make_prefill_inputs([P["T"]] * P["B"], P["H"], P["d"], P["d"],
                                        torch.bfloat16, seed=rank)
    set_bytes, _ = prefill_algorithmic(P["B"], P["H"], P["T"], P["d"])
    nsets = max(2, -(-3 * L2_BYTES // set_bytes))
    sets = [x_host.to(dev)]
    for _ in range(nsets - 1):
        s0 = sets[0]
        sets.append(inputs.PrefillInputs(*(t.clone() if t is not None else None for t in
                                           (s0.q, s0.k, s0.v, s0.z, s0.beta, s0.A,
                                            s0.initial_state, s0.cu_seqlens))))
    return x_host, sets


def four_k_only(args, rank, dev, stream, peaks):
    """--only softplus|backward|conv|prefill4k: one further row (or the 4K
    prefill alone) for profiler captures."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    P = PREFILL_4K_SHAPE
    B, H, T, d = P["B"], P["H"], P["T"], P["d"]
    x_host, sets = four_k_sets(dev, rank)
    cu_host = sets[0].cu_seqlens.cpu()
    o = torch.empty(B * T, H, d, dtype=torch.bfloat16, device=dev)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=dev)
    ws = kda.alloc_workspace(B, B * T, H, d, d, torch.bfloat16, dev)
    if args.only == "softplus":
        r = measure_softplus(sets, ws, o, S, cu_host, args, stream)
        r["tokens_per_s"] = B * T / (r["kernel_ms"] / 1e3)
    elif args.only == "backward":
        r = measure_backward(sets, B, H, T, d, args, stream)
        r["frac"] = r["achieved_gbs"] / peaks["hbm_gbs"]
    elif args.only == "conv":
        r = measure_conv(sets, ws, o, S, cu_host, B, H, T, d, args, stream)
        r["frac"] = r["achieved_gbs"] / peaks["hbm_gbs"]
    else:
        ms = time_prefill(kda, sets, ws, o, S, cu_host, args.steps, args.warmup, stream,
                          "4K prefill")
        byts, flops = prefill_algorithmic(B, H, T, d)
        r = {"kernel_ms": ms, "tokens_per_s": B * T / (ms / 1e3),
             "roofline": roofline(byts, flops, ms, peaks)}
    if rank == 0:
        print(json.dumps(dict(r, only=args.only)), flush=True)


def measure_4k(args, dev, stream, peaks, rank):
    """The 4K prefill (B=1, H=32, T=4096) with its roofline, and the further
    rows measured on it: checkpoints, softplus gate, short convolutions,
    backward."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    P = PREFILL_4K_SHAPE
    B, H, T, d = P["B"], P["H"], P["T"], P["d"]
    x_host, sets = four_k_sets(dev, rank)
    cu_host = sets[0].cu_seqlens.cpu()
    o = torch.empty(B * T, H, d, dtype=torch.bfloat16, device=dev)
    S = torch.empty(B, H, d, d, dtype=torch.float32, device=dev)
    ws = kda.alloc_workspace(B, B * T, H, d, d, torch.bfloat16, dev)
    ms = time_prefill(kda, sets, ws, o, S, cu_host, args.steps, args.warmup, stream, "4K prefill")
    byts, flops = prefill_algorithmic(B, H, T, d)
    prefill_4k = {"workload": "prefill B=1 H=32 T=4096 d_k=d_v=128 bf16", "kernel_ms": ms,
                  "tokens_per_s": B * T / (ms / 1e3),
                  "roofline": roofline(byts, flops, ms, peaks,
                                       profiled_traffic("kda_split_kernel_b1_h32_t4096",
                                                        B * T * H),
                                       "kda_split_kernel")}
    ckpt = measure_checkpointed(sets, ws, o, S, cu_host, B, H, T, d, args, stream)
    ckpt["kernel_ms_plain"] = ms
    softplus = measure_softplus(sets, ws, o, S, cu_host, args, stream)
    softplus["tokens_per_s"] = B * T / (softplus["kernel_ms"] / 1e3)
    conv = measure_conv(sets, ws, o, S, cu_host, B, H, T, d, args, stream)
    conv["frac"] = conv["achieved_gbs"] / peaks["hbm_gbs"]
    bw = measure_backward(sets, B, H, T, d, args, stream)
    bw["frac"] = bw["achieved_gbs"] / peaks["hbm_gbs"]
    return {"prefill_4k": prefill_4k, "prefill_checkpointed": ckpt, "softplus_gate": softplus,
            "short_conv": conv, "backward": bw}


def measure_varlen(args, dev, stream, peaks):
    """The varlen workload: 16 packed sequences with lengths U[512, 16384]
    (seed 0), H=64, nonzero initial states: kernel time, tokens/s, roofline."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    from kimi_delta_attention_12_gb300 import inputs
    w = inputs.VARLEN_16
    H, d, N, T = w.H, w.d_k, w.N, w.total_T
    x = device_prefill_inputs(list(w.seq_lens), H, d, seed=200, dev=dev, nonzero_state=True)
    cu_host = x.cu_seqlens.cpu()
    o = torch.empty(T, H, d, dtype=torch.bfloat16, device=dev)
    S = torch.empty(N, H, d, d, dtype=torch.float32, device=dev)
    ws = kda.alloc_workspace(N, T, H, d, d, torch.bfloat16, dev)
    ms = time_prefill(kda, [x], ws, o, S, cu_host, args.steps, args.warmup, stream,
                      "varlen prefill")
    byts, flops = prefill_algorithmic(1, H, T, d, read_state=True, N=N)
    return {"workload": f"varlen prefill, {N} sequences U[512,16384] (total {T} tokens), "
                        f"H={H} d_k=d_v={d} bf16, initial states N(0,0.02)",
            "seq_lens": list(w.seq_lens), "kernel_ms": ms, "tokens_per_s": T / (ms / 1e3),
            "roofline": roofline(byts, flops, ms, peaks, kernel="kda_split_kernel")}


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
    check_status(kda, ws, "checkpointed prefill")
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
    the call's time and bandwidth on its algorithmic bytes.  With the host
    mirror of cu_seqlens the call runs the chunked backward (the split
    prefill keeping its chunk records and chunk-start states, the reverse
    state chain, the chunk-parallel assembly and the dA sum); with the device
    array alone it runs the recurrent fp32 backward, timed beside it."""
    import torch
    import kimi_delta_attention_12_gb300 as kda
    from kimi_delta_attention_12_gb300 import inputs
    x0 = sets[0]
    cu_host = x0.cu_seqlens.cpu()
    dO, dSf = inputs.make_upstream_grads(B * T, B, H, d, d, torch.bfloat16, seed=21)
    dO, dSf = dO.to(x0.q.device), dSf.to(x0.q.device)
    ws = torch.empty(kda.backward_workspace_bytes(B, B * T, H, d, d, torch.bfloat16),
                     dtype=torch.uint8, device=x0.q.device)
    n = min(args.steps, 3)

    def timed(host_cu, warm):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for i in range(warm + n):
            x = sets[i % len(sets)]
            if i >= warm:
                ev[i - warm][0].record(stream)
            kda.kda_backward(x.q, x.k, x.v, x.z, x.beta, x.A, dO, None, x.cu_seqlens,
                             host_cu, dS_final=dSf, workspace=ws)
            if i >= warm:
                ev[i - warm][1].record(stream)
        torch.cuda.synchronize()
        check_status(kda, ws, "backward")
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    ms = timed(cu_host, 3)
    ms_rec = timed(None, 1)
    byts = backward_algorithmic(B, H, T, d)
    return {"kernel": "kda_bwd_assemble_kernel",
            "form": "chunked, tensor cores (split prefill with chunk records, reverse state "
                    "chain, chunk-parallel assembly, dA sum)",
            "kernel_ms": ms, "steps": n, "tokens_per_s": B * T / (ms / 1e3),
            "algorithmic_bytes": byts, "achieved_gbs": byts / (ms / 1e3) / 1e9,
            "recurrent_fp32_ms": ms_rec}


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
    check_status(kda, ws, "prefill after the short convolutions")
    conv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    both_ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    # the same, fused: kda_prefill_conv (the convolutions inside the split
    # kernel's producers, the convolved tensors never in HBM)
    wsf = torch.empty(kda.prefill_conv_workspace_bytes(B, B * T, H, d, d, torch.bfloat16),
                      dtype=torch.uint8, device=dev)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for i in range(args.warmup + n):
        x = sets[i % len(sets)]
        if i >= args.warmup:
            fev[i - args.warmup][0].record(stream)
        kda.kda_prefill_conv(x.q, x.k, x.v, x.z, x.beta, x.A, w, cs_in, cs_out,
                             cu_seqlens=x.cu_seqlens, cu_seqlens_host=cu_host, silu=True,
                             o=o, final_state=S, workspace=wsf)
        if i >= args.warmup:
            fev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    check_status(kda, wsf, "prefill with the short convolutions fused")
    fused_ms = statistics.mean(a.elapsed_time(b) for a, b in fev)
    byts = conv_algorithmic(B, H, T, d, W)
    return {"kernel": "short_conv_kernel", "width": W, "silu": True, "kernel_ms": conv_ms,
            "algorithmic_bytes": byts, "achieved_gbs": byts / (conv_ms / 1e3) / 1e9,
            "conv_then_prefill_ms": both_ms,
            "conv_then_prefill_tokens_per_s": B * T / (both_ms / 1e3),
            "fused_conv_prefill_ms": fused_ms,
            "fused_conv_prefill_tokens_per_s": B * T / (fused_ms / 1e3)}


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
    check_status(kda, ws, "softplus-gate prefill")
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


def finish(args, world, rank, local, dev, stream, peaks, B, H, T, d, head, headline,
           four_k, varlen, pg):
    import torch
    import kimi_delta_attention_12_gb300 as kda
    x, o, S, ws, cu_host = headline
    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs from pinned host memory, runs kda_prefill
    # and reads o and the final state back into pinned host memory.  Steps are
    # pipelined the way a stream of requests would be: copy-in, prefill and
    # copy-out run on three streams with two device buffer sets, so that the
    # copy-in of step i + 1 overlaps the prefill of step i and the copy-out of
    # step i - 1 (host-to-device copies bound the step).
    pin = lambda t: t.cpu().pin_memory()
    hosts = tuple(pin(t) for t in (x.q, x.k, x.v, x.z, x.beta, x.A, x.cu_seqlens))
    ho = torch.empty(B * T, H, d, dtype=torch.bfloat16).pin_memory()
    hS = torch.empty(B, H, d, d, dtype=torch.float32).pin_memory()
    dbufs = [tuple(t for t in (x.q, x.k, x.v, x.z, x.beta, x.A, x.cu_seqlens)),
             tuple(torch.empty_like(t, device=dev) for t in hosts)]
    douts = [(o, S), (torch.empty_like(o), torch.empty_like(S))]
    h2d = sum(t.numel() * t.element_size() for t in hosts)
    d2h = ho.numel() * ho.element_size() + hS.numel() * hS.element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ws2 = torch.empty_like(ws)   # one workspace per buffer set (their prefills may overlap)
    wss = (ws, ws2)

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
                        o=ob, final_state=Sb, workspace=wss[b], stream=s_cmp)
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
    for w_ in wss:
        check_status(kda, w_, "end-to-end prefill")
    e2e_ms = _max_over_ranks(pg, e0.elapsed_time(e1)) / args.steps
    e2e_value = world * B * T / (e2e_ms / 1e3)
    del dbufs, douts, ws2

    # ---- decode workload: 64 consecutive steps on a resident 1.6 GB state ----
    D = DECODE_SHAPE
    dec_ms, dec_bytes, dec_gbs, dclk_summary = run_decode(dev, rank, local, stream)
    sp_ms, _, sp_gbs, _ = run_decode(dev, rank, local, stream, softplus_gate=True)
    four_k["softplus_gate"].update({"decode_ms_per_step": sp_ms, "decode_gbs": sp_gbs,
                                    "decode_frac": sp_gbs / peaks["hbm_gbs"]})
    cv_ms, cv_bytes, cv_gbs, _ = run_decode(dev, rank, local, stream, conv=True)
    four_k["short_conv"].update({"decode_kernels": "short_conv_decode_kernel + kda_recurrent_kernel",
                                 "decode_ms_per_step": cv_ms, "decode_bytes_per_step": cv_bytes,
                                 "decode_gbs": cv_gbs, "decode_frac": cv_gbs / peaks["hbm_gbs"]})

    if rank != 0:
        return
    # CPU baselines: the oracle on a sample of the headline workload, on the
    # whole 4K workload, and on each further row's workload
    cpu_tps, cpu_threads, cpu_sample = headline_cpu_baseline(H, T, d)
    P4 = PREFILL_4K_SHAPE
    c4_tps, c4_threads, c4_sample = cpu_baseline(P4["H"], P4["T"], P4["d"], cpu_seconds=4.0)
    four_k["prefill_4k"]["cpu_baseline"] = {"value": c4_tps, "unit": "tokens/s",
                                            "cores": c4_threads, "kind": "oracle",
                                            "sample": c4_sample}
    row_cpu = row_cpu_baselines(P4["H"], P4["T"], P4["d"], D["B"], D["H"])
    for key in ("softplus_gate", "short_conv", "backward"):
        four_k[key]["cpu_baseline"] = row_cpu[key]
    byts, flops, kernel_ms = head["byts"], head["flops"], head["kernel_ms"]
    traffic = profiled_traffic("kda_split_kernel_b1_h96_t4096", B * T * H)
    rl = roofline(byts, flops, kernel_ms, peaks, traffic, head["kernel"])
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generators; the long-prefill inputs, 6.4 GB > L2, drawn on "
                "the device with the recipe's distributions)",
        "config": headline_config(),
        "roofline": rl,
        "decode": {"metric": "decode state GB/s", "value": dec_gbs, "unit": "GB/s",
                   "ms_per_step": dec_ms, "bytes_per_step": dec_bytes,
                   "config": {"workload": "decode B=256 H=96 d=128 fp32 state, bf16 inputs",
                              "steps": D["steps"]},
                   "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"]},
                   "clocks": dclk_summary, "cpu_baseline": row_cpu["decode"]},
        "prefill_varlen": varlen,
        **four_k,
        "cpu_baseline": {"value": cpu_tps, "unit": "tokens/s", "cores": cpu_threads,
                         "kind": "oracle", "sample": cpu_sample, "cpu_model": cpu_model()},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelining": "copy-in, prefill and copy-out of consecutive steps overlap "
                              "(three streams, two device buffer sets)"},
        "gpu_launches": head["launches_per_step"] * args.steps,
        "clocks": head["clk"].summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--only", choices=["all", "prefill", "prefill4k", "decode", "conv",
                                       "backward", "softplus"],
                    default="all",
                    help="run one part only (for profiler captures); the default runs all")
    ap.add_argument("--prefill-heads", type=int, default=0,
                    help="--only prefill: heads of the long prefill (default 96; smaller "
                         "cases for profiler captures)")
    ap.add_argument("--prefill-tokens", type=int, default=0,
                    help="--only prefill: tokens of the long prefill (default 65536)")
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
