#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300: chunked prefill and the decode step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kda|reference]

One step is one pass of the hot path over one batch:
  * prefill  -- kda_prefill over prefill_h32_t1m (1 sequence, H=32,
                T=1,048,576, d=128, bf16 q/k/v, fp32 gates and state), the
                long-context workload; the headline ``value`` is its tokens/s;
  * decode   -- kda_decode_step over decode_1024x32 (1024 sequences x 32
                heads, d=128, 2 GiB fp32 state updated in place); reported in
                the ``decode`` object as achieved state GB/s.
Two more prefill workloads are reported beside them: ``varlen`` (varlen16_h32,
16 packed sequences with S0 in and S_final out) and ``short``
(prefill_h16_t4096, one 4096-token prompt of 16 heads).
Each is timed with CUDA events on the launching stream, W untimed warm-up
steps first, each timed region bracketed by a barrier and a device
synchronisation, max over ranks.  Inputs are far larger than L2 (51.7 GB per
prefill step, 2 GiB of state per decode step) except for ``short`` (102 MB),
which flushes L2 before every timed launch.  After each prefill section the
workspace's device status words are read; a wait that gave up voids the run.

Under torchrun each rank processes its own batch (independent sequences, no
data-path collective: weak scaling); the process group is used only for the
barrier and the max-over-ranks reduction of timings.

``--impl reference`` times the float64 CPU oracle (the only reference that
exists for this method) on a bounded sample of the same workload, on this
machine's host cores, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s and decode state GB/s at H=32,d=128; % of GB300 roofline"
PREFILL_WORKLOAD = 4          # prefill_h32_t1m
DECODE_WORKLOAD = 5           # decode_1024x32
VARLEN_WORKLOAD = 3           # varlen16_h32

# Algorithmic work per token x head at d = 128 (counts used for the roofline):
# bytes = q, k, v (bf16) 768 + log_alpha 512 + beta 4 + o (bf16) 256.
BYTES_PER_TOKEN_HEAD = 1540
# flops at chunk 64 with full 64x64 tiles: 2C(3d + 2d) + 6 d^2.
FLOPS_PER_TOKEN_HEAD = 2 * 64 * (3 * 128 + 2 * 128) + 6 * 128 * 128


def state_bytes(d):
    return 4 * d * d


def decode_bytes_per_unit(d):
    # fp32 state read + write, plus the token's q, k, v (bf16), log_alpha (fp32),
    # beta (fp32) and o (bf16).
    return 2 * state_bytes(d) + 3 * 2 * d + 4 * d + 4 + 2 * d


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def kernel_source_sha(files):
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key, files):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)[kernel_key]
    except (OSError, KeyError, ValueError):
        return None
    if t.get("source_sha") != kernel_source_sha(files):
        return None
    return t.get("bytes_per_launch")


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": [], "samples": 0}
        # Median over samples taken while the GPU was loaded (upper half of the
        # observed clocks excludes idle gaps at the edges).
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for_smi(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u and not u.startswith("GPU-"):
            u = "GPU-" + u
        if u and len(u) > 8:
            return u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev]
    return dev


# --------------------------------------------------------------------------
# distributed helpers (host logic, also exercised by gloo tests on CPU)
# --------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(base_seed, rank):
    """Each rank draws its own batch of the same workload (weak scaling)."""
    return base_seed + 1000003 * rank


def max_over_ranks(value, world, device=None):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# the oracle baseline (CPU)
# --------------------------------------------------------------------------
def oracle_sample_inputs(tokens, heads, seed):
    import synth
    w = synth.WORKLOADS[PREFILL_WORKLOAD]
    return synth.generate([tokens], heads, w.d, w.d, dtype=w.dtype, gate=w.gate,
                          q_scale=w.q_scale, seed=seed, device="cpu")


def time_oracle_prefill(tokens, heads, seed, nthreads):
    import oracle
    inp = oracle_sample_inputs(tokens, heads, seed)
    args = [x.double().numpy() for x in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    t0 = time.perf_counter()
    oracle.prefill(*args, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(target_s=15.0, heads=32):
    """Oracle tokens/s at H=32 on a bounded sample: the first ``n`` tokens of
    all 32 heads of a prefill_h32_t1m-shaped batch, n sized to ~target_s."""
    import oracle
    oracle.build()
    threads = min(heads, oracle.default_threads())
    probe = 256
    dt = time_oracle_prefill(probe, heads, 1, threads)
    n = int(max(probe, min(1 << 20, probe * target_s / max(dt, 1e-3))))
    n = max(64, (n // 64) * 64)
    dt = time_oracle_prefill(n, heads, 2, threads)
    return {"value": n / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "first %d tokens x %d heads of a prefill_h32_t1m-shaped batch "
                      "(float64 oracle, %.1f s)" % (n, heads, dt)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    heads = 32
    threads = min(heads, oracle.default_threads())
    # One step = the oracle over a bounded sample of the workload, sized so
    # the whole run stays within a few minutes.
    probe = 128
    dt = time_oracle_prefill(probe, heads, 1, threads)
    per_step_s = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    n = int(max(64, probe * per_step_s / max(dt, 1e-3)) // 64 * 64)
    for i in range(args.warmup):
        time_oracle_prefill(n, heads, 10 + i, threads)
    times = [time_oracle_prefill(n, heads, 100 + i, threads) for i in range(args.steps)]
    total = sum(times)
    value = n * args.steps / total
    sample = ("first %d tokens x %d heads of a prefill_h32_t1m-shaped batch per step "
              "(float64 oracle on %d host threads)" % (n, heads, threads))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill_h32_t1m", "H": 32, "d": 128,
                   "tokens_per_step": n, "sampled": True},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------
class DeviceWaitGaveUp(RuntimeError):
    """A timed launch reported a device-side wait that gave up: its outputs
    are incomplete and its time is not a measurement."""


def check_status_words(ws, what):
    """The prefill workspace's device-side status words after a timed section
    (the caller zeroes the workspace before it): word 2 bit 1 = a wait gave
    up, word 6 = the producer / consumer kernel aborted, word 1 = invalid
    cu_seqlens.  Any of them set voids the section's numbers."""
    words = ws[:28].view(dtype=__import__("torch").int32).cpu().tolist()
    if words[2] & 2 or words[6] != 0 or words[1] != 0:
        raise DeviceWaitGaveUp("%s: device status words timeout=%d abort=%d cu_error=%d; "
                               "refusing to report a time" % (what, words[2], words[6], words[1]))
# The prefill kernel that dominates the timed call, and the sources that
# define it: the producer / consumer kernel when the workspace kda_prefill
# asks for includes its operand ring (few (sequence, head) units), else the
# single-CTA kernel.
_TC_COMMON = ["gated_delta_rule_05_gb300/csrc/kda_tc_chunk.cuh",
              "gated_delta_rule_05_gb300/csrc/kda_sm100.cuh",
              "gated_delta_rule_05_gb300/csrc/kda_internal.cuh"]
PREFILL_KERNELS = {
    "prefill_split_kernel": ["gated_delta_rule_05_gb300/csrc/kda_prefill_split.cu"] + _TC_COMMON,
    "prefill_tc_kernel": ["gated_delta_rule_05_gb300/csrc/kda_prefill_tc.cu"] + _TC_COMMON,
}


def prefill_kernel_name(ws_bytes, num_seqs):
    base = 256 + (num_seqs * 4 + 255) // 256 * 256
    return "prefill_split_kernel" if ws_bytes > base else "prefill_tc_kernel"
DECODE_SOURCES = ["gated_delta_rule_05_gb300/csrc/kda_decode.cu",
                  "gated_delta_rule_05_gb300/csrc/kda_internal.cuh"]
DECODE_KERNEL = "decode_kernel"


def run_kda(args):
    import torch
    import synth
    import gated_delta_rule_05_gb300 as kda

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    kda.build()
    kda.lib()
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)

    line = {}
    smi_id = gpu_id_for_smi(torch, local)
    if args.only in ("all", "prefill"):
        line.update(bench_prefill(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id))
    if args.only in ("all", "decode"):
        line["decode"] = bench_decode(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id)
    if args.only in ("all", "varlen"):
        line["varlen"] = bench_varlen(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id)
    if args.only in ("all", "short"):
        line["short"] = bench_short(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id)
    if rank == 0:
        if "value" not in line:        # one section only: that section leads the line
            d = next(line[k] for k in ("decode", "varlen", "short") if k in line)
            line.update({"metric": METRIC, "value": d["value"], "unit": d["unit"], "n_gpus": world,
                         "steps": args.steps, "warmup": args.warmup,
                         "ms_per_step": d["ms_per_step"], "higher_is_better": True,
                         "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                         "data": "synthetic", "config": {"workload": d["workload"]},
                         "roofline": d["roofline"], "clocks": d["clocks"],
                         "gpu_launches": d["gpu_launches"], "cpu_baseline": None,
                         "e2e": None})
        else:
            line["gpu_launches"] = line.get("gpu_launches", 0) + sum(
                line.get(k, {}).get("gpu_launches", 0) for k in ("decode", "varlen", "short"))
        if args.only == "all" and world == 1 and not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline()   # rank 0 at N=1 only
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def bench_prefill(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id):
    wp = synth.WORKLOADS[PREFILL_WORKLOAD]
    lengths = [args.tokens] if args.tokens else synth.draw_lengths(wp)
    workload = wp.name if not args.tokens else "prefill_h32_t%d" % args.tokens
    inp = synth.generate(lengths, wp.H, wp.d, wp.d, dtype=wp.dtype,
                         gate=wp.gate, q_scale=wp.q_scale, s0_std=wp.s0_std,
                         seed=rank_seed(wp.seed, rank), device=dev)
    T, H, d = inp.q.shape
    o = torch.empty((T, H, d), dtype=inp.q.dtype, device=dev)
    S_final = torch.empty((1, H, d, d), dtype=torch.float32, device=dev)
    # zeroed: the timeout word is never cleared by the library
    ws = torch.zeros(kda.kda_prefill_workspace_bytes(1, H, d, d), dtype=torch.uint8, device=dev)
    kernel = prefill_kernel_name(ws.numel(), 1)

    def prefill():
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, S0=None,
                        cu_seqlens=inp.cu_seqlens, o=o, S_final=S_final,
                        workspace=ws, stream=stream)

    for _ in range(args.warmup):
        prefill()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_id) as clk:
        t_wall = time.perf_counter()
        for s, e in ev:
            s.record(stream)
            prefill()
            e.record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    check_status_words(ws, workload)
    prefill_ms = sum(s.elapsed_time(e) for s, e in ev)
    prefill_ms_max = max_over_ranks(prefill_ms, world, dev)
    ms_per_step = prefill_ms_max / args.steps
    tokens_all = T * world * args.steps
    value = tokens_all / (prefill_ms_max / 1e3)
    launch_ms = prefill_ms / args.steps          # this rank, per launch
    alg_bytes = T * H * BYTES_PER_TOKEN_HEAD + H * state_bytes(d)     # + the S_final write
    alg_flops = T * H * FLOPS_PER_TOKEN_HEAD
    achieved = alg_bytes / (launch_ms / 1e3) / 1e9
    traffic = committed_traffic(workload + "/" + kernel, PREFILL_KERNELS[kernel])
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": peaks["source"], "kernel": kernel,
                "algorithmic_bytes_per_launch": alg_bytes,
                "tensor_tflops_achieved": alg_flops / (launch_ms / 1e3) / 1e12,
                "tensor_frac": (alg_flops / (launch_ms / 1e3) / 1e12) / peaks["bf16_tflops"]}
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload, "num_seqs": 1, "seq_len": T, "H": H,
                   "d_k": d, "d_v": d, "io_dtype": "bf16", "state_dtype": "fp32",
                   "S0": None, "S_final": "written",
                   "tokens_per_step_per_gpu": T, "parallelism": "dp%d" % world,
                   "l2": "inputs larger than L2 (%.1f GB per step)" % (alg_bytes / 1e9)},
        "roofline": roofline,
        # per prefill call: the work-list kernel + the tensor-core kernel
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_prefill": t_wall,
    }
    if not args.no_e2e:
        out["e2e"] = run_e2e(kda, torch, inp, dev, stream, args, world)
    return out


def bench_decode(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id):
    wd = synth.WORKLOADS[DECODE_WORKLOAD]
    dinp = synth.generate(synth.draw_lengths(wd), wd.H, wd.d, wd.d, dtype=wd.dtype,
                          gate=wd.gate, q_scale=wd.q_scale, s0_std=wd.s0_std,
                          seed=rank_seed(wd.seed, rank), device=dev)
    S = dinp.S0
    od = torch.empty_like(dinp.v)
    Nd = dinp.q.shape[0]

    def decode():
        kda.kda_decode_step(dinp.q, dinp.k, dinp.v, dinp.log_alpha, dinp.beta, S,
                            o=od, stream=stream)

    for _ in range(args.warmup):
        decode()
    torch.cuda.synchronize(dev)
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_id) as dclk:
        for s, e in dev_ev:
            s.record(stream)
            decode()
            e.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    dec_ms = sum(s.elapsed_time(e) for s, e in dev_ev)
    dec_ms_max = max_over_ranks(dec_ms, world, dev)
    units = Nd * wd.H
    dec_bytes = units * decode_bytes_per_unit(wd.d)
    dec_gbs_all = dec_bytes * world * args.steps / (dec_ms_max / 1e3) / 1e9
    dec_achieved = dec_bytes / (dec_ms / args.steps / 1e3) / 1e9
    return {
        "value": dec_gbs_all, "unit": "GB/s", "ms_per_step": dec_ms_max / args.steps,
        "workload": "decode_1024x32", "tokens_per_step": Nd * world,
        "roofline": {"bound": "hbm", "achieved": dec_achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": dec_achieved / peaks["hbm_gbs"],
                     "traffic": committed_traffic("decode_1024x32/" + DECODE_KERNEL,
                                                  DECODE_SOURCES),
                     "peak_source": peaks["source"], "kernel": DECODE_KERNEL,
                     "algorithmic_bytes_per_launch": dec_bytes},
        "gpu_launches": args.steps,
        "clocks": dclk.summary(),
    }


def bench_varlen(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id):
    """varlen16_h32: 16 packed sequences x 32 heads with an initial state and
    S_final returned.  512 (sequence, head) units: the single-CTA tensor-core
    kernel, one CTA per unit, longest sequences first."""
    wv = synth.WORKLOADS[VARLEN_WORKLOAD]
    lengths = synth.draw_lengths(wv)
    name = wv.name
    if args.varlen_scale != 1.0:
        lengths = [max(1, int(round(x * args.varlen_scale))) for x in lengths]
        name = "%s_x%g" % (wv.name, args.varlen_scale)
    vin = synth.generate(lengths, wv.H, wv.d, wv.d, dtype=wv.dtype, gate=wv.gate,
                         q_scale=wv.q_scale, s0_std=wv.s0_std, seed=rank_seed(wv.seed, rank),
                         device=dev)
    N = len(vin.lengths)
    T, H, d = vin.q.shape
    ov = torch.empty_like(vin.v)
    Sf = torch.empty_like(vin.S0)
    ws = torch.zeros(kda.kda_prefill_workspace_bytes(N, H, d, d), dtype=torch.uint8, device=dev)
    kernel = prefill_kernel_name(ws.numel(), N)

    def run():
        kda.kda_prefill(vin.q, vin.k, vin.v, vin.log_alpha, vin.beta, S0=vin.S0,
                        cu_seqlens=vin.cu_seqlens, o=ov, S_final=Sf, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_id) as clk:
        for s, e in ev:
            s.record(stream)
            run()
            e.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    check_status_words(ws, name)
    ms = sum(s.elapsed_time(e) for s, e in ev)
    ms_max = max_over_ranks(ms, world, dev)
    alg_bytes = T * H * BYTES_PER_TOKEN_HEAD + 2 * N * H * d * d * 4   # + S0 read, S_final write
    achieved = alg_bytes / (ms / args.steps / 1e3) / 1e9
    return {
        "value": T * world * args.steps / (ms_max / 1e3), "unit": "tokens/s",
        "ms_per_step": ms_max / args.steps, "workload": name, "tokens_per_step": T * world,
        "num_seqs": N, "lengths": [int(x) for x in vin.lengths],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": committed_traffic(name + "/" + kernel, PREFILL_KERNELS[kernel]),
                     "peak_source": peaks["source"], "kernel": kernel,
                     "algorithmic_bytes_per_launch": alg_bytes},
        # per call: the work-list kernel + the tensor-core kernel
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }


SHORT_WORKLOAD = 2            # prefill_h16_t4096
L2_FLUSH_BYTES = 512 << 20    # well above the 129 MB L2


def bench_short(args, kda, torch, synth, peaks, stream, dev, rank, world, smi_id):
    """prefill_h16_t4096: one 4096-token sequence of 16 heads (102 MB of
    inputs and outputs, less than L2), S_final returned.  16 units: the
    producer / consumer kernel with a 64-chunk chain per unit.  L2 is flushed
    (a 512 MB write) before every timed launch, outside its events."""
    ws_ = synth.WORKLOADS[SHORT_WORKLOAD]
    sin = synth.generate(synth.draw_lengths(ws_), ws_.H, ws_.d, ws_.d, dtype=ws_.dtype,
                         gate=ws_.gate, q_scale=ws_.q_scale, s0_std=ws_.s0_std,
                         seed=rank_seed(ws_.seed, rank), device=dev)
    T, H, d = sin.q.shape
    o = torch.empty_like(sin.v)
    Sf = torch.empty((1, H, d, d), dtype=torch.float32, device=dev)
    ws = torch.zeros(kda.kda_prefill_workspace_bytes(1, H, d, d), dtype=torch.uint8, device=dev)
    kernel = prefill_kernel_name(ws.numel(), 1)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # the segmented call cuts this prompt in two (an explicit count: the
    # library's own choice leaves a 64-chunk chain uncut)
    ws_seg = torch.zeros(kda.kda_prefill_segmented_workspace_bytes(T, H, d, d, 2),
                         dtype=torch.uint8, device=dev)

    def run():
        kda.kda_prefill(sin.q, sin.k, sin.v, sin.log_alpha, sin.beta, S0=None,
                        cu_seqlens=None, o=o, S_final=Sf, workspace=ws, stream=stream)

    def run_segmented():
        kda.kda_prefill_segmented(sin.q, sin.k, sin.v, sin.log_alpha, sin.beta, S0=None,
                                  segments=2, o=o, S_final=Sf, workspace=ws_seg, stream=stream)

    steps = max(args.steps, 20)

    def timed(fn, wsb):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        with ClockSampler(smi_id) as clk, torch.cuda.stream(stream):
            for s, e in ev:
                flush.fill_(1)
                s.record(stream)
                fn()
                e.record(stream)
            torch.cuda.synchronize(dev)
        barrier(world)
        check_status_words(wsb, ws_.name)
        return sorted(s.elapsed_time(e) for s, e in ev), clk

    times, clk = timed(run, ws)
    seg_times, _ = timed(run_segmented, ws_seg)
    ms = sum(times)
    ms_max = max_over_ranks(ms, world, dev)
    # A prompt of few heads (one tensor-parallel shard of a layer), where the
    # segmented call pays: 4 heads x 32,768 tokens, the distributions above.
    fh = synth.generate([32768], 4, d, d, dtype=ws_.dtype, gate=ws_.gate, q_scale=ws_.q_scale,
                        seed=rank_seed(ws_.seed, rank) + 1, device=dev)
    fo = torch.empty_like(fh.v)
    fS = torch.empty((1, 4, d, d), dtype=torch.float32, device=dev)
    fws = torch.zeros(kda.kda_prefill_workspace_bytes(1, 4, d, d), dtype=torch.uint8, device=dev)
    fws_seg = torch.zeros(kda.kda_prefill_segmented_workspace_bytes(32768, 4, d, d, 0),
                          dtype=torch.uint8, device=dev)
    fh_plain, _ = timed(lambda: kda.kda_prefill(fh.q, fh.k, fh.v, fh.log_alpha, fh.beta, o=fo,
                                                S_final=fS, workspace=fws, stream=stream), fws)
    fh_seg, _ = timed(lambda: kda.kda_prefill_segmented(fh.q, fh.k, fh.v, fh.log_alpha, fh.beta,
                                                        segments=0, o=fo, S_final=fS,
                                                        workspace=fws_seg, stream=stream), fws_seg)
    del fh, fo, fS, fws, fws_seg
    alg_bytes = T * H * BYTES_PER_TOKEN_HEAD + H * state_bytes(d)       # + the S_final write
    achieved = alg_bytes / (ms / steps / 1e3) / 1e9
    return {
        "value": T * world * steps / (ms_max / 1e3), "unit": "tokens/s",
        "ms_per_step": ms_max / steps, "ms_median": times[len(times) // 2],
        "workload": ws_.name, "tokens_per_step": T * world, "steps": steps,
        "l2": "flushed before each timed launch (%d MB write)" % (L2_FLUSH_BYTES >> 20),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": None, "peak_source": peaks["source"], "kernel": kernel,
                     "algorithmic_bytes_per_launch": alg_bytes},
        # per call: the work-list kernel + the tensor-core kernel; the
        # segmented call adds the scan and the fix-up; both again for the
        # few-heads prompt
        "gpu_launches": 2 * (2 * steps + 4 * steps),
        "clocks": clk.summary(),
        # the same prompt through kda_prefill_segmented in two segments
        # (chunk-group parallel prefill; same results), and a few-heads prompt
        # with the segment count chosen by the library (6 at 4 heads)
        "segmented": {"segments": 2, "ms_per_step": sum(seg_times) / steps,
                      "ms_median": seg_times[len(seg_times) // 2],
                      "tokens_per_s": T * steps / (sum(seg_times) / 1e3),
                      "speedup_vs_kda_prefill": sum(times) / sum(seg_times),
                      "workspace_bytes": int(ws_seg.numel()),
                      "few_heads_h4_t32768": {
                          "kda_prefill_ms": sum(fh_plain) / steps,
                          "segmented_ms": sum(fh_seg) / steps,
                          "speedup_vs_kda_prefill": sum(fh_plain) / sum(fh_seg)}},
    }


def host_memory_available():
    """Bytes of host memory this process may still use (MemAvailable, bounded
    by a cgroup limit when one is set)."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    avail = int(ln.split()[1]) * 1024
    except OSError:
        pass
    for path in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(path) as f:
                lim = f.read().strip()
            if lim.isdigit():
                used = 0
                for up in ("/sys/fs/cgroup/memory.current",
                           "/sys/fs/cgroup/memory/memory.usage_in_bytes"):
                    try:
                        with open(up) as g:
                            used = int(g.read().strip())
                        break
                    except (OSError, ValueError):
                        pass
                left = int(lim) - used
                avail = left if avail is None else min(avail, left)
        except OSError:
            pass
    return avail if avail is not None else 8 << 30


E2E_SEGMENT_TOKENS = 65536


def run_e2e(kda, torch, inp, dev, stream, args, world):
    """Same metric through the C ABI with HOST buffers: kda_prefill_host takes
    the step's inputs in pinned host memory and returns o to pinned host
    memory, pipelining copies in, compute and copies out over segments of
    E2E_SEGMENT_TOKENS tokens on three streams.  Every copy is inside the
    timed region: the copy-in stream waits for the start event, and the
    compute stream (which the end event follows) waits for the last copy out."""
    T_full, H, d = inp.q.shape
    # Pinned host memory is capped at 30 % of what the host reports available;
    # if the whole batch does not fit, the e2e leg runs on its first T tokens
    # and says so.
    per_token = H * BYTES_PER_TOKEN_HEAD
    budget = int(0.3 * host_memory_available())
    T = min(T_full, max(64, budget // per_token // 64 * 64))
    # The host buffers are written by the CPU first, as a caller's prompt
    # buffers are: pinned pages that only the GPU has touched are mapped for
    # it lazily and the first passes over them run at a fraction of the link
    # rate (measured: 37, then 66, then 193 GB/s for 17 GB device-to-host).
    host = {}
    try:
        for name in ("q", "k", "v", "log_alpha", "beta"):
            t = getattr(inp, name)[:T]
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.zero_()
            h.copy_(t)
            host[name] = h
        o_host = torch.empty((T, H, d), dtype=inp.q.dtype, pin_memory=True)
        o_host.zero_()
    except RuntimeError as exc:
        return {"value": None, "unit": "tokens/s", "error": "pinned allocation failed: %s" % exc}
    torch.cuda.synchronize(dev)
    hp = kda.HostPrefill(H, d, inp.q.dtype, segment_tokens=E2E_SEGMENT_TOKENS, device=dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_host.numel() * o_host.element_size()

    def step():
        hp(host["q"], host["k"], host["v"], host["log_alpha"], host["beta"], o_host)

    steps = max(1, min(args.steps, 5))
    for _ in range(min(args.warmup, 2)):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(hp.compute)
    hp.h2d.wait_event(s)
    for _ in range(steps):
        step()
    e.record(hp.compute)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms = max_over_ranks(s.elapsed_time(e), world, dev)
    res = {"value": T * world * steps / (ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
           "ms_per_step": ms / steps, "tokens_per_step_per_gpu": T,
           "whole_batch": T == T_full, "api": "kda_prefill_host",
           "segment_tokens": E2E_SEGMENT_TOKENS,
           "link_gbs": host_link_rates(torch, dev, hp.h2d)}
    del host, o_host, hp
    return res


def host_link_rates(torch, dev, stream, nbytes=1 << 29, reps=8):
    """Plain pinned-copy rates of the host link right after the e2e leg (the
    e2e leg is bound by them and they vary between hosts and over time)."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h.zero_()
    g = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", g, h), ("d2h", h, g)):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)          # first pass maps the pages
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            for _ in range(reps):
                dst.copy_(src, non_blocking=True)
            e.record(stream)
        torch.cuda.synchronize(dev)
        out[name] = nbytes * reps / (s.elapsed_time(e) / 1e3) / 1e9
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "varlen", "short"],
                    default="all",
                    help="time only one part (profiling runs)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="prefill length override (profiling runs on a smaller case)")
    ap.add_argument("--varlen-scale", type=float, default=1.0,
                    help="scale the varlen workload's sequence lengths (profiling a smaller case)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "kda":
        print("bench.py: note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_kda(args)


if __name__ == "__main__":
    sys.exit(main())
