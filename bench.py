#!/usr/bin/env python3
"""Benchmark of the chunked Gated DeltaNet prefill (one JSON line on stdout).

Default workload: B=1, T=4096, Hk=16, Hv=32, dk=dv=128 (bf16 q/k/v, fp32 g/beta,
zero initial state, fp32 final state), synthetic and seeded.  A "step" is one
gdn_prefill call over that batch (all kernels of the path).  The inputs (~104 MB)
fit in L2, so a 256 MB buffer is written between timed steps to flush it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path has
no exchange step) and rank 0 prints the whole-job line.  ``--impl reference``
times the float64 CPU oracle on the host cores instead (its only other user).
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

import numpy as np  # noqa: E402

from hybrid_linear_attention_prefill_gb300.inputs import HEADLINE, WORKLOADS, make_gdn_inputs, workload  # noqa: E402

METRIC = "Gated DeltaNet prefill tokens/s at T=4096,Hv=32; % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CHUNK = 64


# ---------------------------------------------------------------------------
# algorithmic bytes and flops (per workload)
# ---------------------------------------------------------------------------
def algorithmic(inp):
    """Bytes each tensor of the path must move once, and the triangular-half flops."""
    Tt, Hk, Hv, dk, dv, B = inp.total_tokens, inp.Hk, inp.Hv, inp.dk, inp.dv, inp.B
    qk = 2 * Tt * Hk * dk * 2
    vv = Tt * Hv * dv * 2
    oo = Tt * Hv * dv * 2
    gb = 2 * Tt * Hv * 4
    st = B * Hv * dv * dk * 4
    init = st if inp.init is not None else 0
    cu = 4 * (B + 1) if inp.cu_seqlens is not None else 0
    total = qk + vv + oo + gb + st + init + cu
    flops = Tt * Hv * (CHUNK * (3 * dk + 2 * dv) + 6 * dk * dv)
    # per kernel: preparation reads q, k, g, beta; the state carry reads q, k, v, g,
    # beta (and the initial state) and writes o and the final state
    return dict(total=total, flops=flops, prep=qk + gb + cu, chain=total)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, source="fallback")

    def find(keys):
        for k in keys:
            if k in d and isinstance(d[k], (int, float)):
                return float(d[k])
        for v in d.values():
            if isinstance(v, dict):
                for k in keys:
                    if k in v and isinstance(v[k], (int, float)):
                        return float(v[k])
        return None

    hbm = find(["hbm_gbs", "hbm_GBps", "hbm_gb_s"])
    bf16 = find(["bf16_tflops", "bf16_TFLOPs"])
    return dict(hbm=hbm or FALLBACK_HBM_GBS, bf16=bf16 or FALLBACK_BF16_TFLOPS,
                source="measured" if hbm else "fallback")


def traffic_record(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this workload and the
    kernel source is unchanged since."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "hybrid_linear_attention_prefill_gb300", "csrc", rec["source"])
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if sha != rec.get("source_sha256_16"):
        return None
    return rec


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # raw samples (summarised into the JSON line) go to $GDN_BENCH_OUT or the temp directory
        import tempfile

        out_dir = os.environ.get("GDN_BENCH_OUT") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def to_device(inp, torch, dev):
    def t(a, dt=None):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(dt) if dt is not None else x).to(dev)

    return dict(q=t(inp.q.view(np.int16), torch.bfloat16), k=t(inp.k.view(np.int16), torch.bfloat16),
                v=t(inp.v.view(np.int16), torch.bfloat16), g=t(inp.g), beta=t(inp.beta),
                cu=None if inp.cu_seqlens is None else t(inp.cu_seqlens),
                init=None if inp.init is None else t(inp.init))


def host_cores():
    """Core counts of the host: what the C++ runtime would report as its hardware
    concurrency (all online CPUs) and what `nproc` reports (the CPUs this process may
    run on)."""
    hw = os.cpu_count() or 1
    try:
        avail = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        avail = hw
    return hw, avail


def workload_config(args, inp, world):
    """The `config` object both arms print for the same workload."""
    return {"workload": args.workload, "B": inp.B, "T": inp.T, "Hk": inp.Hk, "Hv": inp.Hv, "dk": inp.dk,
            "dv": inp.dv, "tokens": inp.total_tokens, "l2": "flushed between timed steps (256 MB write)",
            "parallelism": f"replicas x{world}", "levels": args.levels}


def cpu_baseline_oracle(inp, target_s=1.5):
    """Time the float64 oracle as it stands on the host cores on a bounded sample:
    all value heads of the first `n` tokens of every sequence, n sized to ~target_s of
    wall time; when the whole workload takes less, it is run again until ~target_s.
    The same sample is then run once on a single thread."""
    import oracle

    cores = oracle.num_cpus()
    # calibrate on a small slice
    n_cal = min(256, inp.total_tokens)
    sub = slice_tokens(inp, n_cal)
    t0 = time.perf_counter()
    oracle.prefill_inputs(sub, want_final=False, nthreads=cores)
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(min(inp.total_tokens, max(n_cal, n_cal * target_s / dt)))
    sub = slice_tokens(inp, n)
    runs, dt = 0, 0.0
    while runs == 0 or (dt < target_s and runs < 64):
        t0 = time.perf_counter()
        oracle.prefill_inputs(sub, want_final=True, nthreads=cores)
        dt += time.perf_counter() - t0
        runs += 1
    t0 = time.perf_counter()
    oracle.prefill_inputs(sub, want_final=True, nthreads=1)
    dt1 = time.perf_counter() - t0
    hw, avail = host_cores()
    return {"value": runs * sub.total_tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "hardware_concurrency": hw, "nproc": avail,
            "single_thread": {"value": sub.total_tokens / dt1, "unit": "tokens/s", "wall_s": round(dt1, 3)},
            "sample": f"first {sub.total_tokens} of {inp.total_tokens} tokens, all {inp.Hv} value heads, "
                      f"float64 token loop, {runs} run(s), {dt:.2f} s wall on {cores} threads; "
                      f"once on 1 thread, {dt1:.2f} s wall"}


def slice_tokens(inp, n):
    """The first n tokens of a single-sequence problem (packed problems: the first sequences)."""
    import copy

    s = copy.copy(inp)
    if inp.cu_seqlens is None and inp.B == 1:
        for f in ("q", "k", "v", "g", "beta"):
            setattr(s, f, getattr(inp, f)[:n])
        s.T = n
        return s
    # packed or batched: keep whole sequences until n tokens are covered
    bounds = inp.seq_bounds()
    keep = 0
    for i, (a, b) in enumerate(bounds):
        keep = i + 1
        if b >= n:
            break
    end = bounds[keep - 1][1]
    for f in ("q", "k", "v", "g", "beta"):
        setattr(s, f, getattr(inp, f)[:end])
    s.B = keep
    if inp.cu_seqlens is not None:
        s.cu_seqlens = inp.cu_seqlens[:keep + 1].copy()
        s.T = end
    if inp.init is not None:
        s.init = inp.init[:keep]
    return s


def whole_job_rate(local_ms, units_per_rank, world, device=None):
    """Max-over-ranks step time (ms) and the whole-job rate: every rank's units over that time.

    Each rank runs an independent replica, so per-rank work is fixed as ranks are added
    (weak scaling) and there is no exchange step; the only collective is this MAX.
    """
    t_max = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([t_max], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t_max = float(t.item())
    return world * units_per_rank / (t_max * 1e-3), t_max


def run_gpu_arm(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from hybrid_linear_attention_prefill_gb300 import build as gbuild
    from hybrid_linear_attention_prefill_gb300 import gdn

    if rank == 0:
        gbuild.build()
    if world > 1:
        dist.barrier()
    gdn.load()

    inp = workload(args.workload, seed=args.seed + rank)  # independent candidates per replica
    d = to_device(inp, torch, dev)
    Tt, B = inp.total_tokens, inp.B
    out = torch.empty((Tt, inp.Hv, inp.dv), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((B, inp.Hv, inp.dv, inp.dk), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    flags = {"auto": None, "one": gdn.GDN_FLAG_ONE_LEVEL, "two": gdn.GDN_FLAG_TWO_LEVEL}[args.levels]

    def step():
        if flags is None:
            return gdn.gdn_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                                   B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, stream)
        return gdn.gdn_prefill_ex(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                                  B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, flags, stream)

    for _ in range(args.warmup):
        flush.zero_()
        gdn.check(step())
    torch.cuda.synchronize()

    K = args.steps
    # The two kernels' own times come from separate steps with an event between them: inside the
    # timed steps that event would stand between the state carry and the preparation kernel it is
    # launched as a programmatic dependent of, and cancel the overlap of its launch.
    KS = min(K, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KS)]
    for e3 in evs:
        for e in e3:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(KS):
        flush.zero_()
        gdn.gdn_set_phase_events(evs[i][0], evs[i][1], evs[i][2])
        gdn.check(step())
    torch.cuda.synchronize()
    prep_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(KS)]
    chain_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(KS)]

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for e2 in ev:  # create the handles before the timed region
        for e in e2:
            e.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.1)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        gdn.gdn_set_phase_events(ev[i][0], None, ev[i][1])
        gdn.check(step())
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()

    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    ms = statistics.mean(step_ms)
    rate, t_max = whole_job_rate(ms, Tt, world, dev)

    peaks = read_peaks()
    alg = algorithmic(inp)
    kernels = {"gdn_prep_kernel": statistics.mean(prep_ms), "gdn_chain_kernel": statistics.mean(chain_ms)}
    dom = max(kernels, key=kernels.get)
    dom_bytes = alg["chain"] if dom == "gdn_chain_kernel" else alg["prep"]
    achieved = dom_bytes / (kernels[dom] * 1e-3) / 1e9
    segs = gdn.gdn_scan_segments(B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, d["cu"] is not None,
                                 0 if flags is None else flags)
    trec = traffic_record(dom, args.workload) if segs == 1 else None  # the record: one single-level launch
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peaks["hbm"], "unit": "GB/s", "frac": round(achieved / peaks["hbm"], 4),
                "traffic": None if trec is None else trec["dram_bytes_per_launch"],
                "peak_source": peaks["source"]}
    if segs > 1:
        roofline["kernel"] = f"{dom} (two-level scan, {segs} segments: three launches)"
    t_hbm = alg["total"] / (peaks["hbm"] * 1e9)
    t_tc = alg["flops"] / (peaks["bf16"] * 1e12)
    path_roof = {"roofline_us": round(max(t_hbm, t_tc) * 1e6, 2), "bound": "hbm" if t_hbm >= t_tc else "tensor",
                 "frac": round(max(t_hbm, t_tc) / (t_max * 1e-3), 4),
                 "tflops": round(alg["flops"] / (t_max * 1e-3) / 1e12, 2),
                 "algorithmic_bytes": alg["total"], "algorithmic_flops": alg["flops"]}

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(inp, gdn, torch, stream, max(3, min(args.e2e_steps, K)))
        e2e["value"], _ = whole_job_rate(e2e.pop("_ms"), Tt, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_oracle(inp)

    if rank == 0:
        line = {
            "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": t_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args, inp, world),
            # bf16 inputs and outputs; the chunk products on the tensor cores take fp16 operands and
            # accumulate in fp32; the state is carried in fp32
            "arith": {"io": "bf16", "products": "fp16 x fp16 -> fp32 (tcgen05)", "state": "fp32"},
            "roofline": roofline, "path_roofline": path_roof,
            "kernels_us": {k: round(v * 1e3, 2) for k, v in kernels.items()},
            "ms_per_step_min": min(step_ms), "ms_per_step_median": statistics.median(step_ms),
            "wall_s": round(wall, 3),
            "cpu_baseline": cpu, "e2e": e2e,
            # prep + state carry (+ chunk table when packed); the two-level scan adds the
            # segment set-up, a second pass-A carry, the combine and pass C
            "gpu_launches": K * (2 + (inp.cu_seqlens is not None) if segs == 1 else 6),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_e2e(inp, gdn, torch, stream, steps):
    """The public host-buffer entry point, copies inside the timed region."""

    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        return t

    q, k, v = pinned(inp.q.view(np.int16)), pinned(inp.k.view(np.int16)), pinned(inp.v.view(np.int16))
    g, beta = pinned(inp.g), pinned(inp.beta)
    cu = None if inp.cu_seqlens is None else pinned(inp.cu_seqlens)
    init = None if inp.init is None else pinned(inp.init)
    out = torch.empty((inp.total_tokens, inp.Hv, inp.dv), dtype=torch.int16).pin_memory()
    fin = torch.empty((inp.B, inp.Hv, inp.dv, inp.dk), dtype=torch.float32).pin_memory()
    args = (q, k, v, g, beta, cu, init, out, fin, inp.B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, stream)
    for _ in range(2):
        gdn.check(gdn.gdn_prefill_host(*args))
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        gdn.check(gdn.gdn_prefill_host(*args))
        times.append(time.perf_counter() - t0)
    h2d = sum(x.numel() * x.element_size() for x in (q, k, v, g, beta, cu, init) if x is not None)
    d2h = out.numel() * 2 + fin.numel() * 4
    return {"_ms": statistics.mean(times) * 1e3, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "api": "gdn_prefill_host (pinned host buffers)"}


# ---------------------------------------------------------------------------
# measurements of the adjacent entry points (one JSON line each, device timing)
# ---------------------------------------------------------------------------
def _timed_steps(torch, stream, flush, step, warmup, K):
    """Mean, min and median milliseconds of `step` over K calls, L2 flushed before each."""
    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    return statistics.mean(ms), min(ms), statistics.median(ms)


def run_extra_arm(args):
    """--op decode | --norm-qk | --graph: the one-token step, the in-kernel q/k
    normalisation and CUDA-graph replay of the caller-workspace entry."""
    import torch

    from hybrid_linear_attention_prefill_gb300 import build as gbuild
    from hybrid_linear_attention_prefill_gb300 import gdn

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    gbuild.build()
    gdn.load()
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    peaks = read_peaks()
    sampler = ClockSampler(0)
    if args.op == "decode":
        base = WORKLOADS[args.workload]
        Hk, Hv, dk, dv, B = base["Hk"], base["Hv"], base["dk"], base["dv"], args.decode_batch
        inp = make_gdn_inputs(B=B, T=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv, seed=args.seed, init_std=0.05)
        d = to_device(inp, torch, dev)
        state = d["init"].clone()
        out = torch.empty((B, Hv, dv), dtype=torch.bfloat16, device=dev)

        def step():
            gdn.check(gdn.gdn_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], state, out,
                                     B, Hk, Hv, dk, dv, stream))

        sampler.start()
        ms, ms_min, ms_med = _timed_steps(torch, stream, flush, step, args.warmup, args.steps)
        clocks = sampler.stop()
        nbytes = 2 * B * Hv * dv * dk * 4 + B * (2 * Hk * dk + 2 * Hv * dv) * 2 + 2 * B * Hv * 4
        achieved = nbytes / (ms * 1e-3) / 1e9
        line = {"metric": "GDN decode tokens/s (one token per sequence, state updated in place)",
                "value": B / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_min": ms_min, "ms_per_step_median": ms_med,
                "higher_is_better": True,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": f"decode_b{B}_hk{Hk}_hv{Hv}", "B": B, "Hk": Hk, "Hv": Hv, "dk": dk,
                           "dv": dv, "state_bytes": B * Hv * dv * dk * 4,
                           "l2": "flushed between timed steps (256 MB write)"},
                "roofline": {"bound": "hbm", "kernel": "gdn_decode_kernel", "achieved": round(achieved, 1),
                             "peak": peaks["hbm"], "unit": "GB/s", "frac": round(achieved / peaks["hbm"], 4),
                             "traffic": None, "peak_source": peaks["source"]},
                "gpu_launches": args.steps, "clocks": clocks}
        print(json.dumps(line), flush=True)
        return
    inp = workload(args.workload, seed=args.seed)
    d = to_device(inp, torch, dev)
    Tt, B = inp.total_tokens, inp.B
    out = torch.empty((Tt, inp.Hv, inp.dv), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((B, inp.Hv, inp.dv, inp.dk), dtype=torch.float32, device=dev)
    args_common = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], d["init"], out, fin,
                   B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv)
    mode = "norm_qk" if args.norm_qk else "graph"
    if args.norm_qk:
        def step():
            gdn.check(gdn.gdn_prefill_ex(*args_common, gdn.GDN_FLAG_L2NORM_QK, stream))
    else:
        nbytes = gdn.gdn_workspace_bytes(B, inp.T, inp.Hk, inp.Hv, inp.dk, inp.dv, d["cu"] is not None)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):  # shared-memory limits set once, before capture
            gdn.check(gdn.gdn_prefill_ws(*args_common, ws, nbytes, side))
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            gdn.check(gdn.gdn_prefill_ws(*args_common, ws, nbytes, side))

        def step():
            graph.replay()
    sampler.start()
    ms, ms_min, ms_med = _timed_steps(torch, stream, flush, step, args.warmup, args.steps)
    clocks = sampler.stop()
    alg = algorithmic(inp)
    t_hbm = alg["total"] / (peaks["hbm"] * 1e9)
    line = {"metric": METRIC, "value": Tt / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_min": ms_min, "ms_per_step_median": ms_med,
                "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "mode": mode, "B": B, "T": inp.T, "Hk": inp.Hk, "Hv": inp.Hv,
                       "dk": inp.dk, "dv": inp.dv, "l2": "flushed between timed steps (256 MB write)"},
            "path_roofline": {"roofline_us": round(t_hbm * 1e6, 2), "bound": "hbm",
                              "frac": round(t_hbm / (ms * 1e-3), 4)},
            "gpu_launches": args.steps * (2 + (inp.cu_seqlens is not None)), "clocks": clocks}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    oracle.build()
    inp = workload(args.workload, seed=args.seed)
    cores = oracle.num_cpus()
    # size each step so that warmup + steps take about a minute in total
    n_cal = min(128, inp.total_tokens)
    t0 = time.perf_counter()
    oracle.prefill_inputs(slice_tokens(inp, n_cal), want_final=False, nthreads=cores)
    per_tok = max(time.perf_counter() - t0, 1e-5) / n_cal
    budget = 60.0 / max(1, args.steps + args.warmup)
    n = int(max(16, min(inp.total_tokens, budget / per_tok)))
    sub = slice_tokens(inp, n)
    for _ in range(args.warmup):
        oracle.prefill_inputs(sub, nthreads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.prefill_inputs(sub, nthreads=cores)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = sub.total_tokens / (ms * 1e-3)
    sample = (f"first {sub.total_tokens} of {inp.total_tokens} tokens, all {inp.Hv} value heads per step, "
              "float64 token loop")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, inp, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "hardware_concurrency": host_cores()[0], "nproc": host_cores()[1]},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--levels", choices=["auto", "one", "two"], default="auto",
                    help="chunk scan: the library's choice, single-level only, or two-level")
    ap.add_argument("--op", choices=["prefill", "decode"], default="prefill",
                    help="decode: time gdn_decode on --decode-batch sequences of the workload's heads")
    ap.add_argument("--decode-batch", type=int, default=128)
    ap.add_argument("--norm-qk", action="store_true", help="time gdn_prefill_ex with GDN_FLAG_L2NORM_QK")
    ap.add_argument("--graph", action="store_true", help="time gdn_prefill_ws captured into a CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference_arm(args)
    elif args.op == "decode" or args.norm_qk or args.graph:
        run_extra_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
