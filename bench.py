"""Benchmark of the GB300 chunked gated delta rule backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step is one full backward (every kernel of the path) over one problem of the workload, with the
inputs resident in HBM.  The default workload is the T=32768, H=16, K=V=128 bf16 one.  Under torchrun
(N > 1) every rank runs its own problem (independent replicas, no collective on the data path:
weak scaling); timing is bracketed by a barrier and a device synchronise and the max over ranks is
reported.  Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on the host cores instead (bounded samples of the same
workload); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN chunked bwd ms & TFLOP/s (T=32k,H=16,K=V=128,bf16), % of roofline"
UNIT = "TFLOP/s"
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
L2_BYTES = 129 * 2 ** 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="gdn_t32k_bf16")
    ap.add_argument("--cpu-sample-tokens", type=int, default=32768)
    ap.add_argument("--flush-steps", type=int, default=20,
                    help="calls timed one by one with a 512 MB write between them (L2 flushed)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", choices=("bwd", "fwd", "wy"), default="bwd",
                    help="bwd: the backward (the headline); fwd: the forward pass (o and the final state); "
                         "wy: the WY-gradient stage taken alone at its own model shape (T=2048, H=32, fp16)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (identity at world size 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(gpu_index)], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons, n = [], [], set(), 0
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(REASONS, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------- peaks and profiles
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summaries, or None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    pat = re.compile(rf"^traffic_bytes_per_launch:\s*{re.escape(kernel)}\s+{re.escape(workload)}\s*=\s*([0-9.eE+]+)")
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for line in f:
                m = pat.match(line.strip())
                if m:
                    return float(m.group(1))
    return None


def workload_config(prob, world):
    return {"workload": prob.name, "B": prob.B, "T": prob.T, "Hk": prob.Hk, "Hv": prob.Hv, "K": prob.K,
            "V": prob.V, "BT": prob.BT, "num_seqs": prob.num_seqs, "gate": "per-channel" if prob.per_channel else "scalar",
            "inputs": f"{str(prob.qkv_dtype).split('.')[-1]} q/k/v/dO, {str(prob.beta_dtype).split('.')[-1]} beta, "
                      f"fp32 g, fp32 h0/dht" + ("" if prob.h0 is not None else " (h0 absent)"),
            "problems_per_rank": 1, "global_batch": world, "parallelism": f"replicas x{world} (no collective)",
            "l2": "inputs + workspace larger than L2 (129 MB); value: no flush between steps; l2_flushed: a "
                  "512 MB write between calls"}


# ---------------------------------------------------------------- oracle timing (CPU baseline / reference arm)
def cpu_sample(prob_name, tokens, heads):
    from chunked_gated_delta_09_gb300.inputs import make_problem, workload
    full_shapes = {
        "gdn_t32k_bf16": dict(Hk=16, Hv=16, K=128, V=128),
        "gdn_t8k_bf16": dict(Hk=16, Hv=16, K=128, V=128),
    }
    if prob_name in full_shapes:
        sh = full_shapes[prob_name]
        G = sh["Hv"] // sh["Hk"]
        hk = max(1, min(sh["Hk"], heads // G))
        T = min(tokens, 32768 if prob_name == "gdn_t32k_bf16" else 8192)  # never more than the workload itself
        return make_problem(prob_name + "_cpu_sample", B=1, T=T, Hk=hk, Hv=hk * G, K=sh["K"], V=sh["V"],
                            BT=64, qkv_dtype=__import__("torch").bfloat16, seed=4242)
    return workload(prob_name)


def time_oracle(prob):
    import oracle
    from chunked_gated_delta_09_gb300 import counts
    a = prob.packed_f64()
    t0 = time.perf_counter()
    oracle.backward(a["cu"], prob.Hk, prob.Hv, prob.K, prob.V, prob.per_channel, prob.scale, a["q"], a["k"], a["v"],
                    a["beta"], a["g"], a["h0"], a["dO"], a["dht"])
    dt = time.perf_counter() - t0
    units = prob.N * prob.Hv
    cores = min(units, oracle.max_threads())
    return dt, counts.total_flops(prob), cores


def cpu_baseline(args):
    import oracle  # noqa: F401  (builds on first use)
    nthr = __import__("oracle").max_threads()
    sample = cpu_sample(args.workload, args.cpu_sample_tokens, min(16, nthr))
    dt, fl, cores = time_oracle(sample)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": dt,
            "sample": f"fp64 C oracle (token recurrence + adjoints), {sample.T} tokens x {sample.Hv} heads of the "
                      f"{args.workload} recipe; FLOPs counted with the chunked-algorithm convention"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    nthr = oracle.max_threads()
    tokens = 8192
    sample = cpu_sample(args.workload, tokens, min(16, nthr))
    for _ in range(args.warmup):
        time_oracle(sample)
    times = []
    for _ in range(args.steps):
        dt, fl, cores = time_oracle(sample)
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = fl / (ms / 1e3) / 1e12
    desc = (f"fp64 C oracle, {sample.T} tokens x {sample.Hv} heads of the {args.workload} recipe per step; "
            f"FLOPs counted with the chunked-algorithm convention")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our path
def run_ours(args):
    import torch
    from chunked_gated_delta_09_gb300 import _lib, counts, ops
    from chunked_gated_delta_09_gb300.build import build
    from chunked_gated_delta_09_gb300.inputs import workload

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    if rank == 0:
        build()
    barrier(world)
    build()

    if args.which == "wy":
        return run_wy_bench(args, world, rank, local)
    prob = workload(args.workload)
    if args.which == "fwd":
        return run_forward_bench(args, prob, world, rank, local)
    plan = ops.plan_for(prob)
    dev = ops.problem_to_device(prob, "cuda")
    out = plan.alloc_outputs("cuda")
    ws = plan.alloc_workspace("cuda")
    stream = torch.cuda.current_stream()
    nst = _lib.NUM_STAGES

    for _ in range(max(args.warmup, 3)):
        plan.run(out=out, workspace=ws, **dev)
    torch.cuda.synchronize()
    st = plan.get_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    # ---- timed region: inputs resident in HBM, per-stage events on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(args.steps)]
    for row in evs:
        for e in row:
            e.record(stream)  # materialise the handles before timing
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    wall0 = time.perf_counter()
    t0.record(stream)
    for i in range(args.steps):
        plan.run_profiled(evs[i], out=out, workspace=ws, **dev)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    ms_local = t0.elapsed_time(t1) / args.steps
    stage_ms = [statistics.mean(evs[i][s].elapsed_time(evs[i][s + 1]) for i in range(args.steps)) for s in range(nst)]
    step_ms = [evs[i][0].elapsed_time(evs[i][nst]) for i in range(args.steps)]

    # ---- the same call timed one at a time with L2 flushed before each (a 512 MB write on the stream)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    fl_ms = []
    for _ in range(max(args.flush_steps, 1)):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plan.run(out=out, workspace=ws, **dev)
        b.record(stream)
        b.synchronize()
        fl_ms.append(a.elapsed_time(b))
    del flush

    # ---- end to end through the C ABI with host buffers (pinned).  Every step copies its inputs in and its
    # results out inside the timed region; the copies run on their own streams so that step i+1's inputs and
    # step i-1's results move while step i computes (two device buffer sets, event-ordered).
    host_in = {k: (None if v is None else v.cpu().pin_memory()) for k, v in dev.items()}
    host_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()} for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values() if v is not None)
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
    dev_in = [dev, {k: (None if v is None else torch.empty_like(v)) for k, v in dev.items()}]
    dev_out = [out, plan.alloc_outputs("cuda")]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(nsteps):
        h2d_done, comp_done, d2h_done = {}, {}, {}
        for i in range(nsteps):
            b = i % 2
            with torch.cuda.stream(s_in):  # inputs of step i, once step i-2 no longer reads this buffer set
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])
                for k, v in host_in.items():
                    if v is not None:
                        dev_in[b][k].copy_(v, non_blocking=True)
                h2d_done[i] = torch.cuda.Event()
                h2d_done[i].record(s_in)
            stream.wait_event(h2d_done[i])
            if i >= 2:
                stream.wait_event(d2h_done[i - 2])  # step i-2's results are out of this buffer set
            plan.run(out=dev_out[b], workspace=ws, stream=stream, **dev_in[b])
            comp_done[i] = torch.cuda.Event()
            comp_done[i].record(stream)
            with torch.cuda.stream(s_out):  # results of step i
                s_out.wait_event(comp_done[i])
                for k, v in dev_out[b].items():
                    host_out[b][k].copy_(v, non_blocking=True)
                d2h_done[i] = torch.cuda.Event()
                d2h_done[i].record(s_out)

    e2e_run(max(args.warmup, 3))
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_run(args.steps)
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    e2e_local = e0.elapsed_time(e1) / args.steps
    st = plan.get_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after timing")

    ms = max_over_ranks(ms_local, world)
    e2e_ms = max_over_ranks(e2e_local, world)
    flops = counts.total_flops(prob)
    value = world * flops / (ms / 1e3) / 1e12
    if rank != 0:
        return

    peaks = measured_peaks()
    alg_bytes = counts.algorithmic_bytes(prob)
    t_roof = max(flops / (peaks["bf16_tflops"] * 1e12), alg_bytes / (peaks["hbm_gbs"] * 1e9))
    stage_flops = counts.stage_flops(prob)
    stage_bytes = counts.stage_bytes(prob)
    tc_peak, bw_peak = peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9
    step_med = statistics.median(step_ms)
    flushed_med = statistics.median(fl_ms)

    def stage_roof(s):
        """Roofline of one stage: the tensor or HBM bound, whichever is longer for its FLOPs and bytes."""
        t = stage_ms[s] / 1e3
        if stage_bytes[s] / bw_peak >= stage_flops[s] / tc_peak:
            ach = stage_bytes[s] / t / 1e9
            return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / peaks["hbm_gbs"]}
        ach = stage_flops[s] / t / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"]}

    dom = max(range(nst), key=lambda s: stage_ms[s])
    dom_name = _lib.STAGE_NAMES[dom]
    # the dominant kernel against the least it must move (its algorithmic bytes) or compute, whichever
    # bound is longer; the design's own stage bytes and the ncu-measured DRAM bytes stand beside it
    t_dom = stage_ms[dom] / 1e3
    dom_alg = counts.gradient_stage_algorithmic_bytes(prob) if dom_name == "k4_intra_grad" else stage_bytes[dom]
    if dom_alg / bw_peak >= stage_flops[dom] / tc_peak:
        dom_roof = {"bound": "hbm", "achieved": dom_alg / t_dom / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": dom_alg / t_dom / bw_peak}
    else:
        dom_roof = {"bound": "tensor", "achieved": stage_flops[dom] / t_dom / 1e12, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": stage_flops[dom] / t_dom / tc_peak}
    traffic = committed_traffic(dom_name, prob.name)
    roof = {"kernel": dom_name, **dom_roof,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": dom_alg, "stage_bytes_per_launch": stage_bytes[dom],
            "flops_per_launch": stage_flops[dom],
            "tensor_frac": stage_flops[dom] / t_dom / tc_peak,
            "wasted_traffic_ratio": (traffic / dom_alg) if traffic else None,
            "ms_per_launch": stage_ms[dom],
            "peak_source": f"{peaks['source']} (HBM copy GB/s; dense bf16 burst TFLOP/s, fp16 operands run at "
                           f"the bf16 rate)"}
    stage_roofs = {_lib.STAGE_NAMES[s]: {k: v for k, v in stage_roof(s).items() if k in ("bound", "achieved", "frac")}
                   for s in range(nst) if stage_ms[s] > 0 and (stage_bytes[s] > 0 or stage_flops[s] > 0)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "data": "synthetic",
        "config": workload_config(prob, world),
        "backward_roofline_frac": t_roof / (ms / 1e3),
        "median_ms_per_step": step_med,
        "l2_flushed": {"median_ms": flushed_med, "calls": len(fl_ms), "flush_bytes": 512 * 2 ** 20,
                       "backward_roofline_frac": t_roof / (flushed_med / 1e3)},
        "roofline": roof,
        "path_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms / 1e3), "flops": flops,
                          "algorithmic_bytes": alg_bytes,
                          "tensor_frac": (flops / (ms / 1e3)) / (peaks["bf16_tflops"] * 1e12),
                          "hbm_frac": (alg_bytes / (ms / 1e3)) / (peaks["hbm_gbs"] * 1e9)},
        "stage_ms": {_lib.STAGE_NAMES[s]: stage_ms[s] for s in range(nst)},
        "stage_roofline": stage_roofs,
        "e2e": {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": plan.launch_count * args.steps,
        "clocks": clk,
        "timed_wall_s": wall,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line), flush=True)


def run_forward_bench(args, prob, world, rank, local):
    """The forward pass (gdr_fwd_run) on the same workload: device time with CUDA events, whole-path
    roofline by the forward FLOP / byte conventions of counts.py."""
    import torch
    from chunked_gated_delta_09_gb300 import counts, ops

    plan = ops.plan_for(prob)
    dev = ops.problem_to_device(prob, "cuda")
    fin = {k: dev[k] for k in ("q", "k", "v", "beta", "g", "h0", "cu_seqlens")}
    out = plan.alloc_forward_outputs("cuda")
    ws = plan.alloc_workspace("cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        plan.run_forward(out=out, workspace=ws, **fin)
    torch.cuda.synchronize()
    if plan.get_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    t0.record(stream)
    for _ in range(args.steps):
        plan.run_forward(out=out, workspace=ws, **fin)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)
    if plan.get_status(ws) != 0:
        raise RuntimeError("device status after timing")
    if rank != 0:
        return
    peaks = measured_peaks()
    flops = counts.forward_total_flops(prob)
    alg = counts.forward_algorithmic_bytes(prob)
    t_roof = max(flops / (peaks["bf16_tflops"] * 1e12), alg / (peaks["hbm_gbs"] * 1e9))
    line = {"metric": "GDN chunked fwd ms & TFLOP/s (o and final state), % of roofline",
            "value": world * flops / (ms / 1e3) / 1e12, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "data": "synthetic", "pass": "fwd",
            "config": workload_config(prob, world),
            "path_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms / 1e3), "flops": flops,
                              "algorithmic_bytes": alg},
            "gpu_launches": plan.forward_launch_count * args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


def run_wy_bench(args, world, rank, local):
    """The WY-gradient stage taken alone (gdr_wy_bwd_run) on the shape its page names: B=1, T=2048, H=32,
    K=V=128, BT=64, fp16, inputs drawn like its usage example (cumulative gate, A a true inverse)."""
    import torch
    from chunked_gated_delta_09_gb300 import counts, ops

    B, T, H, K, V, BT = 1, 2048, 32, 128, 128, 64
    gen = torch.Generator().manual_seed(2024)
    rn = lambda *s_: torch.randn(*s_, generator=gen)
    dt = torch.float16
    q, k, v, v_new, do, dv = (rn(B, T, H, s_).to(dt).cuda() for s_ in (K, K, V, V, V, V))
    beta = torch.sigmoid(rn(B, T, H)).to(dt).cuda()
    g = torch.nn.functional.logsigmoid(rn(B, T // BT, BT, H, K)).cumsum(2).reshape(B, T, H, K).cuda()
    Akk = torch.tril(0.2 * rn(B * T // BT, H, BT, BT), -1)
    A = torch.linalg.inv(torch.eye(BT) + Akk).permute(0, 2, 1, 3).reshape(B, T, H, BT).to(dt).cuda()
    h, dh = rn(B, T // BT, H, K, V).cuda(), rn(B, T // BT, H, K, V).cuda()
    call = lambda: ops.gdr_wy_bwd(q, k, v, v_new, g, beta, A, h, do, dh, dv, scale=K ** -0.5, chunk_size=BT)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    t0.record(stream)
    for _ in range(args.steps):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)
    if rank != 0:
        return
    peaks = measured_peaks()
    flops = B * (T // BT) * H * counts.wy_stage_flops_per_chunk(BT, K, V)
    alg = counts.wy_stage_bytes(B, T, H, K, V, BT, 2)
    t_roof = max(flops / (peaks["bf16_tflops"] * 1e12), alg / (peaks["hbm_gbs"] * 1e9))
    line = {"metric": "KDA WY-gradient stage alone (chunk_kda_bwd_wy_dqkg_fused) ms, % of roofline",
            "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "accumulate": "f32", "data": "synthetic", "pass": "wy",
            "config": {"workload": "kda_wy_t2k_h32_fp16", "B": B, "T": T, "H": H, "K": K, "V": V, "BT": BT,
                       "timing": "includes the host-side plan creation and output allocation of each call"},
            "path_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms / 1e3), "flops": flops,
                              "algorithmic_bytes": alg, "achieved_gbs": alg / (ms / 1e3) / 1e9},
            "clocks": clk}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    world = dist_env()[0]
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
