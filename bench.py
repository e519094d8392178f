"""Benchmark: causal GQA attention fwd+bwd TFLOP/s on one GB300 through libccg.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ccg|reference] [--workload NAME]

One step = one full pass of the CP-emulated path over the workload (for the
"large" workload: A2A pack of q/k/v/dO, CP split, the 8 ring-step forward
partials in one persistent launch, LSE merge, Delta dot, dQ pass, dV and dK passes, A2A unpack of
o/dQ/dK/dV).  Inputs are resident in HBM and far larger than L2 (no flush
needed).  Timing: W warm-up steps, then K steps between CUDA events on the
launching stream, bracketed by a barrier and synchronize, max over ranks.
Per-kernel durations come from events the library records around each of its
launches inside the same timed region.  `e2e` repeats the measurement through
the same public step API from pinned host buffers: every step's H2D of its
inputs and D2H of its outputs are in the timed region, overlapped with the
compute of the neighbouring steps (two device buffer sets, copy streams).
For the "large" workload, `d128` repeats the device-timed measurement on its
D=128 companion (same shapes and protocol, head dim 128), and `head_parts`
times the same step with the ring forward run over 4 head parts (native head
partitioning) and reports its peak device memory next to the unpartitioned
one.  `cpu_baseline`
times the FP64 oracle on a bounded sample on this host's cores.  Under torchrun (N > 1) every rank runs an independent
replica (weak scaling, no data-path collective).

--impl reference times the FP64 CPU oracle instead (one (sequence, q head)
forward+backward per step), on rank 0 only.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from context_causal_gqa_gb300 import workloads as W  # noqa: E402

METRIC = "causal attention fwd+bwd TFLOP/s on 1 GB300 and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"

# extra shapes for profiling and the D=128 companion measurement (not bench defaults)
EXTRA = {
    "ncu_small": W.custom_workload("ncu_small", [8192] * 2, 32, 8, 256, 8, index=9),
    "ncu_small_d128": W.custom_workload("ncu_small_d128", [8192] * 2, 32, 8, 128, 8, index=10),
    "ncu_small_a2a": W.custom_workload("ncu_small_a2a", [8192] * 2, 32, 8, 256, 8, index=12, pack_roundtrip=True),
    "large_d128": W.custom_workload("large_d128", [8192] * 64, 32, 8, 128, 8, index=11, pack_roundtrip=True),
}


def get_workload(name):
    return EXTRA[name] if name in EXTRA else W.WORKLOADS[name]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_burst": d["bf16_tflops"], "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "hbm": d["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ algorithmic work per kernel
def causal_pairs(w):
    return sum(s * (s + 1) / 2 for s in w.seqlens)


def merge_bytes(w):
    """Sum over rows of K_row*(2D+4) partial reads + (2D+4) write."""
    C = 2 * w.cp
    row = 2 * w.head_dim + 4
    tot = 0.0
    for S, P in zip(w.seqlens, w.padded):
        L = P // C
        for c in range(C):
            real = max(0, min(L, S - c * L))
            K = w.cp if c >= w.cp else c + 1
            tot += real * (K + 1) * row + (L - real) * row
    return tot * w.hq


def kernel_work(w):
    """name -> (bound, algorithmic amount [FLOP or byte], "step" or "launch"):
    the amount of one whole step (split evenly over the kernel's launches in
    the step: the dQ and dK passes of the backward that keeps dS run once
    per kv head) or of one launch."""
    D, hq, hkv, T = w.head_dim, w.hq, w.hkv, w.total_tokens
    U = 2.0 * D * hq * causal_pairs(w)           # one D-wide GEMM over all causal pairs
    tq = T * hq * D * 2
    tkv = T * hkv * D * 2
    work = {
        "attn_fwd": ("tensor", 2.0 * U, "step"),            # all ring-step partials (or fused)
        "pad_rows": ("hbm", 0.0, "launch"),
        "attn_bwd_dq": ("tensor", 3.0 * U, "step"),         # S, dP and dQ
        "attn_bwd_dv": ("tensor", 1.0 * U, "step"),
        "attn_bwd_dk": ("tensor", 1.0 * U, "step"),
        "attn_bwd_dkdv": ("tensor", 2.0 * U, "step"),
        "lse_merge": ("hbm", merge_bytes(w), "step"),
        "bwd_dot": ("hbm", 2.0 * tq + T * hq * 4, "step"),
        "thd_pack": ("hbm", (2 * tq + 2 * tkv) / 2.0, "launch"),      # mean over q, k, v, dO
        "thd_unpack": ("hbm", (2 * tq + 2 * tkv) / 2.0, "launch"),    # mean over o, dq, dk, dv
        "plan": ("hbm", 0.0, "launch"),
    }
    return work


def attribute_kernels(prof, work, steps, pk):
    """Per-kernel figures from (name, ms) launch records of `steps` steps:
    launches a step, time a launch, share, and the achieved rate of the
    kernel's algorithmic work a launch against the measured peak.  Returns
    (kernels, {name: [launches, total ms]})."""
    agg = {}
    for name, t in prof:
        a = agg.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += t
    tot = sum(a[1] for a in agg.values()) or 1.0
    kernels = {}
    for name, (n, t) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        bound, amount, per = work.get(name, ("hbm", 0.0, "launch"))
        avg = t / n
        if per == "step":
            amount /= n / steps                             # the step's work over its launches
        if bound == "tensor":
            ach = amount / (avg / 1e3) / 1e12
            peak = pk["bf16_sustained"]
        else:
            ach = amount / (avg / 1e3) / 1e9
            peak = pk["hbm"]
        kernels[name] = {"launches_per_step": n / steps, "ms_per_launch": round(avg, 4),
                         "share": round(t / tot, 4), "bound": bound,
                         "achieved": round(ach, 2), "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
                         "frac": round(ach / peak, 4) if peak else None}
    return kernels, agg


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[1] != self.uuid:
                    continue
                try:
                    sm.append(float(parts[2].split()[0]))
                    smax.append(float(parts[3].split()[0]))
                    power.append(float(parts[4].split()[0]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle sample
def cpu_oracle_units(w, n_units=None, budget_s=12.0, seed=0):
    """Time the FP64 oracle's forward+backward of whole (sequence, q head)
    pairs of the workload on this host.  Returns (flops, seconds, units)."""
    import numpy as np
    import torch
    import oracle
    S = max(w.seqlens)
    D = w.head_dim
    g = torch.Generator().manual_seed(w.seed + 17 + seed)
    flops = 0.0
    units = 0
    t0 = time.perf_counter()
    while True:
        q, k, v, do = (torch.randn(S, D, generator=g).to(torch.bfloat16).double().numpy() for _ in range(4))
        oracle.head_backward(q, k, v, do)
        flops += 3.5 * 4.0 * D * S * (S + 1) / 2
        units += 1
        el = time.perf_counter() - t0
        if (n_units is not None and units >= n_units) or (n_units is None and el >= budget_s):
            break
    del np
    return flops, time.perf_counter() - t0, units


def host_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max((i.get("num_threads", 1) for i in info if i.get("user_api") == "blas"), default=None)
        if n:
            return int(n)
    except Exception:
        pass
    return os.cpu_count()


# ------------------------------------------------------------------ multi-rank aggregation
def reduce_max(pg, v, device="cpu"):
    """Max over ranks of a scalar (identity without a process group)."""
    if pg is None:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step, world, ms_max):
    """Whole-job TFLOP/s: every rank processes its own replica of the
    workload (weak scaling), timed by the slowest rank."""
    return world * flops_per_rank_step / (ms_max / 1e3) / 1e12


# ------------------------------------------------------------------ arms
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return rank, local, world, pg


def bench_config(w, args, world):
    """The `config` object of the JSON line; the same for both arms."""
    cfg = dict(w.describe())
    cfg["workload"] = (f"{w.name}: B={w.batch} x S={max(w.seqlens)} packed THD, Hq{w.hq}/Hkv{w.hkv}, "
                       f"D{w.head_dim}, causal, {w.cp} emulated CP ranks ({2 * w.cp} chunks)"
                       + (", A2A head-split pack/unpack round trip" if w.pack_roundtrip else ""))
    cfg["l2"] = "inputs larger than L2, no flush"
    cfg["schedule"] = args.schedule
    fused = args.fwd == "fused" or args.schedule == "a2a"
    cfg["forward"] = "fused online softmax" if fused else "ring-step partials + LSE merge"
    cfg["backward"] = ("dQ pass keeps dS (and P at D=256), dK/dV passes read them back"
                       if getattr(args, "bwd", "") == "keep-ds"
                       else "dK pass recomputes S^T and dP^T")
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "1 GPU, CP emulated"
    return cfg


def run_reference(args):
    rank, _, world, pg = dist_setup(args.gpus)
    if rank != 0:
        return 0
    w = get_workload(args.workload)
    for _ in range(args.warmup):
        cpu_oracle_units(w, n_units=1, seed=99)
    times, fl = [], 0.0
    for k in range(args.steps):
        f, t, _ = cpu_oracle_units(w, n_units=1, seed=k)
        times.append(t)
        fl = f
    ms = 1e3 * sum(times) / len(times)
    value = fl / (ms / 1e3) / 1e12
    sample = f"one (sequence, q head) forward+backward at S={max(w.seqlens)}, D={w.head_dim} per step (FP64 numpy oracle)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, args, world),
            "cpu_baseline": {"kind": "oracle", "cores": host_threads(), "sample": sample, "value": value,
                             "unit": UNIT},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def measure(w, args, dev, pg, world, rank, clocks_uuid=None, head_parts=0):
    """Device-timed steps of workload `w`: W warm-up steps, then K steps
    between CUDA events on the launching stream, barrier + synchronize on
    both sides, max over ranks; per-kernel events from the library.
    Returns (step, result dict)."""
    import torch
    from context_causal_gqa_gb300.pipeline import AttentionStep, profile_begin, profile_end
    x = W.make_inputs(w, device=dev, seed=w.seed + 1000 * rank)
    step = AttentionStep(w, x, device=dev, schedule=args.schedule, fused=args.fwd == "fused", head_parts=head_parts,
                         keep_ds=args.bwd == "keep-ds")
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize(dev)
    step.check()

    def barrier():
        if pg is not None:
            pg.barrier()

    clocks = ClockSampler(clocks_uuid)
    per_step = step.launches_per_step
    profile_begin(per_step * args.steps + 8)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    # one event between consecutive steps: the whole region and each step
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    e0, e1 = marks[0], marks[-1]
    e0.record(stream)
    launches = 0
    for i in range(args.steps):
        launches += step.run()
        marks[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier()
    prof = profile_end()
    step.check()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = reduce_max(pg, ms, dev)
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    flops = w.flops_fwd_bwd()
    value = job_throughput(flops, world, ms_max)

    # per-kernel attribution inside the timed region
    pk = peaks()
    kernels, agg = attribute_kernels(prof, kernel_work(w), args.steps, pk)
    dom = max(agg.items(), key=lambda kv: kv[1][1])[0]
    dk = kernels[dom]
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            tr = json.load(f)
        ent = tr.get(w.name, {}).get(dom)
        if ent and ent.get("source_sha") == source_sha(dom):
            traffic = ent["bytes_per_launch"]
    roofline = {"bound": dk["bound"], "achieved": dk["achieved"],
                "peak": pk["bf16_sustained"] if dk["bound"] == "tensor" else pk["hbm"],
                "unit": dk["unit"], "frac": dk["frac"], "traffic": traffic, "kernel": dom,
                "peak_source": pk["source"] + (" bf16 sustained (kernel timed inside a long step)"
                                               if dk["bound"] == "tensor" else " hbm copy")}
    res = {"value": round(value, 2), "ms_per_step": round(ms_max, 3), "flops": flops,
           "frac_of_peak": round(value / world / pk["bf16_sustained"], 4), "peak_tflops": pk["bf16_sustained"],
           "roofline": roofline, "kernels": kernels, "clocks": clk, "gpu_launches": launches,
           "step_ms": {"median": round(statistics.median(step_ms), 3), "min": round(min(step_ms), 3),
                       "max": round(max(step_ms), 3)}}
    return step, x, res


def run_ccg(args):
    import torch
    rank, local, world, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import context_causal_gqa_gb300 as ccg
    ccg.load()
    w = get_workload(args.workload)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    stream = torch.cuda.current_stream(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    step, x, res = measure(w, args, dev, pg, world, rank, uuid)
    peak_timed = round(torch.cuda.max_memory_allocated(dev) / 1e9, 2)
    flops = res["flops"]

    def barrier():
        if pg is not None:
            pg.barrier()

    # end to end from pinned host buffers through the same step API: every
    # step copies its inputs in and its outputs out; the copies of one step
    # overlap the compute of its neighbours (two device buffer sets)
    e2e = None
    if not args.no_e2e:
        h_in, h_out = step.host_buffers()
        for d, h in zip(step.input_tensors(), h_in):
            h.copy_(d)
        bi, bo = step.io_bytes()
        s0, s1 = step.run_from_host_pipelined(h_in, h_out, 2, stream=stream)   # warm-up
        torch.cuda.synchronize(dev)
        ke = max(3, min(args.steps, 10))
        barrier()
        s0, s1 = step.run_from_host_pipelined(h_in, h_out, ke, stream=stream)
        torch.cuda.synchronize(dev)
        barrier()
        step.check()
        ms_e2e = reduce_max(pg, s0.elapsed_time(s1) / ke, dev)
        e2e = {"value": job_throughput(flops, world, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": ms_e2e, "steps": ke,
               "copies": "H2D of step i+1 and D2H of step i-1 overlap the compute of step i"}
        del h_in, h_out
    peak_mem = round(torch.cuda.max_memory_allocated(dev) / 1e9, 2)
    del step, x
    torch.cuda.empty_cache()

    # native head partitioning of the ring forward: the same step with the
    # partials and merge run over 4 head parts in turn (workspace for Hq/4)
    head_parts = None
    if args.workload == "large" and not args.no_head_parts and args.fwd == "partials" and args.schedule == "ring":
        torch.cuda.reset_peak_memory_stats(dev)
        sp, xp, rp = measure(w, args, dev, pg, world, rank, uuid, head_parts=4)
        head_parts = {"parts": 4, "value": rp["value"], "ms_per_step": rp["ms_per_step"],
                      "peak_mem_gb": round(torch.cuda.max_memory_allocated(dev) / 1e9, 2),
                      "peak_mem_gb_parts1": peak_timed,
                      "attn_fwd_ms": rp["kernels"].get("attn_fwd", {}).get("ms_per_launch"),
                      "lse_merge_ms": rp["kernels"].get("lse_merge", {}).get("ms_per_launch")}
        del sp, xp
        torch.cuda.empty_cache()

    # the D=128 companion of the large workload, same protocol (device-timed)
    d128 = None
    if args.workload == "large" and not args.no_d128:
        wd = get_workload("large_d128")
        sd, xd, rd = measure(wd, args, dev, pg, world, rank, uuid)
        del sd, xd
        torch.cuda.empty_cache()
        d128 = {"workload": bench_config(wd, args, world)["workload"], "value": rd["value"], "unit": UNIT,
                "ms_per_step": rd["ms_per_step"], "frac_of_peak": rd["frac_of_peak"], "roofline": rd["roofline"],
                "kernels": rd["kernels"], "clocks": rd["clocks"], "step_ms": rd["step_ms"],
                "gpu_launches": rd["gpu_launches"]}

    cpu = None
    if rank == 0 and not args.no_cpu:
        f, t, u = cpu_oracle_units(w, budget_s=args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": host_threads(), "kind": "oracle",
               "sample": f"{u} x one (sequence, q head) forward+backward at S={max(w.seqlens)}, D={w.head_dim} "
                         f"(FP64 numpy oracle, {t:.1f} s)"}

    if rank == 0:
        cfg = bench_config(w, args, world)
        line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": cfg, "frac_of_peak": res["frac_of_peak"],
                "peak_tflops": res["peak_tflops"], "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "kernels": res["kernels"],
                "step_ms": res["step_ms"], "peak_mem_gb": peak_mem, "peak_mem_gb_device_timed": peak_timed,
                "head_parts": head_parts, "d128": d128}
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()
    return 0


def source_sha(kernel):
    import hashlib
    files = {"attn_fwd": "attn_fwd.cu", "lse_merge": "elementwise.cu", "bwd_dot": "elementwise.cu",
             "thd_pack": "elementwise.cu", "thd_unpack": "elementwise.cu"}
    f = files.get(kernel, "attn_bwd.cu")
    with open(os.path.join(ROOT, "context_causal_gqa_gb300", "csrc", f), "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ccg", choices=["ccg", "reference"])
    ap.add_argument("--workload", default="large", choices=list(W.WORKLOADS) + list(EXTRA))
    ap.add_argument("--schedule", default="ring", choices=["ring", "a2a"],
                    help="ring: CP-emulated ring (the measured path); a2a: A2A head-split schedule")
    ap.add_argument("--fwd", default="partials", choices=["partials", "fused"],
                    help="partials: ring-step partials + LSE merge (the measured path); fused: one online softmax")
    ap.add_argument("--bwd", default="keep-ds", choices=["keep-ds", "recompute"],
                    help="keep-ds (the measured path): the backward keeps dS, and at D=256 P (the dQ pass writes "
                         "them, the dK/dV passes read them back); recompute: the dK/dV passes recompute S^T and dP^T")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-d128", action="store_true", help="skip the D=128 companion measurement")
    ap.add_argument("--no-head-parts", action="store_true", help="skip the 4-head-part forward measurement")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ccg":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ccg(args)


if __name__ == "__main__":
    sys.exit(main())
