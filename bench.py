"""Benchmark of the GB300 Muon optimizer step.

One "step" is one full Muon step (momentum + Nesterov, Frobenius
normalisation, 5 Newton-Schulz iterations, weight update) over one rank's
share of one MoE layer: 96 experts x {gate 2048x6144, up 2048x6144, down
6144x2048} = 288 bf16 weight matrices with fp32 momentum -- whole experts on
one rank as in the FlexShard bullet of "How PyTorch Scaled a Near-1T MoE on
Europe's Public Supercomputer" ("Three optimizations that changed the
economics").  Inputs are synthetic (seeded), drawn by
muon_newton_schulz_step_gb300.workloads.

Metric: nominal Newton-Schulz TFLOP/s of the whole step, counting
5 * (4 r^2 k + 2 r^3) FLOPs per matrix (r = min, k = max), plus matrices/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
288-matrix layer (whole matrices partitioned across ranks, no data-path
collective: weak scaling); the time is the max over ranks.
"""
import argparse
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

WORKLOAD = "moe_layer"
METRIC = "Muon NS5 TFLOP/s and matrices/s on 1 GB300; % of bf16 dense tensor-core peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            v = d.get(key)
            if isinstance(v, dict):
                v = v.get("value")
            out[key] = float(v)
        return out, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in self.rows for j in range(4) if r[4 + j].lower() == "active"})
        pw = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "power_w_median": statistics.median(pw) if pw else None,
                "samples": len(self.rows)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _nominal_flops(w):
    from muon_newton_schulz_step_gb300 import workloads as wl
    return sum(wl.nominal_ns_flops(s.rows, s.cols) for s in w.mats)


def _executed_flops(w, steps=5, tile=256):
    """FLOPs the default (pair-CTA, 256 x 256 tile) GEMM kernel executes for the
    workload: symmetric products run only tiles with tm <= tn over the zero-padded
    iterate; the update runs every tile."""
    tot = 0.0
    for s in w.mats:
        r, k = min(s.rows, s.cols), max(s.rows, s.cols)
        rp, kp = -(-r // tile) * tile, -(-k // tile) * tile
        nt = rp // tile
        sym = nt * (nt + 1) // 2 * tile * tile
        tot += steps * (2.0 * sym * kp + 2.0 * sym * rp + 2.0 * rp * kp * rp)
    return tot


def gemm_source_digest():
    """sha256 over the sources that define the dominant kernel: the pair-CTA
    GEMM, the PTX wrappers and the GEMM parameter block of internal.h."""
    import hashlib
    csrc = os.path.join(ROOT, "muon_newton_schulz_step_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("ns_gemm_pair.cu", "ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(csrc, "internal.h")) as f:
        text = f.read()
    a = text.index("// ------------------------------------------------------------------- GEMM --")
    b = text.index("// ------------------------------------------------------------ small path --")
    h.update(text[a:b].encode())
    return h.hexdigest()


def _traffic_record():
    """Per-launch DRAM bytes of the GEMM kernel from a committed ncu capture,
    or None if the kernel's sources have changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "ns_gemm_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_sha256") != gemm_source_digest():
        return None
    return rec


def measure_adamw(mg, torch, dev, steps: int, peaks, big: int = 256000 * 6144):
    """AdamW (the optimizer for the parameters Muon does not cover) on an
    embedding-sized parameter of the pages' model (vocabulary 256,000 x hidden
    6,144, bf16) plus 148 norm vectors of 6,144: HBM-bound, 22 bytes per element
    (P 2+2, G 2, M 4+4, V 4+4)."""
    gen = torch.Generator(device=dev).manual_seed(7)
    sizes = [big] + [6144] * 148
    P = [(0.02 * torch.randn(n, generator=gen, device=dev)).to(torch.bfloat16) for n in sizes]
    G = [(1e-3 * torch.randn(n, generator=gen, device=dev)).to(torch.bfloat16) for n in sizes]
    M = [torch.zeros(n, device=dev) for n in sizes]
    V = [torch.zeros(n, device=dev) for n in sizes]
    for t in range(1, 4):
        mg.muon_adamw_step(P, G, M, V, lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=t)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(4, 4 + steps):
        mg.muon_adamw_step(P, G, M, V, lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, step=t)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    n = sum(sizes)
    gbs = n * 22.0 / (ms * 1e-3) / 1e9
    out = {"workload": f"{big}-element bf16 parameter + 148 x 6144 (bf16 P and G, fp32 M and V)",
           "elements": n, "ms_per_step": ms, "gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
           "bytes_per_element": 22}
    del P, G, M, V
    torch.cuda.empty_cache()
    return out


def measure_all_configs(mg, wl, torch, dev, steps: int = 5, warmup: int = 2):
    """Step time of every workload (the bench value is moe_layer's): per
    workload ms, nominal Newton-Schulz TFLOP/s and matrices/s."""
    out = {}
    for name in wl.WORKLOADS:
        w = wl.workload(name)
        inp = wl.make_inputs(w, dev)
        if w.call == "ns":
            def step():
                mg.muon_ns5_batched(inp["G"])
        else:
            batch = mg.MuonStepBatch(inp["W"], inp["G"], inp["M"])

            def step():
                batch.step(w.lr, w.mu, w.wd)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        flops = sum(wl.nominal_ns_flops(m.rows, m.cols) for m in w.mats)
        out[name] = {"call": "muon_ns5_batched" if w.call == "ns" else "muon_step_ex", "matrices": w.count,
                     "ms": ms, "nominal_tflops": flops / (ms * 1e-3) / 1e12,
                     "matrices_per_s": w.count / (ms * 1e-3)}
        del inp
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------- our arm ---
def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import muon_newton_schulz_step_gb300 as mg
    from muon_newton_schulz_step_gb300 import workloads as wl

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    if args.only_adamw:
        peaks, _ = _peaks()
        out = measure_adamw(mg, torch, dev, args.steps, peaks, args.adamw_elems)
        if rank == 0:
            print(json.dumps({"adamw_only": out}), flush=True)
        return
    w = wl.workload(args.workload)
    if args.max_matrices:
        w.mats = w.mats[:args.max_matrices]   # profiling of a small case only
    inp = wl.make_inputs(w, dev)
    torch.cuda.synchronize()
    batch = mg.MuonStepBatch(inp["W"], inp["G"], inp["M"])
    stream = torch.cuda.current_stream()
    flops = _nominal_flops(w)

    for _ in range(args.warmup):
        batch.step(w.lr, w.mu, w.wd)
    torch.cuda.synchronize()
    if mg.muon_device_status() != 0:
        raise RuntimeError("device status after warm-up is not OK")

    def timed_region():
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        mg.muon_profile_enable(True)
        barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            batch.step(w.lr, w.mu, w.wd)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        prof_ = mg.muon_profile_read()
        mg.muon_profile_enable(False)
        return ev0.elapsed_time(ev1), prof_, sampler.stop()

    # a region whose clock samples show a hardware or thermal slowdown, or SM
    # clocks far below their maximum with no reason given, is measured once more
    ms, prof, clocks = timed_region()
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    stuck = (clocks.get("sm_mhz") and clocks.get("sm_max_mhz") and not clocks.get("reasons")
             and clocks["sm_mhz"] < 0.6 * clocks["sm_max_mhz"])
    flag = torch.tensor([1.0 if (bad & set(clocks.get("reasons") or [])) or stuck else 0.0], device=dev)
    if world > 1:
        dist.all_reduce(flag, op=dist.ReduceOp.MAX)
    if float(flag.item()) > 0:
        first = clocks
        ms, prof, clocks = timed_region()
        clocks["remeasured_after"] = first
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_per_step = ms / args.steps
    total_flops = flops * world
    value = total_flops / (ms_per_step * 1e-3) / 1e12
    mats_per_s = w.count * world / (ms_per_step * 1e-3)
    if mg.muon_device_status() != 0:
        raise RuntimeError("device status after the timed steps is not OK")

    # ---- end to end through the public API with host (pinned) buffers
    e2e = None
    pinned = None
    if not args.no_e2e:
        try:
            pinned = ([t.cpu().pin_memory() for t in inp["W"]], [t.cpu().pin_memory() for t in inp["G"]],
                      [t.cpu().pin_memory() for t in inp["M"]])
        except RuntimeError as exc:   # host memory exhausted (several ranks on one node)
            e2e = {"value": None, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                   "note": f"not measured: pinning the host copies failed ({str(exc)[:120]})"}
    if not args.no_e2e and world > 1:
        # every rank must take part in the e2e timing (it has barriers): agree first
        ok = torch.tensor([1 if pinned is not None else 0], device=dev)
        dist.all_reduce(ok, op=dist.ReduceOp.MIN)
        if int(ok.item()) == 0 and pinned is not None:
            pinned = None
            e2e = {"value": None, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                   "note": "not measured: another rank could not pin its host copies"}
    if pinned is not None:
        hW, hG, hM = pinned
        h2d = sum(t.numel() * t.element_size() for t in hW + hG + hM)
        d2h = sum(t.numel() * t.element_size() for t in hW + hM)

        host_batch = mg.MuonHostStep(hW, hG, hM)

        def e2e_step():
            # W, G, M in pinned host memory: copied in, stepped and copied out in
            # overlapped chunks by the library's host-buffer entry point
            host_batch.step(w.lr, w.mu, w.wd)

        e2e_step()
        torch.cuda.synchronize()
        k2 = max(1, min(args.steps, args.e2e_steps))
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k2):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = e0.elapsed_time(e1) / k2
        if world > 1:
            t = torch.tensor([ems], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ems = float(t.item())
        e2e = {"value": total_flops / (ems * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "muon_step_host: W, G, M in pinned host memory, copied in and W, M copied back "
                       "every step (chunked, copies overlapped with the step)"}

    # ---- roofline of the dominant kernel (the tcgen05 Newton-Schulz GEMM)
    peaks, peak_src = _peaks()
    by = {p["name"]: p for p in prof}
    gemm = [by[k] for k in ("ns_gemm_gram", "ns_gemm_poly", "ns_gemm_update", "ns_gemm_final") if k in by]
    g_launch = sum(p["launches"] for p in gemm)
    g_ms = sum(p["total_ms"] for p in gemm)
    g_flops = sum(p["flops"] for p in gemm)
    achieved = g_flops / (g_ms * 1e-3) / 1e12 if g_ms > 0 else 0.0
    peak = peaks["bf16_tflops_sustained"]
    tr = _traffic_record()
    exec_flops = _executed_flops(w) * args.steps
    roofline = {"kernel": "ns_gemm_pair_kernel (tcgen05 cta_group::2, all three Newton-Schulz products)",
                "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} bf16 sustained",
                "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                "traffic": (tr["bytes_per_launch"] if tr else None),
                "launches": g_launch, "avg_launch_ms": g_ms / max(1, g_launch),
                "flops_per_launch": g_flops / max(1, g_launch),
                "flops_counted": "nominal 5*(4 r^2 k + 2 r^3) per matrix (symmetric products skip "
                                 "lower tiles, so executed FLOPs are fewer)",
                "executed_tflops": exec_flops / (g_ms * 1e-3) / 1e12 if g_ms > 0 else 0.0,
                "executed_frac_of_sustained": (exec_flops / (g_ms * 1e-3) / 1e12) / peak if g_ms > 0 else 0.0}
    kernels = _kernel_rows(prof, args.steps, peaks)
    launches = sum(p["launches"] for p in prof)

    # ---- the same kernels with the batch on one stream: with the two-stream
    # split, a kernel's event time includes the other part's kernels running
    # beside it, so its rate there is not the kernel's own
    one_stream = None
    if not args.no_one_stream:
        prev = os.environ.get("MUON_NO_SPLIT")
        os.environ["MUON_NO_SPLIT"] = "1"
        try:
            batch.step(w.lr, w.mu, w.wd)
            torch.cuda.synchronize()
            mg.muon_profile_enable(True)
            for _ in range(2):
                batch.step(w.lr, w.mu, w.wd)
            torch.cuda.synchronize()
            one_stream = {"steps": 2, "kernels": _kernel_rows(mg.muon_profile_read(), 2, peaks),
                          "note": "MUON_NO_SPLIT=1 (untimed for the metric): each kernel alone on the GPU"}
            mg.muon_profile_enable(False)
        finally:
            if prev is None:
                os.environ.pop("MUON_NO_SPLIT", None)
            else:
                os.environ["MUON_NO_SPLIT"] = prev
        if mg.muon_device_status() != 0:
            raise RuntimeError("device status after the one-stream steps is not OK")

    other = None
    if args.all_configs:
        other = measure_all_configs(mg, wl, torch, dev)

    adamw = None
    if not args.no_adamw:
        adamw = measure_adamw(mg, torch, dev, max(3, args.steps // 2), peaks, args.adamw_elems)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(args.cpu_matrices)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args, w, world),
            "matrices_per_s": mats_per_s,
            "pct_of_bf16_peak": {"burst": value / peaks["bf16_tflops"],
                                 "sustained": value / peaks["bf16_tflops_sustained"],
                                 "source": peak_src},
            "nominal_flops_per_step": total_flops,
            "kernels": kernels, "kernels_one_stream": one_stream, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks, "adamw": adamw, "all_configs": other,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _kernel_rows(prof, steps, peaks):
    """Per-kernel time, share and rate from the library's profile counters."""
    total = max(1e-9, sum(q["total_ms"] for q in prof))
    rows = []
    for p in prof:
        if p["launches"] == 0:
            continue
        k = {"name": p["name"], "launches": p["launches"], "ms_per_step": p["total_ms"] / steps,
             "share": p["total_ms"] / total}
        if p["flops"] > 0 and p["total_ms"] > 0:
            k["tflops"] = p["flops"] / (p["total_ms"] * 1e-3) / 1e12
        if p["bytes"] > 0 and p["total_ms"] > 0:
            k["gbs"] = p["bytes"] / (p["total_ms"] * 1e-3) / 1e9
            k["frac_hbm"] = k["gbs"] / peaks["hbm_gbs"]
        rows.append(k)
    return rows


def workload_config(args, w, world):
    """The ``config`` object of the JSON line (both arms)."""
    return {"workload": (f"{WORKLOAD}: 96 experts x {{gate 2048x6144, up 2048x6144, down "
                         "6144x2048} = 288 matrices per rank, full Muon step (momentum+"
                         "Nesterov, Frobenius normalisation, NS5, weight update)")
                        if args.workload == WORKLOAD else
                        f"{args.workload} (profiling run, not the bench workload): {w.description}",
            "matrices_per_rank": w.count, "steps_ns": 5,
            "coeffs": [3.4445, -4.7750, 2.0315], "lr": w.lr, "mu": w.mu, "wd": w.wd,
            "weights": "bf16", "gradients": "bf16", "momentum": "fp32",
            "parallelism": f"replicas x{world} (whole matrices per rank, no collective)",
            "l2": "inputs larger than L2 (about 29 GB of W, G, M per step)",
            "subset": (f"first {args.max_matrices} matrices only (profiling case)"
                       if args.max_matrices else None)}


# ----------------------------------------------------------- CPU oracle ---
def cpu_baseline_sample(n_mats: int, steps: int = 1):
    """The oracle timed on the host cores on a bounded sample of the same
    workload (the first n_mats matrices, one full Muon step each)."""
    import torch
    import oracle
    from muon_newton_schulz_step_gb300 import workloads as wl

    w = wl.workload(WORKLOAD)
    idx = list(range(n_mats))
    # the sample is drawn by the same seeded recipe on the host
    inp = wl.make_inputs(w, "cpu", indices=idx)
    host = [tuple(x.contiguous() for x in t) for t in zip(inp["W"], inp["G"], inp["M"])]
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(steps):
        for (W, G, M), i in zip(host, idx):
            oracle.muon_step(W.view(torch.int16).numpy().view("uint16"), G.view(torch.int16).numpy().view("uint16"),
                             M.numpy(), w.lr, w.mu, w.wd, w_bf16=True, g_bf16=True)
            flops += wl.nominal_ns_flops(w.mats[i].rows, w.mats[i].cols)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "seconds": dt,
            "sample": f"{n_mats} of the 288 matrices ({', '.join(f'{w.mats[i].rows}x{w.mats[i].cols}' for i in idx)})"
                      f", one full Muon step each, plain C oracle (bf16-emulating NS5, fp32 accumulation)"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from muon_newton_schulz_step_gb300 import workloads as wl

    w = wl.workload(WORKLOAD)
    for _ in range(args.warmup if args.warmup < 1 else 1):
        cpu_baseline_sample(1)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = cpu_baseline_sample(args.cpu_matrices)
        vals.append(r)
    dt = time.perf_counter() - t0
    flops = sum(wl.nominal_ns_flops(w.mats[i].rows, w.mats[i].cols) for i in range(args.cpu_matrices))
    value = flops * args.steps / dt / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16-emulated (fp32 accumulation)",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(args, w, world),
            "sample": (f"each step: {args.cpu_matrices} of the 288 matrices, one full Muon step each, "
                       "on the CPU oracle (bounded sample of the workload)"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": vals[-1]["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-matrices", type=int, default=1)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-adamw", action="store_true")
    ap.add_argument("--no-one-stream", action="store_true",
                    help="skip the per-kernel rates with the batch on one stream")
    ap.add_argument("--adamw-elems", type=int, default=256000 * 6144,
                    help="elements of the large AdamW parameter (default: 256000 x 6144)")
    ap.add_argument("--only-adamw", action="store_true", help="time AdamW alone (profiling)")
    ap.add_argument("--all-configs", action="store_true",
                    help="also time every workload (outside the timed region of the bench value)")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload to step (profiling of other shapes; the bench value is moe_layer)")
    ap.add_argument("--max-matrices", type=int, default=0,
                    help="use only the first N matrices (small profiling case; not a bench value)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
