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


def _executed_by_product(w, tile=256):
    """FLOPs the default (pair-CTA, 256 x 256 tile) GEMM kernel executes for one
    Newton-Schulz iteration over the workload's tensor-core matrices, per
    product: the symmetric products (Gram, polynomial) run only tiles with
    tm <= tn over the zero-padded iterate; the update runs every tile."""
    out = {"gram": 0.0, "poly": 0.0, "update": 0.0}
    for s in w.mats:
        r, k = min(s.rows, s.cols), max(s.rows, s.cols)
        rp, kp = -(-r // tile) * tile, -(-k // tile) * tile
        nt = rp // tile
        sym = nt * (nt + 1) // 2 * tile * tile
        out["gram"] += 2.0 * sym * kp
        out["poly"] += 2.0 * sym * rp
        out["update"] += 2.0 * rp * kp * rp
    return out


def _executed_flops(w, steps=5, tile=256):
    """Executed tensor-core FLOPs of the whole Newton-Schulz phase (all steps)."""
    return steps * sum(_executed_by_product(w, tile).values())


def _product_rows(one_stream_rows, w, peaks, steps=5):
    """Per product (Gram, polynomial, update, fused final update): executed
    and nominal TFLOP/s and the executed rate's fraction of both bf16 peaks,
    from the kernels' own event times with the batch on one stream."""
    ex = _executed_by_product(w)
    nominal = {"gram": 0.0, "poly": 0.0, "update": 0.0}
    for m in w.mats:
        r, k = min(m.rows, m.cols), max(m.rows, m.cols)
        nominal["gram"] += 2.0 * r * r * k
        nominal["poly"] += 2.0 * r ** 3
        nominal["update"] += 2.0 * r * r * k
    per_step = {"ns_gemm_gram": ("gram", steps), "ns_gemm_poly": ("poly", steps),
                "ns_gemm_update": ("update", steps - 1), "ns_gemm_final": ("update", 1)}
    rows = []
    for k in one_stream_rows or []:
        if k["name"] not in per_step or k["ms_per_step"] <= 0:
            continue
        prod, n = per_step[k["name"]]
        sec = k["ms_per_step"] * 1e-3
        ex_t = ex[prod] * n / sec / 1e12
        rows.append({"name": k["name"], "ms_per_step": k["ms_per_step"],
                     "ms_per_iteration": k["ms_per_step"] / n,
                     "executed_tflops": ex_t, "nominal_tflops": nominal[prod] * n / sec / 1e12,
                     "frac_sustained": ex_t / peaks["bf16_tflops_sustained"],
                     "frac_burst": ex_t / peaks["bf16_tflops"]})
    return rows


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


def measure_all_configs(mg, wl, torch, dev, names=("tiny", "expert_gate", "dense_attn", "mixed_block"),
                        steps: int = 5, warmup: int = 2):
    """Step time of the other workloads (the bench value is moe_layer's): per
    workload ms, nominal and executed Newton-Schulz TFLOP/s and matrices/s.
    Each workload's inputs are larger than L2 except the tiny one's, which is
    launch-bound and is stepped 50 times."""
    out = {}
    for name in names:
        w = wl.workload(name)
        inp = wl.make_inputs(w, dev)
        if w.call == "ns":
            batch = None

            def step():
                mg.muon_ns5_batched(inp["G"])
        else:
            batch = mg.MuonStepBatch(inp["W"], inp["G"], inp["M"])

            def step():
                batch.step(w.lr, w.mu, w.wd)
        n = 50 if name == "tiny" else steps
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            step()
        e1.record()
        torch.cuda.synchronize()
        if mg.muon_device_status() != 0:
            raise RuntimeError(f"device status after {name} is not OK")
        ms = e0.elapsed_time(e1) / n
        flops = sum(wl.nominal_ns_flops(m.rows, m.cols) for m in w.mats)
        row = {"call": "muon_ns5_batched" if w.call == "ns" else "muon_step_ex", "matrices": w.count,
               "steps_timed": n, "ms": ms, "nominal_tflops": flops / (ms * 1e-3) / 1e12,
               "matrices_per_s": w.count / (ms * 1e-3)}
        if name != "tiny":   # the tiny matrices run on the CUDA cores, not the tensor cores
            row["executed_tflops"] = _executed_flops(w) / (ms * 1e-3) / 1e12
        out[name] = row
        del inp, batch
        mg.muon_release_workspace()
        torch.cuda.empty_cache()
    return out


def cublas_comparator(torch, dev, peaks, count: int = 288, r: int = 2048, k: int = 6144, reps: int = 12):
    """cuBLAS (torch.bmm, bf16 in, fp32 accumulation, bf16 out) on the shapes of
    the Newton-Schulz products of the 288-matrix layer: the update's
    [r x r] . [r x k] with the row-major iterate as the right operand, and the
    Gram's [r x k] . [k x r] computed densely.  A comparator on the same box
    only; the library never calls it.  `reps` back-to-back calls after as many
    untimed ones (about 0.1 s each way), so that the board sits at the power-capped
    clock the step's own products run at, not at the higher clock of a short burst."""
    gen = torch.Generator(device=dev).manual_seed(5)
    B = torch.randn(count, r, r, generator=gen, device=dev).to(torch.bfloat16)
    X = torch.randn(count, r, k, generator=gen, device=dev).to(torch.bfloat16)
    out = {}
    for name, fn, flops in (("update", lambda: torch.bmm(B, X), 2.0 * count * r * r * k),
                            ("gram_dense", lambda: torch.bmm(X, X.transpose(1, 2)), 2.0 * count * r * r * k)):
        for _ in range(reps):
            y = fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            y = fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        t = flops / (ms * 1e-3) / 1e12
        out[name] = {"shape": f"{count} x [{r}x{r}].[{r}x{k}]" if name == "update" else
                     f"{count} x [{r}x{k}].[{k}x{r}] (all tiles)",
                     "ms": ms, "tflops": t, "frac_sustained": t / peaks["bf16_tflops_sustained"]}
        del y
    del B, X
    torch.cuda.empty_cache()
    return out


def _gpu_pci_ids(dev_index: int):
    """Candidate sysfs names (dddd:bb:dd.f) of the GPU's PCI device."""
    out = []
    try:
        import torch
        p = torch.cuda.get_device_properties(dev_index)
        dom, bus, dv = (getattr(p, k, None) for k in ("pci_domain_id", "pci_bus_id", "pci_device_id"))
        if all(isinstance(v, int) for v in (dom, bus, dv)):
            out.append(f"{dom:04x}:{bus:02x}:{dv:02x}.0")
    except Exception:
        pass
    try:
        r = subprocess.run(["nvidia-smi", "-i", str(dev_index), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=20)
        b = r.stdout.strip().lower()
        if b:
            dom, rest = b.split(":", 1)
            out.append(f"{int(dom, 16):04x}:{rest}")
    except Exception:
        pass
    return out


def _gpu_numa_node(dev_index: int):
    """NUMA node the GPU is attached to (from its PCI device in sysfs), or None."""
    for b in _gpu_pci_ids(dev_index):
        try:
            with open(f"/sys/bus/pci/devices/{b}/numa_node") as f:
                node = int(f.read().strip())
            return node if node >= 0 else None
        except Exception:
            continue
    return None


def _node_cpus(node: int):
    try:
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            text = f.read().strip()
    except Exception:
        return set()
    cpus = set()
    for part in text.split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def _numa_nodes_of(tensors):
    """Pages per NUMA node of the host tensors' mappings (/proc/self/numa_maps)."""
    try:
        with open("/proc/self/numa_maps") as f:
            maps = f.read().splitlines()
    except Exception:
        return None
    starts = []
    for line in maps:
        parts = line.split()
        try:
            starts.append((int(parts[0], 16), parts))
        except (ValueError, IndexError):
            continue
    starts.sort()
    nodes, seen = {}, set()
    for t in tensors:
        addr = t.data_ptr()
        best = None
        for a, parts in starts:
            if a <= addr:
                best = (a, parts)
            else:
                break
        if best is None or best[0] in seen:
            continue                     # each mapping counted once
        seen.add(best[0])
        for tok in best[1][1:]:
            if tok.startswith("N") and "=" in tok:
                n, c = tok[1:].split("=")
                nodes[int(n)] = nodes.get(int(n), 0) + int(c)
    return {str(k): v for k, v in sorted(nodes.items())} or None


class bind_to_node:
    """Runs the calling thread on the CPUs of one NUMA node while host memory is
    allocated and pinned, so that first-touch placement puts the pages on that
    node (the one the GPU is attached to).  No-op when the node is unknown."""

    def __init__(self, node):
        self.node = node
        self.saved = None

    def __enter__(self):
        cpus = _node_cpus(self.node) if self.node is not None else set()
        if cpus and hasattr(os, "sched_setaffinity"):
            try:
                self.saved = os.sched_getaffinity(0)
                os.sched_setaffinity(0, cpus & self.saved or cpus)
            except OSError:
                self.saved = None
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            try:
                os.sched_setaffinity(0, self.saved)
            except OSError:
                pass
        return False


def link_probe(torch, dev, node, nbytes: int = 4 << 30, reps: int = 3):
    """Host<->device copy rates on pinned buffers of ``nbytes``: host->device
    alone, device->host alone, and both at once on two streams (GB/s)."""
    with bind_to_node(node):
        h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        h_in.fill_(1)
        h_out.fill_(0)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.ones(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    def both():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    t_h2d = timed(lambda: d_in.copy_(h_in, non_blocking=True))
    t_d2h = timed(lambda: h_out.copy_(d_out, non_blocking=True))
    t_both = timed(both)
    out = {"bytes": nbytes, "h2d_gbs": nbytes / t_h2d / 1e9, "d2h_gbs": nbytes / t_d2h / 1e9,
           "both_ways_gbs": 2 * nbytes / t_both / 1e9, "host_numa_pages": _numa_nodes_of([h_in, h_out])}
    del h_in, h_out, d_in, d_out
    torch.cuda.empty_cache()
    return out


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


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
    batch = mg.MuonStepBatch(inp["W"], inp["G"], inp["M"], fp8_gram=args.fp8_gram)
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
    gpu_node = _gpu_numa_node(local)
    if not args.no_e2e:
        try:
            # host copies on the NUMA node the GPU is attached to (first touch
            # from that node's CPUs), so copies do not cross the CPU-CPU link
            with bind_to_node(gpu_node):
                pinned = tuple([t.cpu().pin_memory() for t in inp[k]] for k in ("W", "G", "M"))
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
               "gpu_numa_node": gpu_node, "host_numa_pages": _numa_nodes_of(hW + hG + hM),
               "note": "muon_step_host: W, G, M in pinned host memory, copied in and W, M copied back "
                       "every step (chunked, copies overlapped with the step)"}
        del host_batch, pinned, hW, hG, hM
        if not args.no_link_probe:
            try:
                probe = link_probe(torch, dev, gpu_node)
                e2e["link_probe"] = probe
                # the step's bytes over the time the link needs for them: copies
                # in and out overlap, so the floor is the larger of the both-ways
                # time and each direction's time alone
                floor_s = max((h2d + d2h) / (probe["both_ways_gbs"] * 1e9), h2d / (probe["h2d_gbs"] * 1e9),
                              d2h / (probe["d2h_gbs"] * 1e9))
                e2e["link_floor_ms"] = floor_s * 1e3
                e2e["frac_of_link"] = floor_s / (ems * 1e-3)
            except RuntimeError as exc:
                e2e["link_probe"] = {"error": str(exc)[:160]}

    # ---- roofline of the dominant kernel (the tcgen05 Newton-Schulz GEMM):
    # the FLOPs it executes (upper tiles only for the symmetric products) over
    # its launches' event time; the nominal count of the metric beside it
    peaks, peak_src = _peaks()
    by = {p["name"]: p for p in prof}
    gemm = [by[k] for k in ("ns_gemm_gram", "ns_gemm_poly", "ns_gemm_update", "ns_gemm_final") if k in by]
    g_launch = sum(p["launches"] for p in gemm)
    g_ms = sum(p["total_ms"] for p in gemm)
    g_flops = sum(p["flops"] for p in gemm)
    peak = peaks["bf16_tflops_sustained"]
    tr = _traffic_record()
    exec_flops = _executed_flops(w) * args.steps
    achieved = exec_flops / (g_ms * 1e-3) / 1e12 if g_ms > 0 else 0.0
    nominal_rate = g_flops / (g_ms * 1e-3) / 1e12 if g_ms > 0 else 0.0
    roofline = {"kernel": "ns_gemm_pair_kernel (tcgen05 cta_group::2, all three Newton-Schulz products)",
                "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} bf16 sustained",
                "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                "traffic": (tr["bytes_per_launch"] if tr else None),
                "launches": g_launch, "avg_launch_ms": g_ms / max(1, g_launch),
                "flops_per_launch": exec_flops / max(1, g_launch),
                "flops_counted": "executed: the kernel's tiles (symmetric Gram and polynomial products "
                                 "run only tiles with tm <= tn), per launch over its event time",
                "achieved_nominal": nominal_rate, "frac_nominal": nominal_rate / peak,
                "flops_per_launch_nominal": g_flops / max(1, g_launch),
                "nominal_counted": "5*(4 r^2 k + 2 r^3) per matrix, the metric's count"}
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
            rows1 = _kernel_rows(mg.muon_profile_read(), 2, peaks)
            prods = _product_rows(rows1, w, peaks)
            per_it = {r["name"]: r["ms_per_iteration"] for r in prods}
            one_stream = {"steps": 2, "kernels": rows1, "products": prods,
                          # the fused final update against a plain update launch over the same matrices
                          "final_over_update": (per_it["ns_gemm_final"] / per_it["ns_gemm_update"]
                                                if per_it.get("ns_gemm_final") and per_it.get("ns_gemm_update")
                                                else None),
                          "note": "MUON_NO_SPLIT=1 (untimed for the metric): each kernel alone on the GPU"}
            mg.muon_profile_enable(False)
        finally:
            if prev is None:
                os.environ.pop("MUON_NO_SPLIT", None)
            else:
                os.environ["MUON_NO_SPLIT"] = prev
        if mg.muon_device_status() != 0:
            raise RuntimeError("device status after the one-stream steps is not OK")

    # ---- the FP8 variant (E4M3 Gram operands) on the same layer, untimed for the metric
    fp8 = None
    if not args.no_fp8:
        b8 = mg.MuonStepBatch(inp["W"], inp["G"], inp["M"], fp8_gram=True)
        b8.step(w.lr, w.mu, w.wd)
        torch.cuda.synchronize()
        mg.muon_profile_enable(True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n8 = max(3, min(args.steps, 5))
        e0.record(stream)
        for _ in range(n8):
            b8.step(w.lr, w.mu, w.wd)
        e1.record(stream)
        torch.cuda.synchronize()
        rows8 = _kernel_rows(mg.muon_profile_read(), n8, peaks)
        mg.muon_profile_enable(False)
        ms8 = e0.elapsed_time(e1) / n8
        if mg.muon_device_status() != 0:
            raise RuntimeError("device status after the FP8 steps is not OK")
        fp8 = {"ms_per_step": ms8, "nominal_tflops": flops / (ms8 * 1e-3) / 1e12,
               "step_vs_bf16": ms8 / ms_per_step, "steps": n8, "kernels": rows8,
               "note": "ns_fp8_gram = 1: each Newton-Schulz iteration's Gram product on E4M3 operands "
                       "(per-matrix power-of-two scale), polynomial and update in bf16; the FLOP count is "
                       "the metric's nominal one"}
        del b8

    del batch, inp
    mg.muon_release_workspace()
    torch.cuda.empty_cache()
    other = None
    if not args.no_all_configs:
        other = measure_all_configs(mg, wl, torch, dev)
    comparator = None
    if not args.no_cublas:
        comparator = cublas_comparator(torch, dev, peaks)
        upd = [r for r in (one_stream or {}).get("products", []) if r["name"] == "ns_gemm_update"]
        if upd:
            comparator["update_product_vs_cublas"] = upd[0]["executed_tflops"] / comparator["update"]["tflops"]

    adamw = None
    if not args.no_adamw:
        adamw = measure_adamw(mg, torch, dev, max(3, args.steps // 2), peaks, args.adamw_elems)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_all_shapes)

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
            "cublas_comparator": comparator, "fp8_gram": fp8,
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
                       if args.max_matrices else None),
            "fp8_gram": bool(getattr(args, "fp8_gram", False))}


# ----------------------------------------------------------- CPU oracle ---
def _oracle_steps(w, idx):
    """Time the oracle's full Muon step on matrices ``idx`` of workload ``w``
    (drawn on the host by the same seeded recipe).  Returns per-matrix
    seconds."""
    import torch
    import oracle
    from muon_newton_schulz_step_gb300 import workloads as wl

    inp = wl.make_inputs(w, "cpu", indices=idx)
    secs = []
    for j in range(len(idx)):
        G = inp["G"][j].contiguous()
        if w.call == "ns":
            g = G.view(torch.int16).numpy().view("uint16")
            t0 = time.perf_counter()
            oracle.ns(oracle.bf16_to_f32(g), 5)
            secs.append(time.perf_counter() - t0)
            continue
        W, M = inp["W"][j].contiguous(), inp["M"][j].contiguous()
        bf = W.dtype == torch.bfloat16
        wv = W.view(torch.int16).numpy().view("uint16") if bf else W.numpy()
        gv = G.view(torch.int16).numpy().view("uint16") if G.dtype == torch.bfloat16 else G.numpy()
        t0 = time.perf_counter()
        oracle.muon_step(wv, gv, M.numpy(), w.lr, w.mu, w.wd, w_bf16=bf, g_bf16=G.dtype == torch.bfloat16)
        secs.append(time.perf_counter() - t0)
    return secs


def cpu_baseline(all_shapes: bool = False):
    """The oracle on the host cores: the whole tiny batch, and two matrices of
    each distinct shape of the other workloads (the 6144 x 6144 dense shape only
    with ``all_shapes``: about 40 s a matrix), with each workload's full time
    extrapolated from the per-shape seconds.  Returns the cpu_baseline object;
    its value is the nominal TFLOP/s over every matrix timed."""
    import oracle
    from muon_newton_schulz_step_gb300 import workloads as wl

    per_shape, flops, total = {}, 0.0, 0.0
    tiny = wl.workload("tiny")
    t_tiny = _oracle_steps(tiny, list(range(tiny.count)))
    flops += sum(wl.nominal_ns_flops(m.rows, m.cols) for m in tiny.mats)
    total += sum(t_tiny)
    picks = [("moe_layer", [0, 1]), ("moe_layer", [2, 5]), ("dense_attn", [4, 5])]
    if all_shapes:
        picks.append(("dense_attn", [0, 1]))
    for name, idx in picks:
        w = wl.workload(name)
        secs = _oracle_steps(w, idx)
        m = w.mats[idx[0]]
        per_shape[f"{m.rows}x{m.cols}"] = sum(secs) / len(secs)
        flops += sum(wl.nominal_ns_flops(w.mats[i].rows, w.mats[i].cols) for i in idx)
        total += sum(secs)
    rate = flops / total   # FLOP/s over the sample, for shapes not timed
    extrap = {"tiny": {"seconds": sum(t_tiny), "how": "measured (whole batch)"}}
    for name in ("expert_gate", "dense_attn", "moe_layer", "mixed_block"):
        w = wl.workload(name)
        sec, by_rate = 0.0, 0
        for m in w.mats:
            key = f"{m.rows}x{m.cols}"
            if key in per_shape:
                sec += per_shape[key]
            else:
                sec += wl.nominal_ns_flops(m.rows, m.cols) / rate
                by_rate += 1
        how = "extrapolated from the per-shape seconds"
        if by_rate:
            how += f" ({by_rate} matrices of untimed shapes at the sample's FLOP rate)"
        extrap[name] = {"seconds": sec, "how": how}
    return {"value": flops / total / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "nproc": os.cpu_count(), "cpu_model": _cpu_model(), "kind": "oracle", "seconds": total,
            "seconds_per_matrix": per_shape, "tiny_batch_seconds": sum(t_tiny),
            "extrapolated_workload_seconds": extrap,
            "sample": "the tiny batch (8 x 64x256) and 2 matrices of each shape: " + ", ".join(per_shape)
                      + "; one full Muon step each on the plain C oracle (bf16-emulating NS5, fp32 "
                        "accumulation)"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from muon_newton_schulz_step_gb300 import workloads as wl

    w = wl.workload(WORKLOAD)
    # each step: the oracle's full Muon step on one matrix of the layer, taking
    # gate, up and down matrices in turn (both orientations)
    order = [0, 1, 2]
    for j in range(min(1, args.warmup)):
        _oracle_steps(w, [order[j % 3]])
    secs, flops = [], 0.0
    for j in range(args.steps):
        i = order[j % 3]
        secs += _oracle_steps(w, [i])
        flops += wl.nominal_ns_flops(w.mats[i].rows, w.mats[i].cols)
    dt = sum(secs)
    value = flops / dt / 1e12
    sample = ("each step: one of the 288 matrices (gate 2048x6144, up 2048x6144, down 6144x2048 in turn), "
              "one full Muon step on the CPU oracle (bounded sample of the workload)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16-emulated (fp32 accumulation)",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(args, w, world),
            "sample": sample,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "cpu_model": _cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-all-shapes", action="store_true",
                    help="CPU baseline also times two 6144x6144 matrices (about 80 s more)")
    ap.add_argument("--no-link-probe", action="store_true", help="skip the host link probe")
    ap.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS comparator")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8-variant steps")
    ap.add_argument("--fp8-gram", action="store_true",
                    help="step the measured batch with the FP8 Gram (profiling of that variant; not the metric)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-adamw", action="store_true")
    ap.add_argument("--no-one-stream", action="store_true",
                    help="skip the per-kernel rates with the batch on one stream")
    ap.add_argument("--adamw-elems", type=int, default=256000 * 6144,
                    help="elements of the large AdamW parameter (default: 256000 x 6144)")
    ap.add_argument("--only-adamw", action="store_true", help="time AdamW alone (profiling)")
    ap.add_argument("--no-all-configs", action="store_true",
                    help="skip timing the other workloads (outside the timed region of the bench value)")
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
