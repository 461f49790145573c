"""Host-side pieces of bench.py that need no GPU: the per-kernel rows built
from the library's profile counters and the config object both arms print."""
import types

import bench
from muon_newton_schulz_step_gb300 import workloads as wl

PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}


def test_kernel_rows_rates_and_shares():
    prof = [{"name": "norm_pass", "launches": 4, "total_ms": 10.0, "flops": 0.0, "bytes": 60e9},
            {"name": "ns_gemm_gram", "launches": 10, "total_ms": 30.0, "flops": 45e12, "bytes": 0.0},
            {"name": "unpack", "launches": 0, "total_ms": 0.0, "flops": 0.0, "bytes": 0.0}]
    rows = bench._kernel_rows(prof, 2, PEAKS)
    assert [r["name"] for r in rows] == ["norm_pass", "ns_gemm_gram"]        # unlaunched kernels left out
    norm, gram = rows
    assert norm["ms_per_step"] == 5.0 and abs(norm["share"] - 0.25) < 1e-12
    assert abs(norm["gbs"] - 6000.0) < 1e-9 and abs(norm["frac_hbm"] - 0.75) < 1e-12
    assert abs(gram["tflops"] - 1500.0) < 1e-9 and "gbs" not in gram and "tflops" not in norm


def test_both_arms_share_one_config():
    args = types.SimpleNamespace(workload=bench.WORKLOAD, max_matrices=0)
    cfg = bench.workload_config(args, wl.workload(bench.WORKLOAD), 1)
    assert cfg["matrices_per_rank"] == 288 and cfg["subset"] is None
    assert "{gate 2048x6144, up 2048x6144, down 6144x2048} = 288" in cfg["workload"]
    assert cfg["parallelism"].startswith("replicas x1")
    sub = bench.workload_config(types.SimpleNamespace(workload="tiny", max_matrices=3), wl.workload("tiny"), 2)
    assert sub["workload"].startswith("tiny (profiling run") and sub["subset"].startswith("first 3")


def test_executed_flops_count_only_upper_tiles():
    w = wl.workload(bench.WORKLOAD)
    ex = bench._executed_by_product(w)
    # 2048 x 6144: 8 x 8 tiles of 256, 36 in the upper triangle; the update runs all 64
    per_mat_gram = 2.0 * 36 * 256 * 256 * 6144
    assert ex["gram"] == 288 * per_mat_gram
    assert ex["poly"] == 288 * 2.0 * 36 * 256 * 256 * 2048
    assert ex["update"] == 288 * 2.0 * 2048 * 6144 * 2048
    assert abs(bench._executed_flops(w) - 1.2988e14) / 1.2988e14 < 1e-3
    assert bench._executed_flops(w) < bench._nominal_flops(w)


def test_product_rows_from_one_stream_kernels():
    w = wl.workload(bench.WORKLOAD)
    rows = [{"name": "ns_gemm_gram", "ms_per_step": 25.0}, {"name": "ns_gemm_update", "ms_per_step": 40.0},
            {"name": "ns_gemm_final", "ms_per_step": 10.0}, {"name": "norm_pass", "ms_per_step": 5.0}]
    out = {r["name"]: r for r in bench._product_rows(rows, w, PEAKS)}
    assert set(out) == {"ns_gemm_gram", "ns_gemm_update", "ns_gemm_final"}
    ex = bench._executed_by_product(w)
    assert abs(out["ns_gemm_gram"]["executed_tflops"] - 5 * ex["gram"] / 25e-3 / 1e12) < 1e-6
    assert out["ns_gemm_update"]["ms_per_iteration"] == 10.0          # four of the five iterations
    assert out["ns_gemm_final"]["ms_per_iteration"] == 10.0
    assert abs(out["ns_gemm_final"]["frac_sustained"] * 1800.0 - out["ns_gemm_final"]["executed_tflops"]) < 1e-6


def test_numa_helpers_on_the_host():
    import torch
    t = torch.empty(1 << 20, dtype=torch.uint8)
    t.fill_(1)
    nodes = bench._numa_nodes_of([t])
    assert nodes is None or sum(nodes.values()) >= 1
    with bench.bind_to_node(None):      # unknown node: nothing changes
        pass
    assert isinstance(bench._cpu_model(), str)
