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
