"""GPU parity on knife-edge spectra at the shapes the tensor cores serve.

The recipe is the tiny workload's: rank-4 signal with singular values
s ~ U[0.1, 10] plus N(0, 1e-3) noise, which after normalisation puts the noise
directions at sigma of about 1e-3 to 4e-3, where the quintic's fifth iterate
is steepest.  Here it runs at every shape above the shared-memory path's
capacity up to 1024 x 2048, so the matrices go through the tcgen05 products
(whose fp32 accumulation truncates rather than rounding to nearest) with the
default routing.  O must stay within the contract (relative Frobenius error
1e-2, per-element absolute error 2e-2 against the oracle) on every matrix that
is well-conditioned for bf16 Newton-Schulz, and within the contract plus the
oracle's own spread between its two legal summation orders on the others
(tests/conditioning.py); the momentum is bit-exact and W bit-exact given O.

Shapes are Muon's whole-matrix orthogonalisation targets of every size one
rank holds ("How PyTorch Scaled a Near-1T MoE on Europe's Public
Supercomputer", section "Three optimizations that changed the economics",
FlexShard bullet).
"""
import numpy as np
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
import oracle
from muon_newton_schulz_step_gb300 import workloads as wl
from tests.conditioning import bound_for, order_spread
from tests.gpu_util import bits, compare_o, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = [(128, 384), (256, 768), (768, 256), (512, 1536), (1024, 2048)]


def _knife_workload(shape, count, g_dtype, seed_id):
    mats = [wl.MatrixSpec(*shape, "uniform", 4, 0.1, 10.0, 1e-3, "knife_edge") for _ in range(count)]
    return wl.Workload("knife_edge", seed_id, "step", mats, g_dtype=g_dtype, w_dtype=g_dtype,
                       m_std=0.0, on_host=True)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_knife_edge_spectrum_on_the_tensor_core_route(shape, dtype, monkeypatch):
    for var in ("MUON_DISABLE_SMALL_NS", "MUON_NO_FUSED_UPDATE"):
        monkeypatch.delenv(var, raising=False)
    count = 4 if shape[0] * shape[1] > 1 << 20 else 8
    w = _knife_workload(shape, count, dtype, seed_id=40 + SHAPES.index(shape))
    inp = wl.make_inputs(w, DEV)
    bf = dtype == torch.bfloat16
    host = {k: [bits(t) if t.dtype == torch.bfloat16 else f32(t).copy() for t in inp[k]] for k in ("W", "G", "M")}
    O = [torch.empty(shape, dtype=torch.bfloat16, device=DEV) for _ in range(count)]
    mg.muon_profile_enable(True)
    try:
        mg.muon_step_ex(inp["W"], inp["G"], inp["M"], w.lr, w.mu, w.wd, o_out=O)
        torch.cuda.synchronize()
        launched = {p["name"]: p["launches"] for p in mg.muon_profile_read()}
    finally:
        mg.muon_profile_enable(False)
    assert mg.muon_device_status() == 0
    # the default routing sends these shapes to the tensor cores, not the shared-memory kernel
    assert launched.get("ns_gemm_gram", 0) >= 1 and launched.get("ns_small", 0) == 0, launched
    well = 0
    for i in range(count):
        def ref():
            return oracle.muon_step(host["W"][i], host["G"][i], host["M"][i], w.lr, w.mu, w.wd,
                                    w_bf16=bf, g_bf16=bf)
        W1, M1, Oref = ref()
        assert np.array_equal(f32(inp["M"][i]).view(np.uint32), M1.view(np.uint32)), f"M of matrix {i}"
        Og = f32(O[i])
        rel_b, abs_b, ok = bound_for(order_spread(lambda: ref()[2]))
        well += ok
        rel, mx = compare_o(Og, Oref)
        assert rel <= rel_b and mx <= abs_b, \
            f"O of matrix {i} ({shape}, {dtype}): rel {rel:.3e} (bound {rel_b:.3e}), max {mx:.3e} (bound {abs_b:.3e})"
        dcy, s = oracle.update_scalars(w.lr, w.wd, *shape)
        Wexp = oracle.weight_update(host["W"][i], Og, dcy, s, w_bf16=bf)
        Wgot = bits(inp["W"][i]) if bf else f32(inp["W"][i]).view(np.uint32)
        assert np.array_equal(Wgot, Wexp if bf else Wexp.view(np.uint32)), f"W of matrix {i}"
    # the contract itself is what most of these matrices are held to
    assert well >= count // 2, f"only {well} of {count} matrices well-conditioned"
