"""AdamW kernel (the optimizer for the parameters Muon does not cover) against
the oracle: every operation is one IEEE fp32 rounding on both sides, so P, M
and V must match bit for bit."""
import numpy as np
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
import oracle
from tests.gpu_util import bits, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)


def _host(t):
    return bits(t) if t.dtype == torch.bfloat16 else f32(t).copy()


@pytest.mark.parametrize("p_dtype,g_dtype", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
                                             (torch.float32, torch.bfloat16), (torch.bfloat16, torch.float32)])
def test_adamw_bit_exact_against_oracle(p_dtype, g_dtype):
    sizes = [6144, 1, 7, 2048 * 3 + 5, 0, 100003, 384 * 6144]
    gen = torch.Generator(device=DEV).manual_seed(61)
    P = [(0.05 * torch.randn(n, generator=gen, device=DEV)).to(p_dtype) for n in sizes]
    M = [torch.zeros(n, device=DEV) for n in sizes]
    V = [torch.zeros(n, device=DEV) for n in sizes]
    hP, hM, hV = [_host(t) for t in P], [f32(t).copy() for t in M], [f32(t).copy() for t in V]
    for step in (1, 2, 3):
        G = [(torch.randn(n, generator=gen, device=DEV) * 1e-2).to(g_dtype) for n in sizes]
        hG = [_host(t) for t in G]
        mg.muon_adamw_step(P, G, M, V, step=step, **HP)
        torch.cuda.synchronize()
        for i, n in enumerate(sizes):
            hP[i], hM[i], hV[i] = oracle.adamw(hP[i], hG[i], hM[i], hV[i], step=step,
                                               p_bf16=p_dtype == torch.bfloat16,
                                               g_bf16=g_dtype == torch.bfloat16, **HP)
            assert np.array_equal(_host(P[i]).ravel(), hP[i]), f"P of tensor {i} ({n}) at step {step}"
            assert np.array_equal(f32(M[i]).view(np.uint32).ravel(), hM[i].view(np.uint32)), f"M {i}"
            assert np.array_equal(f32(V[i]).view(np.uint32).ravel(), hV[i].view(np.uint32)), f"V {i}"


def test_adamw_many_tensors_span_several_launches():
    n_t = 600
    gen = torch.Generator(device=DEV).manual_seed(62)
    sizes = [int(s) for s in torch.randint(1, 5000, (n_t,), generator=torch.Generator().manual_seed(3))]
    P = [(0.05 * torch.randn(n, generator=gen, device=DEV)).to(torch.bfloat16) for n in sizes]
    G = [(1e-2 * torch.randn(n, generator=gen, device=DEV)).to(torch.bfloat16) for n in sizes]
    M = [torch.zeros(n, device=DEV) for n in sizes]
    V = [torch.zeros(n, device=DEV) for n in sizes]
    hP, hG = [bits(t) for t in P], [bits(t) for t in G]
    mg.muon_profile_enable(True)
    mg.muon_adamw_step(P, G, M, V, step=1, **HP)
    torch.cuda.synchronize()
    prof = {p["name"]: p for p in mg.muon_profile_read()}
    mg.muon_profile_enable(False)
    assert prof["adamw"]["launches"] == 3          # 256 tensors per launch
    for i in (0, 255, 256, 511, 512, 599):
        want, _, _ = oracle.adamw(hP[i], hG[i], np.zeros(sizes[i], np.float32), np.zeros(sizes[i], np.float32),
                                  step=1, p_bf16=True, g_bf16=True, **HP)
        assert np.array_equal(bits(P[i]), want)


def test_adamw_rejects_bad_arguments():
    p = torch.zeros(16, device=DEV)
    with pytest.raises(mg.MuonError):
        mg.muon_adamw_step([p], [p.clone()], [p.clone()], [p.clone()], lr=1e-3, step=0)
    with pytest.raises(mg.MuonError):
        mg.muon_adamw_step([p], [p.clone()], [p.clone()], [p.clone()], lr=1e-3, beta1=1.0, step=1)
    with pytest.raises(mg.MuonError):
        mg.muon_adamw_step([p], [p], [p.clone()], [p.clone()], lr=1e-3, step=1)   # P aliases G
