"""Matrices of one batch do not affect each other.

They share launches, shape buckets, tiles of the persistent kernels and the
workspace, so a non-finite gradient in one matrix is a sharp probe: that
matrix's result turns non-finite (values propagate; nothing scans for them),
and every other matrix must come out bit-identical to a batch without it.
"""
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _batch(shapes, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W = [(0.02 * torch.randn(s, generator=gen, device=DEV)).to(torch.bfloat16) for s in shapes]
    G = [torch.randn(s, generator=gen, device=DEV).to(torch.bfloat16) for s in shapes]
    M = [1e-3 * torch.randn(s, generator=gen, device=DEV) for s in shapes]
    return W, G, M


@pytest.mark.parametrize("route", ["small", "tensor_core", "tensor_core_fp8"])
def test_non_finite_gradient_stays_in_its_matrix(route, monkeypatch):
    """The FP8 route adds per-matrix state shared through one launch: each
    matrix's max |X| (gathered with atomics) sets its own E4M3 scale, so a
    non-finite matrix must not move any other matrix's scale either."""
    if route.startswith("tensor_core"):
        monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    else:
        monkeypatch.delenv("MUON_DISABLE_SMALL_NS", raising=False)
    fp8 = route == "tensor_core_fp8"
    shapes = [(64, 256), (256, 64), (64, 256), (96, 200), (300, 700), (700, 300)]
    bad = [1, 4]
    Wa, Ga, Ma = _batch(shapes, 41)
    Wb, Gb, Mb = [w.clone() for w in Wa], [g.clone() for g in Ga], [m.clone() for m in Ma]
    Gb[bad[0]][3, 5] = float("nan")
    Gb[bad[1]][0, 0] = float("inf")
    mg.muon_step_ex(Wa, Ga, Ma, 0.02, 0.95, 0.1, fp8_gram=fp8)
    mg.muon_step_ex(Wb, Gb, Mb, 0.02, 0.95, 0.1, fp8_gram=fp8)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        if i in bad:
            assert not torch.isfinite(Wb[i].float()).all(), f"matrix {i}: non-finite input vanished"
            continue
        assert torch.equal(Wa[i].view(torch.int16), Wb[i].view(torch.int16)), f"W[{i}] changed"
        assert torch.equal(Ma[i].view(torch.int32), Mb[i].view(torch.int32)), f"M[{i}] changed"
