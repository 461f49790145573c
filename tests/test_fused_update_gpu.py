"""The fused last update against the unfused path, through the C ABI.

By default the last Newton-Schulz update of a tensor-core matrix writes its
result straight to the caller's matrix: the weight update W <- dcy*W - s*O
(muon_step) or the store of O (muon_ns5_batched), in the stored orientation.
MUON_NO_FUSED_UPDATE=1 makes the same product write X and leaves the weight
update to the separate kernel.  Both round O to bf16 and then apply one fp32
fma, so W, M and O must agree bit for bit: every orientation, ragged widths
(scalar stores), fp32 W, the optional O copy and more than one launch group
of shape buckets.  Past the fused kernel's table size the library falls back
to the separate kernel; that case and the fused one are also checked
against the oracle.
"""
import numpy as np
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
import oracle
from tests.gpu_util import assert_o_close, bits, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"

# transposed and not, widths that are and are not multiples of 8, padded edges
SHAPES = [(256, 768), (768, 256), (300, 700), (700, 300), (512, 512), (200, 1030), (1030, 200),
          (64, 4100), (4100, 64), (1, 600), (600, 1), (260, 777), (777, 260)]


@pytest.fixture(autouse=True)
def tensor_core_path(monkeypatch):
    monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    monkeypatch.delenv("MUON_NO_FUSED_UPDATE", raising=False)


def _state(shapes, w_dtype, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W = [(0.02 * torch.randn(s, generator=gen, device=DEV)).to(w_dtype) for s in shapes]
    G = [torch.randn(s, generator=gen, device=DEV).to(torch.bfloat16) for s in shapes]
    M = [1e-3 * torch.randn(s, generator=gen, device=DEV) for s in shapes]
    return W, G, M


def _step(shapes, w_dtype, fused, monkeypatch, seed=5, with_o=True):
    if fused:
        monkeypatch.delenv("MUON_NO_FUSED_UPDATE", raising=False)
    else:
        monkeypatch.setenv("MUON_NO_FUSED_UPDATE", "1")
    W, G, M = _state(shapes, w_dtype, seed)
    O = [torch.full(s, 7.0, dtype=torch.bfloat16, device=DEV) for s in shapes] if with_o else None
    mg.muon_profile_enable(True)
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, o_out=O)
    torch.cuda.synchronize()
    prof = {p["name"]: p["launches"] for p in mg.muon_profile_read()}
    mg.muon_profile_enable(False)
    return W, M, O, prof


def _same(a, b, what):
    for i, (x, y) in enumerate(zip(a, b)):
        xv = x.contiguous().view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32)
        yv = y.contiguous().view(torch.int16 if y.dtype == torch.bfloat16 else torch.int32)
        nd = int((xv != yv).sum())
        assert nd == 0, f"{what}[{i}] {tuple(x.shape)}: {nd} elements differ"


@pytest.mark.parametrize("w_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("with_o", [True, False])
def test_fused_step_matches_unfused_bit_for_bit(w_dtype, with_o, monkeypatch):
    Wf, Mf, Of, pf = _step(SHAPES, w_dtype, True, monkeypatch, with_o=with_o)
    Wu, Mu, Ou, pu = _step(SHAPES, w_dtype, False, monkeypatch, with_o=with_o)
    assert pf.get("ns_gemm_final", 0) >= 1 and pf.get("unpack", 0) == 0
    assert pu.get("ns_gemm_final", 0) == 0 and pu.get("unpack", 0) >= 1
    _same(Wf, Wu, "W")
    _same(Mf, Mu, "M")
    if with_o:
        _same(Of, Ou, "O")


ALIGNED = [(256, 768), (768, 256), (296, 712), (712, 296), (512, 512), (200, 1032), (1032, 200), (1, 600),
           (600, 8), (264, 776), (776, 264)]


@pytest.mark.parametrize("w_dtype", [torch.bfloat16, torch.float32])
def test_fused_step_with_16_byte_rows(w_dtype, monkeypatch):
    Wf, Mf, Of, pf = _step(ALIGNED, w_dtype, True, monkeypatch, seed=6)
    Wu, Mu, Ou, _ = _step(ALIGNED, w_dtype, False, monkeypatch, seed=6)
    assert pf.get("ns_gemm_final", 0) >= 1 and pf.get("unpack", 0) == 0
    _same(Wf, Wu, "W")
    _same(Mf, Mu, "M")
    _same(Of, Ou, "O")


def test_fused_step_against_oracle(monkeypatch):
    shapes = [(300, 700), (700, 300), (260, 777)]
    W, G, M = _state(shapes, torch.bfloat16, 11)
    W0 = [bits(w) for w in W]
    G0 = [bits(g) for g in G]
    M0 = [f32(m) for m in M]
    O = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, o_out=O)
    torch.cuda.synchronize()
    for i, s in enumerate(shapes):
        _, M1, Oref = oracle.muon_step(W0[i], G0[i], M0[i], 0.02, 0.95, 0.1, w_bf16=True, g_bf16=True)
        assert np.array_equal(f32(M[i]).view(np.uint32), M1.view(np.uint32))
        assert_o_close(f32(O[i]), Oref, f"O {s}")
        dcy, sc = oracle.update_scalars(0.02, 0.1, *s)
        assert np.array_equal(bits(W[i]), oracle.weight_update(W0[i], f32(O[i]), dcy, sc, w_bf16=True))


def test_fused_ns_store_matches_unfused(monkeypatch):
    gen = torch.Generator(device=DEV).manual_seed(3)
    src = [torch.randn(s, generator=gen, device=DEV).to(torch.bfloat16) for s in SHAPES]
    out = {}
    for fused in (True, False):
        if fused:
            monkeypatch.delenv("MUON_NO_FUSED_UPDATE", raising=False)
        else:
            monkeypatch.setenv("MUON_NO_FUSED_UPDATE", "1")
        X = [t.clone() for t in src]
        mg.muon_ns5_batched(X)
        torch.cuda.synchronize()
        out[fused] = X
    _same(out[True], out[False], "O")


def test_more_than_eight_buckets(monkeypatch):
    # 10 padded shapes -> two GEMM launches per product, each with its own table
    shapes = [(r, k) for r in (200, 500) for k in (250, 500, 760, 1000, 1270)]
    shapes += [(k, r) for r, k in shapes[:3]]
    Wf, Mf, Of, pf = _step(shapes, torch.bfloat16, True, monkeypatch, seed=8)
    Wu, Mu, Ou, _ = _step(shapes, torch.bfloat16, False, monkeypatch, seed=8)
    assert pf["ns_gemm_final"] == 2
    _same(Wf, Wu, "W")
    _same(Of, Ou, "O")


def test_table_overflow_falls_back_to_separate_update(monkeypatch):
    # more tensor-core matrices in one launch than the fused kernel's table holds
    shapes = [(64, 128)] * 450 + [(128, 64)] * 2
    W, G, M = _state(shapes, torch.bfloat16, 9)
    sample = [0, 449, 450, 451]
    W0 = {i: bits(W[i]) for i in sample}
    G0 = {i: bits(G[i]) for i in sample}
    M0 = {i: f32(M[i]) for i in sample}
    O = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_profile_enable(True)
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, o_out=O)
    torch.cuda.synchronize()
    prof = {p["name"]: p["launches"] for p in mg.muon_profile_read()}
    mg.muon_profile_enable(False)
    assert prof.get("ns_gemm_final", 0) == 0 and prof["unpack"] >= 1
    for i in sample:
        _, M1, Oref = oracle.muon_step(W0[i], G0[i], M0[i], 0.02, 0.95, 0.1, w_bf16=True, g_bf16=True)
        assert np.array_equal(f32(M[i]).view(np.uint32), M1.view(np.uint32))
        assert_o_close(f32(O[i]), Oref, f"O[{i}]")
        dcy, sc = oracle.update_scalars(0.02, 0.1, *shapes[i])
        assert np.array_equal(bits(W[i]), oracle.weight_update(W0[i], f32(O[i]), dcy, sc, w_bf16=True))
