"""Alternative launch forms of the Newton-Schulz products give the same bits.

MUON_GEMM_MULTICAST=1 runs the update products (plain and fused final) on
clusters of two CTA pairs that load the A operand once and multicast it
(tiles beyond an odd number of tile columns are computed and discarded);
MUON_GEMM_NO_TMA_EPI=1 gives the plain update its register epilogue instead
of the TMA one.  MUON_GEMM_MIRROR=1 stores the symmetric products (A = X X^T
and B = b A + c A A) in full, where by default only their tiles with
tm <= tn are stored and the polynomial and the update read the K blocks left
of a row tile's diagonal as MN-major blocks of the stored transpose.  Every
output element is the same sum in the same order in all forms, so W, M and O
must match the default bit for bit.
"""
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg

pytestmark = pytest.mark.gpu
DEV = "cuda"

# odd and even numbers of 256-wide tile columns, both orientations, ragged edges
SHAPES = [(256, 768), (768, 256), (512, 1024), (300, 1300), (1300, 300), (1024, 2048)]


def _step(monkeypatch, env, w_dtype, fp8=False):
    for var in ("MUON_GEMM_MULTICAST", "MUON_GEMM_NO_TMA_EPI", "MUON_GEMM_MIRROR", "MUON_DISABLE_SMALL_NS",
                "MUON_NO_FUSED_UPDATE"):
        monkeypatch.delenv(var, raising=False)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    gen = torch.Generator(device=DEV).manual_seed(17)
    W = [(0.02 * torch.randn(s, generator=gen, device=DEV)).to(w_dtype) for s in SHAPES]
    G = [torch.randn(s, generator=gen, device=DEV).to(torch.bfloat16) for s in SHAPES]
    M = [1e-3 * torch.randn(s, generator=gen, device=DEV) for s in SHAPES]
    O = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in SHAPES]
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, o_out=O, fp8_gram=fp8)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0
    return W, M, O


@pytest.mark.parametrize("env", [{"MUON_GEMM_MULTICAST": "1"}, {"MUON_GEMM_NO_TMA_EPI": "1"},
                                 {"MUON_GEMM_MIRROR": "1"}],
                         ids=["multicast", "register_epilogue", "full_symmetric_storage"])
@pytest.mark.parametrize("w_dtype", [torch.bfloat16, torch.float32])
def test_launch_forms_are_bit_identical(env, w_dtype, monkeypatch):
    ref = _step(monkeypatch, {}, w_dtype)
    alt = _step(monkeypatch, env, w_dtype)
    for name, a, b in zip(("W", "M", "O"), ref, alt):
        for i, (x, y) in enumerate(zip(a, b)):
            assert torch.equal(x, y), f"{name}[{i}] {tuple(x.shape)}"


def test_full_symmetric_storage_is_bit_identical_with_the_fp8_gram(monkeypatch):
    ref = _step(monkeypatch, {}, torch.bfloat16, fp8=True)
    alt = _step(monkeypatch, {"MUON_GEMM_MIRROR": "1"}, torch.bfloat16, fp8=True)
    for name, a, b in zip(("W", "M", "O"), ref, alt):
        for i, (x, y) in enumerate(zip(a, b)):
            assert torch.equal(x, y), f"{name}[{i}] {tuple(x.shape)}"


@pytest.mark.parametrize("env", [{"MUON_GEMM_MIRROR": "1"}, {"MUON_GEMM_MULTICAST": "1"}],
                         ids=["full_symmetric_storage", "multicast"])
def test_newton_schulz_only_call_is_bit_identical(env, monkeypatch):
    """The Newton-Schulz-only entry point (its last update stores O in place of the input)."""
    def run(e):
        for var in ("MUON_GEMM_MULTICAST", "MUON_GEMM_NO_TMA_EPI", "MUON_GEMM_MIRROR", "MUON_DISABLE_SMALL_NS"):
            monkeypatch.delenv(var, raising=False)
        for k, v in e.items():
            monkeypatch.setenv(k, v)
        gen = torch.Generator(device=DEV).manual_seed(23)
        X = [torch.randn(s, generator=gen, device=DEV).to(torch.bfloat16) for s in SHAPES]
        mg.muon_ns5_batched(X)
        torch.cuda.synchronize()
        assert mg.muon_device_status() == 0
        return X
    ref, alt = run({}), run(env)
    for i, (x, y) in enumerate(zip(ref, alt)):
        assert torch.equal(x, y), f"X[{i}] {tuple(x.shape)}"
