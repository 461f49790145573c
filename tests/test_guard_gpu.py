"""Out-of-bounds writes into caller memory, checked with guard regions.

Every caller matrix (W, G, M and the optional O copy) is the head of a larger
buffer whose tail holds a fixed bit pattern; after the call the tails must be
unchanged.  Shapes cover both orientations, widths that are and are not
multiples of 8 (vector and scalar stores), single rows and columns, padded tile
edges, fp32 weights, the small-matrix path and the tensor-core path with the
fused final update and with the separate weight-update kernel.
"""
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096                      # elements after each matrix
PATTERN = 0x5A5A5A5A              # as int32 words


SHAPES = [(64, 256), (256, 64), (300, 700), (700, 300), (257, 513), (513, 257), (1, 600), (600, 1),
          (33, 65), (128, 384), (260, 777), (777, 260)]


def _guarded(shape, dtype, fill):
    rows, cols = shape
    n = rows * cols
    esz = torch.tensor([], dtype=dtype).element_size()
    words = (n * esz + GUARD * esz + 3) // 4
    raw = torch.full((words,), PATTERN, dtype=torch.int32, device=DEV)
    buf = raw.view(dtype)
    head = buf[:n].view(rows, cols)
    head.copy_(fill.to(dtype))
    return raw, head, n * esz


def _tail_intact(raw, head_bytes):
    b = raw.view(torch.uint8)
    start = (head_bytes + 3) // 4 * 4          # first whole guard word
    gap = b[head_bytes:start]                   # bytes between the matrix and the first guard word
    tail = raw[start // 4:]
    return bool((tail == PATTERN).all()) and bool((gap == 0x5A).all())


@pytest.mark.parametrize("route", ["small", "tensor_core_fused", "tensor_core_separate"])
@pytest.mark.parametrize("w_dtype", [torch.bfloat16, torch.float32])
def test_step_writes_nothing_past_caller_buffers(route, w_dtype, monkeypatch):
    if route == "small":
        monkeypatch.delenv("MUON_DISABLE_SMALL_NS", raising=False)
    else:
        monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    if route == "tensor_core_separate":
        monkeypatch.setenv("MUON_NO_FUSED_UPDATE", "1")
    else:
        monkeypatch.delenv("MUON_NO_FUSED_UPDATE", raising=False)
    gen = torch.Generator(device=DEV).manual_seed(21)
    Ws, Gs, Ms, Os = [], [], [], []
    for s in SHAPES:
        Ws.append(_guarded(s, w_dtype, 0.02 * torch.randn(s, generator=gen, device=DEV)))
        Gs.append(_guarded(s, torch.bfloat16, torch.randn(s, generator=gen, device=DEV)))
        Ms.append(_guarded(s, torch.float32, 1e-3 * torch.randn(s, generator=gen, device=DEV)))
        Os.append(_guarded(s, torch.bfloat16, torch.zeros(s, device=DEV)))
    mg.muon_step_ex([w[1] for w in Ws], [g[1] for g in Gs], [m[1] for m in Ms], 0.02, 0.95, 0.1,
                    o_out=[o[1] for o in Os])
    torch.cuda.synchronize()
    for name, group in (("W", Ws), ("G", Gs), ("M", Ms), ("O", Os)):
        for s, (raw, _, nbytes) in zip(SHAPES, group):
            assert _tail_intact(raw, nbytes), f"{name} {s}: guard region overwritten"


@pytest.mark.parametrize("route", ["small", "tensor_core_fused", "tensor_core_separate"])
def test_ns_writes_nothing_past_caller_buffers(route, monkeypatch):
    if route == "small":
        monkeypatch.delenv("MUON_DISABLE_SMALL_NS", raising=False)
    else:
        monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    if route == "tensor_core_separate":
        monkeypatch.setenv("MUON_NO_FUSED_UPDATE", "1")
    else:
        monkeypatch.delenv("MUON_NO_FUSED_UPDATE", raising=False)
    gen = torch.Generator(device=DEV).manual_seed(22)
    Xs = [_guarded(s, torch.bfloat16, torch.randn(s, generator=gen, device=DEV)) for s in SHAPES]
    mg.muon_ns5_batched([x[1] for x in Xs])
    torch.cuda.synchronize()
    for s, (raw, _, nbytes) in zip(SHAPES, Xs):
        assert _tail_intact(raw, nbytes), f"{s}: guard region overwritten"


GUARD_SHAPES = [(64, 256), (256, 64), (300, 700), (700, 300), (257, 513), (1, 600), (33, 65), (128, 384)]


def _step_copy(shapes, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W = [(0.02 * torch.randn(s, generator=gen, device=DEV)).to(torch.bfloat16) for s in shapes]
    G = [torch.randn(s, generator=gen, device=DEV).to(torch.bfloat16) for s in shapes]
    M = [1e-3 * torch.randn(s, generator=gen, device=DEV) for s in shapes]
    mg.muon_step(W, G, M, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    return W, M


@pytest.mark.parametrize("shapes", [GUARD_SHAPES, [(2048, 6144)] * 4 + [(6144, 2048)] * 2],
                         ids=["ragged", "two-stream split"])
def test_workspace_guard_regions_stay_intact(shapes, monkeypatch):
    # MUON_DEBUG_GUARD=1: guard regions around every workspace region, filled
    # before the first kernel of a call and checked after the last one
    monkeypatch.delenv("MUON_DEBUG_GUARD", raising=False)
    W0, M0 = _step_copy(shapes, 31)
    assert mg.muon_device_status() == 0
    monkeypatch.setenv("MUON_DEBUG_GUARD", "1")
    W1, M1 = _step_copy(shapes, 31)
    assert mg.muon_device_status() == 0
    for a, b in zip(W0 + M0, W1 + M1):   # the layout change does not change the result
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def test_workspace_guard_check_reports_an_overwritten_guard(monkeypatch):
    # "poison": the library clears one guard byte right after filling the guards,
    # so the check at the end of the call must report MUON_ERR_CORRUPT
    monkeypatch.setenv("MUON_DEBUG_GUARD", "poison")
    _step_copy(GUARD_SHAPES, 32)
    assert mg.muon_device_status() == 6   # MUON_ERR_CORRUPT
    assert mg.muon_device_status() == 0
    monkeypatch.setenv("MUON_DEBUG_GUARD", "1")
    _step_copy(GUARD_SHAPES, 32)
    assert mg.muon_device_status() == 0
