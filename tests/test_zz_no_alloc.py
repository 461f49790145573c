"""muon_ns5_batched_static: Newton-Schulz for callers that cannot allocate
device memory (a framework allocator owns the device budget, a path cannot
take cudaMalloc's synchronisation, or the host fixes the library's memory).
Its scratch is one fixed device array inside the library.

Checked through the C ABI against muon_ns5_batched on the same inputs, on two
calls in a row (the second one reuses the array the first one left behind),
and directly against the oracle.  With every library workspace allocation made
to fail (MUON_FAULT_INJECT=alloc), the allocating call fails and this one still
runs.  The library's two-stream split needs at least 2 TFLOP of work per call,
more than a batch that fits in the 64 MiB scratch can hold, so this entry point
always runs on the caller's stream alone.
This file is collected last so that a run stopping at the first failure has
already run every other test; it passes alone in a fresh process too.
"""
import ctypes

import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
import oracle
from tests.gpu_util import assert_o_close, bits, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
# small-path shapes and tensor-core shapes, ragged, tall and wide
SHAPES = [(64, 256), (256, 64), (7, 13), (512, 1024), (1024, 512), (300, 700)]


def _call_static(mats, steps=5):
    L = mg.lib()
    n = len(mats)
    ptrs = (ctypes.c_void_p * n)(*[m.data_ptr() for m in mats])
    rows = (ctypes.c_int * n)(*[int(m.shape[0]) for m in mats])
    cols = (ctypes.c_int * n)(*[int(m.shape[1]) for m in mats])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.muon_ns5_batched_static(ptrs, rows, cols, n, steps, None, stream)


def test_static_entry_point_matches_the_allocating_one_on_two_calls():
    assert mg.muon_workspace_bytes(SHAPES) <= mg.MUON_STATIC_SCRATCH_BYTES
    g = torch.Generator(device=DEV).manual_seed(77)
    for call in range(2):
        inputs = [torch.randn(s, generator=g, device=DEV).to(torch.bfloat16) for s in SHAPES]
        host = [bits(x) for x in inputs]
        got = [x.clone() for x in inputs]
        ref = [x.clone() for x in inputs]
        rc = _call_static(got)
        assert rc == 0, mg.lib().muon_last_error().decode()
        mg.muon_ns5_batched(ref)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(got, ref)):
            assert_o_close(f32(a), f32(b), f"call {call}, matrix {i} {tuple(a.shape)}")
            assert torch.equal(a, b), f"call {call}, matrix {i}: same kernels should give the same bits"
            # and first-hand against the oracle, at the parity contract
            assert_o_close(f32(a), oracle.ns(oracle.bf16_to_f32(host[i]), 5), f"oracle, call {call}, matrix {i}")
    assert mg.muon_device_status() == 0


def test_static_entry_point_allocates_no_device_memory():
    x = [torch.randn(s, device=DEV).to(torch.bfloat16) for s in SHAPES]
    assert _call_static(x) == 0                       # first call: per-device set-up
    torch.cuda.synchronize()
    mg.muon_release_workspace()                       # no library workspace left behind
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call_static(x) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    need = mg.muon_workspace_bytes(SHAPES)
    assert free0 - free1 < need // 4, (free0 - free1, need)


def test_static_entry_point_runs_when_every_workspace_allocation_fails(monkeypatch):
    g = torch.Generator(device=DEV).manual_seed(78)
    x = [torch.randn(s, generator=g, device=DEV).to(torch.bfloat16) for s in SHAPES]
    want = [t.clone() for t in x]
    mg.muon_ns5_batched(want)
    torch.cuda.synchronize()
    mg.muon_release_workspace()
    torch.cuda.synchronize()
    monkeypatch.setenv("MUON_FAULT_INJECT", "alloc")
    # the allocating entry point now fails: it has no workspace and may get none
    y = [t.clone() for t in x]
    L = mg.lib()
    n = len(y)
    rc = L.muon_ns5_batched((ctypes.c_void_p * n)(*[t.data_ptr() for t in y]),
                            (ctypes.c_int * n)(*[int(t.shape[0]) for t in y]),
                            (ctypes.c_int * n)(*[int(t.shape[1]) for t in y]), n, 5, None,
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 4, rc
    # the static one makes no allocation, so it still runs, with the same bits
    for _ in range(2):
        z = [t.clone() for t in x]
        assert _call_static(z) == 0, mg.lib().muon_last_error().decode()
        torch.cuda.synchronize()
        for a, b in zip(z, want):
            assert torch.equal(a, b)
    monkeypatch.delenv("MUON_FAULT_INJECT")
    assert mg.muon_device_status() == 0


def test_static_entry_point_rejects_batches_beyond_its_scratch():
    x = torch.zeros((2048, 6144), dtype=torch.bfloat16, device=DEV)
    assert mg.muon_workspace_bytes([tuple(x.shape)]) > mg.MUON_STATIC_SCRATCH_BYTES
    rc = _call_static([x])
    assert rc == 2
    assert b"MUON_STATIC_SCRATCH_BYTES" in mg.lib().muon_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(x) == 0               # nothing was enqueued
