"""Behaviour of the C ABI on the GPU: failure injection on the host, caller
workspace, checkpoint / resume, streams, degenerate inputs, host-buffer steps."""
import ctypes

import numpy as np
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
import oracle
from muon_newton_schulz_step_gb300 import workloads as wl
from tests.gpu_util import assert_o_close, bits, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(shapes, seed, w_dtype=torch.bfloat16):
    g = torch.Generator(device=DEV).manual_seed(seed)
    W = [(0.02 * torch.randn(s, generator=g, device=DEV)).to(w_dtype) for s in shapes]
    G = [(1e-2 * torch.randn(s, generator=g, device=DEV)).to(torch.bfloat16) for s in shapes]
    M = [1e-3 * torch.randn(s, generator=g, device=DEV) for s in shapes]
    return W, G, M


def test_injected_allocation_failure_enqueues_nothing(monkeypatch):
    shapes = [(512, 1024), (1024, 512)]
    W, G, M = _inputs(shapes, 1)
    W0, M0 = [w.clone() for w in W], [m.clone() for m in M]
    torch.cuda.synchronize()
    mg.muon_release_workspace()
    monkeypatch.setenv("MUON_FAULT_INJECT", "alloc")
    with pytest.raises(mg.MuonError) as e:
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1)
    assert e.value.status == 4 and "injected" in str(e.value)
    torch.cuda.synchronize()
    for a, b in zip(W + M, W0 + M0):
        assert torch.equal(a, b)
    monkeypatch.delenv("MUON_FAULT_INJECT")
    mg.muon_step(W, G, M, 0.02, 0.95, 0.1)        # recovers once allocation works
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0


def test_caller_workspace_matches_library_workspace():
    shapes = [(300, 700), (700, 300), (512, 512)]
    Wa, Ga, Ma = _inputs(shapes, 2)
    Wb, Gb, Mb = [t.clone() for t in Wa], [t.clone() for t in Ga], [t.clone() for t in Ma]
    nbytes = mg.muon_workspace_bytes(shapes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    mg.muon_step_ex(Wa, Ga, Ma, 0.02, 0.95, 0.1, workspace=ws)
    mg.muon_step_ex(Wb, Gb, Mb, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    for a, b in zip(Wa + Ma, Wb + Mb):
        assert torch.equal(a, b)
    # a workspace that cannot hold even one of the matrices is rejected up front
    tiny = torch.empty(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(mg.MuonError) as e:
        mg.muon_step_ex(Wa, Ga, Ma, 0.02, 0.95, 0.1, workspace=tiny)
    assert e.value.status == 4


def test_library_workspace_falls_back_to_groups_when_allocation_fails(monkeypatch):
    # allocations above a third of what the batch needs fail (injected on the
    # host): the library retries with smaller groups and gets the same results
    shapes = [(512, 1536), (1536, 512), (300, 700), (64, 256), (700, 300), (512, 512), (96, 200)]
    Wa, Ga, Ma = _inputs(shapes, 16)
    Wb, Gb, Mb = [t.clone() for t in Wa], [t.clone() for t in Ga], [t.clone() for t in Ma]
    mg.muon_step(Wa, Ga, Ma, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    mg.muon_release_workspace()
    monkeypatch.setenv("MUON_FAULT_INJECT", f"alloc>{mg.muon_workspace_bytes(shapes) // 3}")
    mg.muon_step(Wb, Gb, Mb, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    monkeypatch.delenv("MUON_FAULT_INJECT")
    assert mg.muon_device_status() == 0
    for a, b in zip(Wa, Wb):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(Ma, Mb):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    mg.muon_release_workspace()


def test_small_caller_workspace_runs_the_batch_in_groups():
    # a workspace for about a third of the batch: the library runs consecutive
    # groups that fit, with results identical to one call on its own workspace
    shapes = [(512, 1536), (1536, 512), (300, 700), (64, 256), (700, 300), (512, 512), (96, 200)]
    Wa, Ga, Ma = _inputs(shapes, 15)
    Wb, Gb, Mb = [t.clone() for t in Wa], [t.clone() for t in Ga], [t.clone() for t in Ma]
    need = mg.muon_workspace_bytes(shapes)
    ws = torch.empty(need // 3 + 4096, dtype=torch.uint8, device=DEV)
    Oa = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    Ob = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step_ex(Wa, Ga, Ma, 0.02, 0.95, 0.1, o_out=Oa)
    mg.muon_step_ex(Wb, Gb, Mb, 0.02, 0.95, 0.1, o_out=Ob, workspace=ws)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0
    for a, b in zip(Wa + Oa, Wb + Ob):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(Ma, Mb):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_checkpoint_resume_is_bit_exact():
    shapes = [(384, 1280), (1280, 384), (64, 256)]
    W, G, M = _inputs(shapes, 3)
    Wr, Gr, Mr = [t.clone() for t in W], [t.clone() for t in G], [t.clone() for t in M]
    for _ in range(2):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1)
    # interrupted run: one step, state to the host, reload into fresh buffers, one more step
    mg.muon_step(Wr, Gr, Mr, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    saved = [(w.cpu(), m.cpu()) for w, m in zip(Wr, Mr)]
    del Wr, Mr
    torch.cuda.empty_cache()
    Wr = [w.to(DEV) for w, _ in saved]
    Mr = [m.to(DEV) for _, m in saved]
    mg.muon_step(Wr, Gr, Mr, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    for a, b in zip(W + M, Wr + Mr):
        assert torch.equal(a, b)


def test_side_stream_and_stream_switching():
    shapes = [(256, 768), (768, 256)]
    W, G, M = _inputs(shapes, 4)
    Wr, Gr, Mr = [t.clone() for t in W], [t.clone() for t in G], [t.clone() for t in M]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1, stream=s1)
    with torch.cuda.stream(s2):   # the library orders its shared workspace across streams
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1, stream=s2)
    torch.cuda.synchronize()
    for _ in range(2):
        mg.muon_step(Wr, Gr, Mr, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    for a, b in zip(W + M, Wr + Mr):
        assert torch.equal(a, b)


@pytest.mark.parametrize("path", ["tensor_core", "small"])
def test_zero_gradient_and_zero_lr(path, monkeypatch):
    if path == "tensor_core":
        monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    shapes = [(128, 384), (384, 128)]
    W, _, _ = _inputs(shapes, 5)
    G = [torch.zeros(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    M = [torch.zeros(s, dtype=torch.float32, device=DEV) for s in shapes]
    W0 = [w.clone() for w in W]
    O = [torch.full(s, 7.0, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, o_out=O)
    torch.cuda.synchronize()
    for i, s in enumerate(shapes):
        assert torch.count_nonzero(O[i]) == 0                       # zero matrix -> O = 0
        assert torch.count_nonzero(M[i]) == 0
        dcy, sc = oracle.update_scalars(0.02, 0.1, *s)               # W only decays
        assert np.array_equal(bits(W[i]), oracle.weight_update(bits(W0[i]), f32(O[i]), dcy, sc, w_bf16=True))
    # lr = 0 leaves W bit-exact
    W1 = [w.clone() for w in W]
    G2 = [torch.ones(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step(W, G2, M, 0.0, 0.95, 0.1)
    torch.cuda.synchronize()
    for a, b in zip(W, W1):
        assert torch.equal(a, b)


def test_profile_counters_and_launch_counts():
    shapes = [(512, 1024)] * 3 + [(64, 256)] * 2
    W, G, M = _inputs(shapes, 6)
    mg.muon_profile_enable(True)
    mg.muon_step(W, G, M, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    prof = {p["name"]: p for p in mg.muon_profile_read()}
    mg.muon_profile_enable(False)
    # the last update carries the weight update (fused epilogue)
    assert prof["ns_gemm_gram"]["launches"] == 5 and prof["ns_gemm_update"]["launches"] == 4
    assert prof["ns_gemm_final"]["launches"] == 1 and prof["unpack"]["launches"] == 1   # small ones
    assert prof["ns_small"]["launches"] == 1 and prof["norm_pass"]["launches"] == 1
    assert prof["ns_gemm_gram"]["flops"] == pytest.approx(5 * 3 * 2.0 * 512 * 512 * 1024)
    assert all(p["total_ms"] >= 0 for p in prof.values())


def test_many_matrices_span_several_chunks():
    # more matrices than one elementwise launch and one small-path launch take
    shapes = [(8, 40)] * 530 + [(40, 8)] * 10
    rng = np.random.default_rng(7)
    hosts = [oracle.bf16_rne(rng.standard_normal(s).astype(np.float32)) for s in shapes]
    mats = [torch.from_numpy(oracle.bf16_to_f32(h)).to(DEV).to(torch.bfloat16) for h in hosts]
    mg.muon_ns5_batched(mats, steps=5)
    torch.cuda.synchronize()
    for i in (0, 223, 224, 511, 512, 529, 530, 539):
        assert_o_close(f32(mats[i]), oracle.ns(oracle.bf16_to_f32(hosts[i]), steps=5), f"matrix {i}")


def test_host_buffer_step_matches_device_step_over_several_chunks():
    # 24 matrices of 2048 x 6144 hold ~2.4 GB of W + G + M: three staging chunks
    shapes = [(2048, 6144)] * 16 + [(6144, 2048)] * 8
    W, G, M = _inputs(shapes, 8)
    hW = [t.cpu().pin_memory() for t in W]
    hG = [t.cpu().pin_memory() for t in G]
    hM = [t.cpu().pin_memory() for t in M]
    torch.cuda.synchronize()
    for _ in range(2):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1)
        mg.muon_step_host(hW, hG, hM, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    for d, h in zip(W + M, hW + hM):
        assert torch.equal(d.cpu(), h)


def test_host_buffer_step_rejects_unpinned_memory():
    W = [torch.zeros((64, 64), dtype=torch.bfloat16)]
    G = [torch.zeros((64, 64), dtype=torch.bfloat16).pin_memory()]
    M = [torch.zeros((64, 64), dtype=torch.float32).pin_memory()]
    L = mg.lib()
    o = mg._Opts()
    L.muon_step_opts_init(o)
    rows = (ctypes.c_int * 1)(64)
    cols = (ctypes.c_int * 1)(64)
    rc = L.muon_step_host(mg._ptr_array(W), mg._ptr_array(G), mg._ptr_array(M), rows, cols, 1,
                          0.02, 0.95, 0.1, ctypes.byref(o), None)
    assert rc == 1 and b"pinned" in L.muon_last_error()


def test_cuda_graph_capture_replays_the_step():
    shapes = [(512, 1536), (1536, 512), (64, 256)]
    W, G, M = _inputs(shapes, 9)
    Wr, Gr, Mr = [t.clone() for t in W], [t.clone() for t in G], [t.clone() for t in M]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1, stream=s)    # outside the capture: creates the workspace
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1, stream=s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for _ in range(4):
        mg.muon_step(Wr, Gr, Mr, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    for a, b in zip(W + M, Wr + Mr):
        assert torch.equal(a, b)


def test_expired_device_wait_reports_timeout_and_the_context_survives(monkeypatch):
    # MUON_TEST_STALL: the first tensor-core launch issues no MMA, so its bounded
    # waits (50 ms in that launch) run out; the kernel records MUON_ERR_TIMEOUT,
    # drains its copies, frees TMEM and returns -- no fault, no hang
    monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    shapes = [(256, 512), (512, 256)]
    W, G, M = _inputs(shapes, 12)
    assert mg.muon_device_status() == 0
    monkeypatch.setenv("MUON_TEST_STALL", "1")
    mg.muon_step(W, G, M, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 5   # MUON_ERR_TIMEOUT
    assert mg.muon_device_status() == 0   # reading clears it
    # the context is still usable: a normal step matches the oracle
    monkeypatch.delenv("MUON_TEST_STALL")
    W, G, M = _inputs(shapes, 13)
    W0, G0, M0 = [bits(w) for w in W], [bits(g) for g in G], [f32(m) for m in M]
    O = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, o_out=O)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0
    for i, s in enumerate(shapes):
        _, M1, Oref = oracle.muon_step(W0[i], G0[i], M0[i], 0.02, 0.95, 0.1, w_bf16=True, g_bf16=True)
        assert np.array_equal(f32(M[i]).view(np.uint32), M1.view(np.uint32))
        assert_o_close(f32(O[i]), Oref, f"O {s}")


def test_cuda_graph_capture_of_a_split_batch(monkeypatch):
    # 6 x 2048x6144 exceed the split threshold: the capture records the fork to the
    # library's side stream and the join back through events
    monkeypatch.delenv("MUON_NO_SPLIT", raising=False)
    shapes = [(2048, 6144)] * 4 + [(6144, 2048)] * 2
    W, G, M = _inputs(shapes, 14)
    Wr, Gr, Mr = [t.clone() for t in W], [t.clone() for t in G], [t.clone() for t in M]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1, stream=s)    # outside the capture: creates the workspace
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        mg.muon_step(W, G, M, 0.02, 0.95, 0.1, stream=s)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for _ in range(3):
        mg.muon_step(Wr, Gr, Mr, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0
    for a, b in zip(W + M, Wr + Mr):
        assert torch.equal(a, b)


def test_calls_from_two_host_threads_on_two_streams():
    # the library serialises calls from several host threads internally; each
    # thread steps its own batch on its own stream, results as if sequential
    import threading
    shapes_a = [(512, 1536), (1536, 512), (64, 256)]
    shapes_b = [(300, 700), (700, 300), (96, 200)]
    A = _inputs(shapes_a, 17)
    B = _inputs(shapes_b, 18)
    Ar = [[t.clone() for t in group] for group in A]
    Br = [[t.clone() for t in group] for group in B]
    errors = []

    def worker(W, G, M):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.default_stream())
            with torch.cuda.stream(s):
                for _ in range(3):
                    mg.muon_step(W, G, M, 0.02, 0.95, 0.1, stream=s)
            s.synchronize()
        except Exception as e:   # surfaced in the main thread
            errors.append(e)

    torch.cuda.synchronize()
    threads = [threading.Thread(target=worker, args=tuple(A)), threading.Thread(target=worker, args=tuple(B))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for _ in range(3):
        mg.muon_step(*Ar, 0.02, 0.95, 0.1)
        mg.muon_step(*Br, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0
    for got, want in ((A, Ar), (B, Br)):
        for a, b in zip(got[0] + got[2], want[0] + want[2]):
            assert torch.equal(a, b)
