"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Tolerances: O within relative Frobenius error 1e-2 and per-element absolute
error 2e-2 of the oracle; the momentum bit-exact; W bit-exact given the GPU's
O.  Where all arithmetic is exact (power-of-two data and coefficients, whose
fp32 sums carry no rounding), the GPU must match the oracle bit for bit,
which pins the tile indexing, the symmetric mirroring, orientation and the
MN-major operand of the update product.
"""
import numpy as np
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
import oracle
from muon_newton_schulz_step_gb300 import workloads as wl
from tests.conditioning import bound_for, order_spread
from tests.gpu_util import assert_o_close, bits, compare_o, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(params=["tensor_core", "small", "small_one_cta"])
def path(request, monkeypatch):
    """Run a test through the tcgen05 pair-CTA kernel (small path disabled), or
    with the default routing, where matrices that fit in shared memory take the
    small-matrix kernel: on a cluster of CTAs per matrix (default) or one CTA per
    matrix (its fallback)."""
    monkeypatch.delenv("MUON_SMALL_NO_CLUSTER", raising=False)
    if request.param == "tensor_core":
        monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    else:
        monkeypatch.delenv("MUON_DISABLE_SMALL_NS", raising=False)
        if request.param == "small_one_cta":
            monkeypatch.setenv("MUON_SMALL_NO_CLUSTER", "1")
    return request.param


def _ternary(m, n, nnz, seed):
    """m x n fp32 matrix with `nnz` entries of +-1 (others 0): its norm is
    sqrt(nnz), so for nnz = 256 the normalisation scale is exactly 1/16."""
    rng = np.random.default_rng(seed)
    U = np.zeros(m * n, dtype=np.float32)
    pos = rng.choice(m * n, size=nnz, replace=False)
    U[pos] = rng.choice([-1.0, 1.0], size=nnz)
    return U.reshape(m, n)


def _gpu_ns(U32, steps, coeffs=None):
    X = torch.from_numpy(U32).to(DEV).to(torch.bfloat16)
    mg.muon_ns5_batched([X], steps=steps, coeffs=coeffs)
    torch.cuda.synchronize()
    return X


@pytest.mark.parametrize("shape", [(64, 256), (256, 64), (300, 200), (512, 768), (256, 1024), (1, 300),
                                   (300, 1)])
@pytest.mark.parametrize("coeffs", [(0.0, 1.0, 0.0), (0.5, 0.25, 1.0), (1.0, 0.0, 0.0)])
def test_ns_one_step_bit_exact_on_exact_data(shape, coeffs, path):
    m, n = shape
    nnz = min(256, m * n)
    U = _ternary(m, n, nnz, seed=m * 7 + n)
    X = _gpu_ns(U, 1, coeffs)
    ref = oracle.ns_bf16_bits(oracle.bf16_rne(U), steps=1, coeffs=coeffs)
    got = bits(X)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} of {got.size} elements differ"


@pytest.mark.parametrize("shape", [(64, 256), (384, 640), (640, 384), (7, 13), (1, 1), (1000, 3)])
def test_ns_identity_coefficients_leave_x0(shape, path):
    m, n = shape
    rng = np.random.default_rng(sum(shape))
    U = rng.standard_normal(shape).astype(np.float32)
    X0 = bits(_gpu_ns(U, 0))
    X3 = bits(_gpu_ns(U, 3, (1.0, 0.0, 0.0)))
    assert np.array_equal(X0, X3)
    # X0 = bf16(U * sigma): identical to the oracle unless the two norms round sigma differently
    ref = oracle.ns_bf16_bits(oracle.bf16_rne(U), steps=0)
    diff = np.abs(X0.astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3


@pytest.mark.parametrize("shape", [(64, 256), (256, 64), (128, 128), (300, 500), (500, 300), (7, 13),
                                   (1, 1000), (1000, 1), (257, 513), (1024, 3072), (32768, 256)])
def test_ns5_parity_against_oracle(shape, path):
    rng = np.random.default_rng(shape[0] * 31 + shape[1])
    m, n = shape
    r = min(m, n)
    # spectrum spread over [1e-2, 1] plus a small noise floor
    Uf, _ = np.linalg.qr(rng.standard_normal((m, r)))
    Vf, _ = np.linalg.qr(rng.standard_normal((n, r)))
    s = np.exp(rng.uniform(np.log(1e-2), 0, r))
    G = ((Uf * s) @ Vf.T + 1e-3 * rng.standard_normal((m, n))).astype(np.float32)
    Gb = oracle.bf16_rne(G)
    X = torch.from_numpy(oracle.bf16_to_f32(Gb)).to(DEV).to(torch.bfloat16)
    mg.muon_ns5_batched([X], steps=5)
    torch.cuda.synchronize()
    ref = oracle.ns(oracle.bf16_to_f32(Gb), steps=5)
    assert_o_close(f32(X), ref, f"{shape}")


def test_ns5_ragged_batch_in_one_call(path):
    shapes = [(64, 256), (256, 64), (300, 500), (500, 300), (7, 13), (128, 384), (64, 256), (1, 77)]
    rng = np.random.default_rng(5)
    hosts = [oracle.bf16_rne(rng.standard_normal(s).astype(np.float32)) for s in shapes]
    mats = [torch.from_numpy(oracle.bf16_to_f32(h)).to(DEV).to(torch.bfloat16) for h in hosts]
    mg.muon_ns5_batched(mats, steps=5)
    torch.cuda.synchronize()
    for h, X, s in zip(hosts, mats, shapes):
        ref = oracle.ns(oracle.bf16_to_f32(h), steps=5)
        assert_o_close(f32(X), ref, f"{s}")


@pytest.mark.parametrize("route", ["tensor_core", "default"])
def test_longest_side_at_the_dimension_limit(route, monkeypatch):
    # one side at MUON_MAX_DIM (32768): the widest TMA coordinates, tile counts and
    # padding of the oriented iterate, with a short side small enough for the oracle
    if route == "tensor_core":
        monkeypatch.setenv("MUON_DISABLE_SMALL_NS", "1")
    else:
        monkeypatch.delenv("MUON_DISABLE_SMALL_NS", raising=False)
    shapes = [(1, 32768), (32768, 3), (2, 32767), (40, 32768)]
    rng = np.random.default_rng(9)
    hosts = [oracle.bf16_rne(rng.standard_normal(s).astype(np.float32)) for s in shapes]
    mats = [torch.from_numpy(oracle.bf16_to_f32(h)).to(DEV).to(torch.bfloat16) for h in hosts]
    mg.muon_ns5_batched(mats, steps=5)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0
    for h, X, s in zip(hosts, mats, shapes):
        ref = oracle.ns(oracle.bf16_to_f32(h), steps=5)
        assert_o_close(f32(X), ref, f"{s}")


@pytest.mark.parametrize("shape", [(64, 256), (256, 64), (100, 300), (7, 13), (128, 256)])
def test_small_path_five_steps_bit_exact(shape, monkeypatch):
    """The shared-memory path sums in the oracle's order: with an exactly
    representable X0 (norm 16), all five default-coefficient iterations are
    bit-identical to the oracle."""
    monkeypatch.delenv("MUON_DISABLE_SMALL_NS", raising=False)
    m, n = shape
    U = _ternary(m, n, min(256, m * n), seed=3 * m + n)
    if m * n < 256:
        pytest.skip("needs 256 non-zeros")
    X = _gpu_ns(U, 5)
    ref = oracle.ns_bf16_bits(oracle.bf16_rne(U), steps=5)
    got = bits(X)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} of {got.size} elements differ"


def _run_step(w, inp, **kw):
    O = [torch.empty(t.shape, dtype=torch.bfloat16, device=DEV) for t in inp["W"]]
    mg.muon_step_ex(inp["W"], inp["G"], inp["M"], w.lr, w.mu, w.wd, o_out=O, **kw)
    torch.cuda.synchronize()
    return O


def _check_step(w, host, inp, O, idx, w_bf16, g_bf16, by_conditioning=False):
    for j, i in enumerate(idx):
        W0, G0, M0 = host["W"][j], host["G"][j], host["M"][j]
        W1, M1, Oref = oracle.muon_step(W0, G0, M0, w.lr, w.mu, w.wd, w_bf16=w_bf16, g_bf16=g_bf16)
        assert np.array_equal(f32(inp["M"][i]).view(np.uint32), M1.view(np.uint32)), f"M of matrix {i}"
        Og = f32(O[i])
        if by_conditioning:
            rel_b, abs_b, _ = bound_for(order_spread(
                lambda: oracle.muon_step(W0, G0, M0, w.lr, w.mu, w.wd, w_bf16=w_bf16, g_bf16=g_bf16)[2]))
            rel, mx = compare_o(Og, Oref)
            assert rel <= rel_b and mx <= abs_b, f"O of matrix {i}: rel {rel:.3e}, max {mx:.3e}"
        else:
            assert_o_close(Og, Oref, f"O of matrix {i}")
        dcy, s = oracle.update_scalars(w.lr, w.wd, *W0.shape)
        Wexp = oracle.weight_update(W0, Og, dcy, s, w_bf16=w_bf16)
        Wgot = bits(inp["W"][i]) if w_bf16 else f32(inp["W"][i]).view(np.uint32)
        Wexp = Wexp if w_bf16 else Wexp.view(np.uint32)
        assert np.array_equal(Wgot, Wexp), f"W of matrix {i}"


def _host_copy(w, inp, idx):
    def h(t):
        return bits(t) if t.dtype == torch.bfloat16 else f32(t).copy()
    return {k: [h(inp[k][i]) for i in idx] for k in ("W", "G", "M")}


def test_tiny_workload_full_step(path):
    """The 8 x 64x256 rank-4 workload.  With default routing these matrices
    take the shared-memory path, whose sums follow the oracle's order, and
    every matrix meets the contract.  Forced through the tensor cores (whose
    fp32 accumulation truncates), matrix 6 flips one bf16 rounding of its Gram
    product and O moves by about 1.6 %.  That matrix is ill-conditioned for the
    oracle itself: its two legal summation orders alone give O 1.6 % apart
    (tests/test_oracle_conditioning.py), so on the tensor-core routes it is
    held to the contract plus that spread (tests/conditioning.py); every other
    matrix, and M and W of all eight, are held to the normal bar."""
    w = wl.workload("tiny")
    inp = wl.make_inputs(w, DEV)
    idx = list(range(w.count))
    host = _host_copy(w, inp, idx)
    O = _run_step(w, inp)
    _check_step(w, host, inp, O, idx, w_bf16=False, g_bf16=False, by_conditioning=path == "tensor_core")
    assert mg.muon_device_status() == 0


def test_bf16_step_small_shapes_and_plain_momentum(path):
    shapes = [(96, 200), (200, 96), (256, 256), (33, 65)]
    rng = np.random.default_rng(9)
    W = [torch.from_numpy(rng.standard_normal(s).astype(np.float32) * 0.02).to(DEV).to(torch.bfloat16) for s in shapes]
    G = [torch.from_numpy(rng.standard_normal(s).astype(np.float32) * 1e-2).to(DEV).to(torch.bfloat16) for s in shapes]
    M = [torch.from_numpy(rng.standard_normal(s).astype(np.float32) * 1e-3).to(DEV) for s in shapes]
    inp = {"W": W, "G": G, "M": M}
    w = wl.Workload("small_bf16", 99, "step", [wl.MatrixSpec(*s, "none", 0) for s in shapes])
    for nesterov in (True, False):
        host = _host_copy(w, inp, range(len(shapes)))
        O = _run_step(w, inp, nesterov=nesterov)
        for j in range(len(shapes)):
            W1, M1, Oref = oracle.muon_step(host["W"][j], host["G"][j], host["M"][j], w.lr, w.mu, w.wd,
                                            w_bf16=True, g_bf16=True, nesterov=nesterov)
            assert np.array_equal(f32(inp["M"][j]).view(np.uint32), M1.view(np.uint32))
            assert_o_close(f32(O[j]), Oref, f"{shapes[j]} nesterov={nesterov}")


def test_determinism_two_runs_bit_identical(path):
    rng = np.random.default_rng(11)
    shapes = [(512, 1536), (1536, 512), (300, 700)]
    hosts = [rng.standard_normal(s).astype(np.float32) for s in shapes]
    outs = []
    for _ in range(2):
        mats = [torch.from_numpy(h).to(DEV).to(torch.bfloat16) for h in hosts]
        mg.muon_ns5_batched(mats, steps=5)
        torch.cuda.synchronize()
        outs.append([bits(x) for x in mats])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


SCHEDULE = [oracle.COEFFS] * 3 + [(2.0, -1.5, 0.5), (1.875, -1.25, 0.375)]


@pytest.mark.parametrize("shape", [(64, 256), (300, 700), (700, 300), (1024, 2048)])
def test_coefficient_schedule_parity(shape, path):
    rng = np.random.default_rng(sum(shape) + 5)
    G = oracle.bf16_rne(rng.standard_normal(shape).astype(np.float32))
    X = torch.from_numpy(oracle.bf16_to_f32(G)).to(DEV).to(torch.bfloat16)
    mg.muon_ns_batched_ex([X], steps=len(SCHEDULE), coeffs=SCHEDULE)
    torch.cuda.synchronize()
    assert_o_close(f32(X), oracle.ns_schedule(oracle.bf16_to_f32(G), SCHEDULE), f"{shape}")


@pytest.mark.parametrize("sched", [[(0.5, 0.25, 1.0), (1.0, 0.0, 0.0)], [(1.0, 0.0, 0.0), (0.5, 0.25, 1.0)]])
@pytest.mark.parametrize("shape", [(64, 256), (512, 768), (768, 512)])
def test_coefficient_schedule_bit_exact_on_exact_data(shape, sched, path):
    """Each iteration must use its own triple.  One triple is the identity
    (1, 0, 0), which leaves X exactly unchanged, and the other acts on the
    exactly representable X0, so every fp32 sum is exact in either order."""
    U = _ternary(*shape, 256, seed=11 * shape[0] + shape[1])
    X = torch.from_numpy(U).to(DEV).to(torch.bfloat16)
    mg.muon_ns_batched_ex([X], steps=2, coeffs=sched)
    torch.cuda.synchronize()
    ref = oracle.bf16_rne(oracle.ns_schedule(oracle.bf16_to_f32(oracle.bf16_rne(U)), sched))
    got = bits(X)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} of {got.size} elements differ"


def test_step_with_coefficient_schedule(path):
    shapes = [(256, 768), (768, 256), (96, 200)]
    rng = np.random.default_rng(31)
    W = [torch.from_numpy(rng.standard_normal(s).astype(np.float32) * 0.02).to(DEV).to(torch.bfloat16) for s in shapes]
    G = [torch.from_numpy(rng.standard_normal(s).astype(np.float32) * 1e-2).to(DEV).to(torch.bfloat16) for s in shapes]
    M = [torch.from_numpy(rng.standard_normal(s).astype(np.float32) * 1e-3).to(DEV) for s in shapes]
    host = {"W": [bits(t) for t in W], "G": [bits(t) for t in G], "M": [f32(t).copy() for t in M]}
    O = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, steps=len(SCHEDULE), coeffs=SCHEDULE, o_out=O)
    torch.cuda.synchronize()
    for j in range(len(shapes)):
        M1, U = oracle.momentum(oracle.bf16_to_f32(host["G"][j]), host["M"][j], 0.95)
        assert np.array_equal(f32(M[j]).view(np.uint32), M1.view(np.uint32))
        assert_o_close(f32(O[j]), oracle.ns_schedule(U, SCHEDULE), f"{shapes[j]}")


@pytest.mark.parametrize("g_dtype,K", [(torch.bfloat16, 3), (torch.float32, 2), (torch.bfloat16, 1)])
def test_stacked_gradients_summed_in_fp32(g_dtype, K, path):
    shapes = [(256, 768), (768, 256), (33, 65), (96, 200)]
    gen = torch.Generator(device=DEV).manual_seed(41 + K)
    W = [(0.02 * torch.randn(s, generator=gen, device=DEV)).to(torch.bfloat16) for s in shapes]
    G = [(1e-2 * torch.randn((K,) + s, generator=gen, device=DEV)).to(g_dtype) for s in shapes]
    if K == 1:
        G = [g[0] for g in G]          # plain 2-D gradients take the same path with g_count = 1
    M = [1e-3 * torch.randn(s, generator=gen, device=DEV) for s in shapes]
    g_bf16 = g_dtype == torch.bfloat16
    host = {"W": [bits(t) for t in W], "M": [f32(t).copy() for t in M],
            "G": [bits(t) if g_bf16 else f32(t).copy() for t in G]}
    O = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1, o_out=O)
    torch.cuda.synchronize()
    for j, s in enumerate(shapes):
        W1, M1, Oref = oracle.muon_step(host["W"][j], host["G"][j], host["M"][j], 0.02, 0.95, 0.1,
                                        w_bf16=True, g_bf16=g_bf16)
        assert np.array_equal(f32(M[j]).view(np.uint32), M1.view(np.uint32)), f"M of {s}"
        assert_o_close(f32(O[j]), Oref, f"{s}")
        dcy, sc = oracle.update_scalars(0.02, 0.1, *s)
        assert np.array_equal(bits(W[j]), oracle.weight_update(host["W"][j], f32(O[j]), dcy, sc, w_bf16=True))


def test_stacked_gradients_through_host_buffers():
    shapes = [(512, 1536), (1536, 512)]
    gen = torch.Generator(device=DEV).manual_seed(43)
    W = [(0.02 * torch.randn(s, generator=gen, device=DEV)).to(torch.bfloat16) for s in shapes]
    G = [(1e-2 * torch.randn((4,) + s, generator=gen, device=DEV)).to(torch.bfloat16) for s in shapes]
    M = [1e-3 * torch.randn(s, generator=gen, device=DEV) for s in shapes]
    hW, hG, hM = ([t.cpu().pin_memory() for t in L] for L in (W, G, M))
    torch.cuda.synchronize()
    mg.muon_step_ex(W, G, M, 0.02, 0.95, 0.1)
    mg.muon_step_host(hW, hG, hM, 0.02, 0.95, 0.1)
    torch.cuda.synchronize()
    for d, h in zip(W + M, hW + hM):
        assert torch.equal(d.cpu(), h)
