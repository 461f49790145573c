"""Pins of the oracle's FP8 variant of Newton-Schulz (CPU).

The pages leave FP8 for expert matrix math as an open question ("Domyn is
training a 1T-parameter MoE on Europe's Jupiter supercomputer, and published
the recipe", section "What moved the number").  The variant built here rounds
only the Gram product's operands to E4M3, after the exact scaling X * 2^8;
the polynomial and the update stay bf16 (FP8 operands there cost 10-50 % of
O, because X' = a X + B X cancels to 0.7 X near convergence).  These tests pin
the E4M3 rounding against torch's float8 cast, the fixed scale against the
bound that makes it safe (no iterate element reaches 448 / 2^8), the FP8 Gram
against the bf16 mode on data E4M3 holds exactly, and the variant's distance
from bf16.
"""
import numpy as np
import pytest
import torch

import oracle
from muon_newton_schulz_step_gb300 import workloads as wl
from tests.gpu_util import compare_o


def _torch_e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2       # S.1111.111 only
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_rounding_matches_torch_on_grid_ties_and_random_values():
    finite = oracle.e4m3_to_f32(np.arange(0, 127, dtype=np.uint8)).astype(np.float64)   # 0 .. 448
    mids = (finite[:-1] + finite[1:]) / 2                       # exact ties
    nudge = np.concatenate([mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    rng = np.random.default_rng(1)
    rand = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(460.0), 200000))
    x = np.concatenate([finite, mids, nudge, rand]).astype(np.float32)
    x = np.concatenate([x, -x])
    x = x[np.abs(x) < 464]                                      # torch does not saturate; below 464 it rounds to <= 448
    assert np.array_equal(oracle.e4m3_rne(x), _torch_e4m3(x))


def test_e4m3_saturates_and_keeps_nan():
    big = np.float32([448, 464, 500, 1e4, 3e38, np.inf])
    assert list(oracle.e4m3_rne(big)) == [0x7e] * 6
    assert list(oracle.e4m3_rne(-big)) == [0xfe] * 6
    assert oracle.e4m3_rne(np.float32([np.nan]))[0] & 0x7f == 0x7f


def test_fixed_scale_never_saturates_on_the_iterates():
    # |X_ij| <= sigma_max(X): sigma_max(X0) <= ||X0||_F = 1, and the quintic maps
    # [0, 1.21] into [0, 1.2024] (its maximum, near s = 0.5545), so every iterate's
    # elements stay below 1.21 and 1.21 * 2^8 = 310 < 448
    a, b, c = (np.float64(v) for v in oracle.COEFFS)
    s = np.linspace(0.0, 1.21, 2000001)
    p = a * s + b * s ** 3 + c * s ** 5
    assert p.min() >= 0.0 and 1.2023 < p.max() < 1.2025
    assert abs(s[np.argmax(p)] - 0.5545) < 1e-3
    assert 1.21 * 2.0 ** 8 < 448.0 < 1.75 * 2.0 ** 8 + 1e-9
    # and on an actual run: the output (the fifth iterate) of a full-rank matrix
    rng = np.random.default_rng(5)
    U = rng.standard_normal((96, 320)).astype(np.float32)
    assert np.abs(oracle.ns_fp8_gram(U)).max() * 2.0 ** 8 < 448.0


def _ternary(m, n, nnz, seed):
    rng = np.random.default_rng(seed)
    U = np.zeros(m * n, dtype=np.float32)
    U[rng.choice(m * n, size=nnz, replace=False)] = rng.choice([-1.0, 1.0], size=nnz)
    return U.reshape(m, n)


@pytest.mark.parametrize("shape", [(64, 256), (48, 96), (100, 40)])
@pytest.mark.parametrize("sched", [[(0.5, 0.25, 1.0)], [(1.0, 0.0, 0.0), (0.5, 0.25, 1.0)]])
def test_fp8_gram_equals_bf16_where_e4m3_is_exact(shape, sched):
    # 256 entries of +-1: X0 = +-1/16 exactly, scaled by 2^8 to +-16, an E4M3
    # value; every product and partial sum is exact, so the FP8 Gram and the
    # bf16 Gram agree bit for bit (a wrong scale, exponent or unscaling breaks it)
    U = _ternary(*shape, 256, seed=sum(shape))
    a = oracle.ns_schedule(U, sched)
    b = oracle.ns_fp8_gram(U, schedule=sched)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_fp8_gram_is_active_and_close_to_the_closed_form():
    rng = np.random.default_rng(8)
    m, n = 96, 320
    Uf, _ = np.linalg.qr(rng.standard_normal((m, m)))
    Vf, _ = np.linalg.qr(rng.standard_normal((n, m)))
    s = np.linspace(0.2, 1.0, m)
    U = ((Uf * s) @ Vf.T).astype(np.float32)
    exact = oracle.ns(U.astype(np.float64), 5, mode="f64")
    f8 = oracle.ns_fp8_gram(U)
    bf = oracle.ns(U, 5)
    assert not np.array_equal(f8, bf)                 # the quantisation is applied
    assert compare_o(f8, exact)[0] < 8e-2
    assert compare_o(bf, exact)[0] < 2.5e-2


# The FP8 variant's accuracy reading: on the workloads' spectra its O stays
# within 8e-2 relative Frobenius (and 2e-2 per element) of the bf16 oracle.
FP8_REL, FP8_ABS = 8e-2, 2e-2


@pytest.mark.parametrize("kind", ["rank16_noise", "full_rank", "gauss"])
def test_fp8_variant_distance_from_bf16(kind):
    spec = {"rank16_noise": wl.MatrixSpec(256, 768, "loguniform", 16, 1e-2, 1.0, 1e-3),
            "full_rank": wl.MatrixSpec(256, 768, "loguniform", None, 1e-3, 1.0, 0.0),
            "gauss": wl.MatrixSpec(256, 768, "none", 0, 0.0, 0.0, 1.0)}[kind]
    w = wl.Workload("fp8", 61, "ns", [spec], on_host=True)
    U = oracle.bf16_to_f32(oracle.bf16_rne(wl.gradient(w, 0, "cpu").numpy()))
    rel, mx = compare_o(oracle.ns_fp8_gram(U), oracle.ns(U, 5))
    assert 1e-3 < rel <= FP8_REL and mx <= FP8_ABS, (rel, mx)
