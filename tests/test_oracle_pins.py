"""Pins of the CPU oracle against things other than itself.

The pages ("How PyTorch Scaled a Near-1T MoE on Europe's Public
Supercomputer", "Three optimizations that changed the economics", FlexShard
bullet) print no worked example, no formula and no constant for the Muon step,
so nothing here is a stored value from them.  Each pin is instead one of:
  * a library routine the step reduces to (torch's bf16 cast),
  * exact rational arithmetic (fractions.Fraction) for every fp32 rounding
    of the elementwise parts,
  * the closed form of an odd matrix polynomial iteration: for
    X = U diag(s) V^T the iteration acts on the singular values alone, so
    fp64 Newton-Schulz gives U diag(p^5(s / (|s|_2 + eps))) V^T, p(x) = a x +
    b x^3 + c x^5,
  * special cases (rank one, multiples of I, zero, diagonal inputs whose
    bf16 recursion is a scalar one),
  * the singular-value band that p^5 maps (0, 1] into.
Several tests plant a mistake in an oracle call (wrong coefficient order,
transposed input) and check that the pin notices.
"""
from fractions import Fraction
import math

import numpy as np
import pytest
import torch

import oracle
from tests import exact

A, B, C = oracle.COEFFS
EPS = oracle.EPS


def p(x, coeffs=oracle.COEFFS):
    a, b, c = coeffs
    return a * x + b * x ** 3 + c * x ** 5


def p5(x, steps=5, coeffs=oracle.COEFFS):
    for _ in range(steps):
        x = p(x, coeffs)
    return x


def haar(rng, n, k):
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


def closed_form(Uf, s, Vf, steps=5, coeffs=oracle.COEFFS):
    sh = s / (np.linalg.norm(s) + EPS)
    return (Uf * p5(sh, steps, coeffs)) @ Vf.T


# ------------------------------------------------------------------ bf16 ---
def _torch_bf16_bits(x32):
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch_cast():
    rng = np.random.default_rng(1)
    rand_bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # exact ties (dropped half = 0x8000) with even and odd kept parts
    hi = rng.integers(0, 0x7f7f, size=4096, dtype=np.uint32)
    ties = (hi << 16) | 0x8000
    edges = np.array([0x00000000, 0x80000000, 0x00000001, 0x807fffff, 0x00008000,
                      0x00018000, 0x7f7fffff, 0xff7fffff, 0x7f7f8000, 0x7f800000,
                      0xff800000, 0x3f808000, 0x3f818000, 0x3f7fffff], dtype=np.uint32)
    bits = np.concatenate([rand_bits, ties, ties | 0x80000000, edges])
    x = bits.view(np.float32)
    finite_or_inf = ~np.isnan(x)
    ours = oracle.bf16_rne(x)
    ref = _torch_bf16_bits(x)
    assert np.array_equal(ours[finite_or_inf], ref[finite_or_inf])
    # NaN stays NaN
    assert np.all(np.isnan(oracle.bf16_to_f32(ours[~finite_or_inf])))


def test_bf16_to_f32_is_exact_widening():
    h = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(h)
    back = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    ok = ~np.isnan(f)
    assert np.array_equal(f[ok].view(np.uint32), back[ok].view(np.uint32))


# -------------------------------------------------------------- momentum ---
def _momentum_exact(g, m, mu, nesterov=True):
    qmu = exact.f32_to_frac(mu)
    mp = exact.rn_f32(qmu * exact.f32_to_frac(m) + exact.f32_to_frac(g))
    u = exact.rn_f32(qmu * exact.f32_to_frac(mp) + exact.f32_to_frac(g)) if nesterov else mp
    return mp, u


def test_momentum_nesterov_bit_exact_vs_rational():
    rng = np.random.default_rng(2)
    n = 40000
    g = (rng.standard_normal(n) * 10.0 ** rng.integers(-6, 2, n)).astype(np.float32)
    M = (rng.standard_normal(n) * 10.0 ** rng.integers(-6, 2, n)).astype(np.float32)
    # subnormals, zeros, signed zeros, opposite signs that cancel
    g[:8] = np.array([0.0, -0.0, 1e-45, -1e-44, 3e-39, 0.0, 1.0, -1.0], dtype=np.float32)
    M[:8] = np.array([0.0, 0.0, 2e-45, 1e-45, -2e-39, 1e-40, -1.0 / 0.95, 1.0], dtype=np.float32)
    mu = np.float32(0.95)
    M1, U = oracle.momentum(g, M, mu, nesterov=True)
    for e in range(n):
        mp, u = _momentum_exact(g[e], M[e], mu)
        assert M1[e].view(np.uint32) == mp.view(np.uint32) or (M1[e] == 0 and mp == 0), e
        assert U[e].view(np.uint32) == u.view(np.uint32) or (U[e] == 0 and u == 0), e


def test_momentum_ties_round_to_even():
    # mu*M + g lands exactly half-way between two fp32 values
    mu = np.float32(0.5)
    M = np.array([2.0, 2.0, -2.0, 2.0 ** 20], dtype=np.float32)
    g = np.array([2.0 ** -24, 3 * 2.0 ** -24, -(2.0 ** -24), 2.0 ** -5], dtype=np.float32)
    M1, _ = oracle.momentum(g, M, mu)
    want = [exact.rn_f32(Fraction(1, 2) * exact.f32_to_frac(M[i]) + exact.f32_to_frac(g[i]))
            for i in range(4)]
    assert np.array_equal(M1.view(np.uint32), np.array(want, dtype=np.float32).view(np.uint32))
    assert M1[0] == 1.0 and M1[1] == np.float32(1 + 2.0 ** -22)


def test_momentum_plain_and_zero_state():
    rng = np.random.default_rng(3)
    g = rng.standard_normal(1000).astype(np.float32)
    M1, U = oracle.momentum(g, np.zeros_like(g), 0.95, nesterov=False)
    assert np.array_equal(M1, g) and np.array_equal(U, g)   # M = 0 -> M' = g exactly


# ------------------------------------------------------ Newton-Schulz f64 ---
@pytest.mark.parametrize("m,n,seed", [(8, 8, 0), (16, 48, 1), (48, 16, 2), (32, 96, 3), (64, 64, 4)])
def test_ns_f64_closed_form(m, n, seed):
    rng = np.random.default_rng(seed)
    r = min(m, n)
    Uf, Vf = haar(rng, m, r), haar(rng, n, r)
    s = np.exp(rng.uniform(np.log(1e-3), 0.0, r))
    X = (Uf * s) @ Vf.T
    O = oracle.ns(X, mode="f64")
    ref = closed_form(Uf, s, Vf)
    assert np.linalg.norm(O - ref) / np.linalg.norm(ref) < 1e-10


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 7])
def test_ns_f64_closed_form_any_step_count(steps):
    rng = np.random.default_rng(10 + steps)
    Uf, Vf = haar(rng, 12, 12), haar(rng, 40, 12)
    s = np.exp(rng.uniform(np.log(1e-2), 0.0, 12))
    O = oracle.ns((Uf * s) @ Vf.T, steps=steps, mode="f64")
    ref = closed_form(Uf, s, Vf, steps=steps)
    assert np.linalg.norm(O - ref) / np.linalg.norm(ref) < 1e-10


@pytest.mark.parametrize("shape", [(1, 1), (1, 5), (5, 1), (3, 3), (4, 8), (8, 5), (16, 64), (7, 13)])
def test_ns_f64_brute_force_tiny_shapes(shape):
    rng = np.random.default_rng(sum(shape))
    X = rng.standard_normal(shape)
    Uf, s, Vt = np.linalg.svd(X, full_matrices=False)
    O = oracle.ns(X, mode="f64")
    ref = closed_form(Uf, s, Vt.T)
    assert np.allclose(O, ref, rtol=0, atol=1e-11 * max(1.0, np.abs(ref).max()))


def test_ns_f64_rank_one_and_vector():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 37))
    nx = np.linalg.norm(x)
    want = p5(nx / (nx + EPS)) * x / nx
    assert np.allclose(oracle.ns(x, mode="f64"), want, atol=1e-13)
    assert np.allclose(oracle.ns(x.T, mode="f64"), want.T, atol=1e-13)
    # value: p^5 of (almost) 1 is 0.6964... (x/|x| scaled)
    assert abs(p5(1.0) - 0.696436) < 1e-6


# p^5 at sample points, computed outside this code from the coefficients
# (3.4445, -4.7750, 2.0315) to 6 decimals; with the position and height of
# the maximum on (0, 1] and the point where p^5 reaches 0.6
P5_TABLE = [(1.0, 0.696436), (0.5, 0.765439), (0.1, 0.712120), (0.01, 0.698917), (0.005, 1.154366),
            (0.002, 0.860039), (0.001, 0.470544), (1e-4, 0.048473)]


def test_p5_scalar_table_and_band_thresholds():
    for x, want in P5_TABLE:
        assert abs(p5(x) - want) < 1e-6, (x, p5(x), want)
    assert abs(p(1.0) - 0.701) < 1e-12          # a + b + c
    xs = np.geomspace(1e-4, 1.0, 400001)
    ys = p5(xs)
    i = int(np.argmax(ys))
    assert abs(ys[i] - 1.20237) < 1e-5 and abs(xs[i] - 4.11e-3) < 2e-5
    tau = xs[np.argmax(ys >= 0.6)]              # first x with p^5(x) >= 0.6
    assert abs(tau - 1.3021e-3) < 1e-7
    assert ys[xs >= tau].min() >= 0.6 - 1e-12


@pytest.mark.parametrize("r", [1, 4, 9, 64])
def test_ns_f64_multiple_of_identity(r):
    X = 3.0 * np.eye(r)
    O = oracle.ns(X, mode="f64")
    want = p5(3.0 * math.sqrt(r) / (3.0 * math.sqrt(r) + EPS) / math.sqrt(r))
    assert np.allclose(O, want * np.eye(r), atol=1e-13)


@pytest.mark.parametrize("mode", ["f64", "bf16"])
def test_ns_zero_matrix_gives_zero(mode):
    O = oracle.ns(np.zeros((6, 10)), mode=mode)
    assert np.all(O == 0)


def test_ns_f64_singular_value_band():
    # p^5 maps [2e-3, 1] into [0.6, 1.25]; and all of (0, 1] below 1.25
    xs = np.concatenate([np.geomspace(1e-6, 1.0, 20001)])
    ys = p5(xs)
    assert ys.max() < 1.21 and ys.max() > 1.20
    assert ys[xs >= 2e-3].min() > 0.6
    rng = np.random.default_rng(6)
    Uf, Vf = haar(rng, 32, 32), haar(rng, 80, 32)
    s = np.exp(rng.uniform(np.log(1e-5), 0.0, 32))
    O = oracle.ns((Uf * s) @ Vf.T, mode="f64")
    so = np.linalg.svd(O, compute_uv=False)
    assert so.max() <= 1.25
    sh = np.sort(s / (np.linalg.norm(s) + EPS))[::-1]
    # singular vectors are shared, so the output spectrum is p^5 of the input one
    assert np.allclose(np.sort(so)[::-1], np.sort(p5(sh))[::-1], atol=1e-10)
    assert so[np.sort(p5(sh))[::-1] > 0][: int((sh >= 2e-3).sum())].min() >= 0.6 - 1e-12


def test_planted_mistakes_are_caught_by_closed_form():
    rng = np.random.default_rng(7)
    Uf, Vf = haar(rng, 16, 16), haar(rng, 24, 16)
    s = np.exp(rng.uniform(np.log(1e-2), 0.0, 16))
    X = (Uf * s) @ Vf.T
    ref = closed_form(Uf, s, Vf)
    rel = lambda O: np.linalg.norm(O - ref) / np.linalg.norm(ref)
    assert rel(oracle.ns(X, mode="f64")) < 1e-10
    assert rel(oracle.ns(X, coeffs=(A, C, B), mode="f64")) > 1e-2          # swapped b, c
    assert rel(oracle.ns(X, coeffs=(A, -B, C), mode="f64")) > 1e-2         # sign of b
    assert rel(oracle.ns(X, steps=4, mode="f64")) > 1e-3                    # a step dropped
    Xsq = (haar(rng, 16, 16) * s) @ haar(rng, 16, 16).T                     # square, non-symmetric
    Us, ss, Vst = np.linalg.svd(Xsq)
    ref_sq = closed_form(Us, ss, Vst.T)
    assert np.linalg.norm(oracle.ns(Xsq, mode="f64") - ref_sq) < 1e-9
    assert np.linalg.norm(oracle.ns(Xsq.T, mode="f64").T - ref_sq) < 1e-9  # O(X^T) = O(X)^T
    assert np.linalg.norm(oracle.ns(Xsq.T, mode="f64") - ref_sq) > 1e-2    # transposed operand


# ----------------------------------------------------- Newton-Schulz bf16 ---
def _rb(x):
    return exact.rn_bf16(exact.f32_to_frac(x))


def _f32(x):
    return np.float32(x)


def _scalar_bf16_recursion(x0, steps, coeffs=oracle.COEFFS):
    """bf16 emulation on a diagonal input: every product in the matrix
    algorithm has a single non-zero term, so it reduces to this scalar one
    (fp32 ops are correctly rounded numpy float32 ops; bf16 rounding is the
    rational rounding from tests/exact.py)."""
    a, b, c = (np.float32(v) for v in coeffs)
    x = x0
    for _ in range(steps):
        A_ = _rb(_f32(x * x))
        S = _f32(A_ * A_)
        B_ = _rb(_f32(_f32(b * A_) + _f32(c * S)))
        x = _rb(_f32(_f32(a * x) + _f32(B_ * x)))
    return x


def test_ns_bf16_diagonal_input_matches_scalar_recursion():
    rng = np.random.default_rng(8)
    r, k = 6, 10
    s = np.exp(rng.uniform(np.log(1e-3), 0.0, r)).astype(np.float32)
    X = np.zeros((r, k), dtype=np.float32)
    X[np.arange(r), np.arange(r)] = s
    for steps in (0, 1, 2, 5):
        O = oracle.ns(X, steps=steps)
        d = math.sqrt(float(np.sum(s.astype(np.float64) ** 2))) + EPS
        sigma = np.float32(1.0 / d)
        want = np.zeros_like(X)
        for i in range(r):
            x0 = _rb(_f32(s[i] * sigma))
            want[i, i] = _scalar_bf16_recursion(x0, steps)
        assert np.array_equal(O, want), steps
        # and the tall orientation gives the transpose
        assert np.array_equal(oracle.ns(X.T.copy(), steps=steps), want.T)


def test_ns_bf16_close_to_closed_form_when_well_conditioned():
    rng = np.random.default_rng(9)
    for m, n in [(32, 96), (96, 32), (64, 64)]:
        r = min(m, n)
        Uf, Vf = haar(rng, m, r), haar(rng, n, r)
        s = np.exp(rng.uniform(np.log(0.05), 0.0, r))
        X = ((Uf * s) @ Vf.T).astype(np.float32)
        ref = closed_form(Uf, s, Vf)
        O = oracle.ns(X)
        assert np.linalg.norm(O - ref) / np.linalg.norm(ref) < 2.5e-2
        # a planted transposed operand (B X -> X^T-based) is far outside this bound
        Ot = oracle.ns(X.T.copy()).T
        assert np.linalg.norm(Ot - O) / np.linalg.norm(O) < 2.5e-2  # transpose-equivariant
    so = np.linalg.svd(O, compute_uv=False)
    assert so.max() <= 1.25 and so.min() >= 0.6


def test_ns_bf16_output_is_bf16_and_band():
    rng = np.random.default_rng(11)
    X = rng.standard_normal((48, 160)).astype(np.float32)
    O = oracle.ns(X)
    assert np.array_equal(oracle.bf16_to_f32(oracle.bf16_rne(O)), O)
    so = np.linalg.svd(O.astype(np.float64), compute_uv=False)
    assert so.max() <= 1.25 and so.min() >= 0.6


def test_ns_bf16_normalisation_step():
    rng = np.random.default_rng(12)
    X = (rng.standard_normal((20, 30)) * 37.0).astype(np.float32)
    O0 = oracle.ns(X, steps=0)
    ref = X.astype(np.float64) / (np.linalg.norm(X.astype(np.float64)) + EPS)
    # within half a bf16 ulp (+ the fp32 multiply) of the exact quotient
    # half a bf16 ulp is at most 2^-8 of the value
    assert np.all(np.abs(O0 - ref) <= np.abs(ref) * (2.0 ** -8) * (1 + 1e-5) + 1e-30)
    # and a wrong norm (e.g. squared, or without the square root) is far outside it
    assert np.abs(O0).max() < 1.0 and abs(np.linalg.norm(O0.astype(np.float64)) - 1.0) < 1e-2


# ---------------------------------------------------------------- update ---
def test_update_scalars_and_formula_exact():
    rng = np.random.default_rng(13)
    lr, wd = np.float32(0.02), np.float32(0.1)
    for (m, n) in [(64, 256), (6144, 2048), (1024, 6144), (7, 3)]:
        dcy, s = oracle.update_scalars(lr, wd, m, n)
        assert dcy == np.float32(1.0 - float(lr) * float(wd))
        want_s = float(lr) * 0.2 * math.sqrt(max(m, n))
        assert abs(float(s) - want_s) <= abs(want_s) * 2.0 ** -24
    dcy, s = oracle.update_scalars(lr, wd, 2048, 6144)
    n = 20000
    W = (rng.standard_normal(n) * 0.02).astype(np.float32)
    O = oracle.bf16_to_f32(oracle.bf16_rne(rng.uniform(-1.2, 1.2, n).astype(np.float32)))
    W32 = oracle.weight_update(W, O, dcy, s, w_bf16=False)
    Wb = oracle.bf16_rne(W)
    Wb1 = oracle.weight_update(Wb, O, dcy, s, w_bf16=True)
    qs, qd = exact.f32_to_frac(s), exact.f32_to_frac(dcy)
    for e in range(0, n, 7):
        dec = exact.rn_f32(qd * exact.f32_to_frac(W[e]))
        want = exact.rn_f32(-qs * exact.f32_to_frac(O[e]) + exact.f32_to_frac(dec))
        assert W32[e] == want
        decb = exact.rn_f32(qd * exact.f32_to_frac(oracle.bf16_to_f32(Wb[e:e + 1])[0]))
        fm = exact.rn_f32(-qs * exact.f32_to_frac(O[e]) + exact.f32_to_frac(decb))
        assert oracle.bf16_to_f32(Wb1[e:e + 1])[0] == exact.rn_bf16(exact.f32_to_frac(fm))


def test_update_lr_zero_keeps_weights_bit_exact():
    rng = np.random.default_rng(14)
    W = (rng.standard_normal(500) * 0.02).astype(np.float32)
    O = rng.uniform(-1, 1, 500).astype(np.float32)
    dcy, s = oracle.update_scalars(0.0, 0.1, 30, 40)
    assert dcy == 1.0 and s == 0.0
    assert np.array_equal(oracle.weight_update(W, O, dcy, s, w_bf16=False).view(np.uint32),
                          W.view(np.uint32))


def test_full_step_composition():
    rng = np.random.default_rng(15)
    m, n = 40, 24
    G = rng.standard_normal((m, n)).astype(np.float32)
    M = (rng.standard_normal((m, n)) * 1e-3).astype(np.float32)
    W = (rng.standard_normal((m, n)) * 0.02).astype(np.float32)
    W1, M1, O = oracle.muon_step(W, G, M, 0.02, 0.95, 0.1, w_bf16=False, g_bf16=False)
    Mm, U = oracle.momentum(G, M, 0.95)
    assert np.array_equal(M1, Mm)
    assert np.array_equal(O, oracle.ns(U))
    dcy, s = oracle.update_scalars(0.02, 0.1, m, n)
    assert np.array_equal(W1, oracle.weight_update(W, O, dcy, s, w_bf16=False))


# ------------------------------------------------- coefficient schedules ---
SCHEDULE = [oracle.COEFFS] * 3 + [(2.0, -1.5, 0.5), (1.875, -1.25, 0.375)]


def test_ns_schedule_f64_closed_form_is_the_composed_polynomial():
    rng = np.random.default_rng(21)
    Uf, Vf = haar(rng, 24, 24), haar(rng, 56, 24)
    s = np.exp(rng.uniform(np.log(1e-2), 0.0, 24))
    O = oracle.ns_schedule((Uf * s) @ Vf.T, SCHEDULE, mode="f64")
    x = s / (np.linalg.norm(s) + EPS)
    for coeffs in SCHEDULE:
        x = p(x, coeffs)
    ref = (Uf * x) @ Vf.T
    assert np.linalg.norm(O - ref) / np.linalg.norm(ref) < 1e-10
    # the schedule's last polynomial has p(1) = 1, p'(1) = 0: the spectrum ends closer to 1
    assert np.abs(x - 1).max() < np.abs(p5(s / (np.linalg.norm(s) + EPS)) - 1).max()


def test_ns_schedule_of_one_triple_equals_the_fixed_form_bit_for_bit():
    rng = np.random.default_rng(22)
    X = rng.standard_normal((40, 72)).astype(np.float32)
    assert np.array_equal(oracle.ns_schedule(X, [oracle.COEFFS] * 5), oracle.ns(X, steps=5))
    assert np.array_equal(oracle.ns_schedule(X, []), oracle.ns(X, steps=0))
    # order matters: reversing a non-constant schedule changes the result
    assert not np.array_equal(oracle.ns_schedule(X, SCHEDULE), oracle.ns_schedule(X, SCHEDULE[::-1]))


# -------------------------------------------------- gradient accumulation ---
def test_grad_sum_is_the_in_order_fp32_sum():
    rng = np.random.default_rng(23)
    K, n = 5, 3000
    G = (rng.standard_normal((K, n)) * 10.0 ** rng.integers(-4, 2, (K, n))).astype(np.float32)
    Gb = oracle.bf16_rne(G).reshape(K, n)
    for g_bf16, stack in ((True, Gb), (False, G)):
        got = oracle.grad_sum(stack, g_bf16)
        vals = oracle.bf16_to_f32(stack).reshape(K, n) if g_bf16 else stack
        for e in range(0, n, 3):
            acc = exact.f32_to_frac(vals[0, e])
            want = np.float32(vals[0, e])
            for j in range(1, K):
                want = exact.rn_f32(exact.f32_to_frac(want) + exact.f32_to_frac(vals[j, e]))
            assert got[e].view(np.uint32) == want.view(np.uint32) or (got[e] == 0 and want == 0)
    # one gradient: the sum is that gradient, bit for bit
    assert np.array_equal(oracle.grad_sum(Gb[:1], True), oracle.bf16_to_f32(Gb[0]))


def test_step_with_stacked_gradients_equals_step_on_their_sum():
    rng = np.random.default_rng(24)
    m, n, K = 24, 40, 3
    Gs = oracle.bf16_rne((rng.standard_normal((K, m, n)) * 1e-2).astype(np.float32)).reshape(K, m, n)
    W = oracle.bf16_rne((rng.standard_normal((m, n)) * 0.02).astype(np.float32))
    M = (rng.standard_normal((m, n)) * 1e-3).astype(np.float32)
    W1, M1, O1 = oracle.muon_step(W, Gs, M, 0.02, 0.95, 0.1, w_bf16=True, g_bf16=True)
    g = oracle.grad_sum(Gs, True)
    W2, M2, O2 = oracle.muon_step(W, g, M, 0.02, 0.95, 0.1, w_bf16=True, g_bf16=False)
    assert np.array_equal(M1, M2) and np.array_equal(O1, O2) and np.array_equal(W1, W2)
