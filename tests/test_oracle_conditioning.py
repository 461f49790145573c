"""The oracle's second summation order and the conditioning reading (CPU).

The pages fix no order for the fp32 sums of the Newton-Schulz products; the
oracle sums in ascending order and can switch to descending order only to
measure how far a legal change of order alone moves O (tests/conditioning.py).
These tests pin that the switch changes nothing but the order, and that the
tiny workload's matrix 6 -- the one the tensor cores move by 1.6 % -- is
ill-conditioned by that measure while its siblings are not.
"""
import numpy as np
import pytest

import oracle
from muon_newton_schulz_step_gb300 import workloads as wl
from tests.conditioning import bound_for, order_spread
from tests.gpu_util import ABS_TOL, REL_TOL, compare_o


def _ternary(m, n, nnz, seed):
    rng = np.random.default_rng(seed)
    U = np.zeros(m * n, dtype=np.float32)
    U[rng.choice(m * n, size=nnz, replace=False)] = rng.choice([-1.0, 1.0], size=nnz)
    return U.reshape(m, n)


@pytest.mark.parametrize("shape", [(64, 256), (96, 40), (33, 65)])
@pytest.mark.parametrize("coeffs", [(0.5, 0.25, 1.0), (1.0, 0.0, 0.0), (0.0, 1.0, 0.0)])
def test_descending_order_is_identical_on_exact_data(shape, coeffs):
    # every partial sum is exact (power-of-two data and coefficients), so the
    # two orders must agree bit for bit: the switch only reorders the sums
    X = oracle.bf16_rne(_ternary(*shape, min(256, shape[0] * shape[1]), seed=sum(shape)))
    asc = oracle.ns_bf16_bits(X, steps=1, coeffs=coeffs)
    with oracle.descending_sums():
        desc = oracle.ns_bf16_bits(X, steps=1, coeffs=coeffs)
    assert np.array_equal(asc, desc)


def test_descending_order_differs_on_inexact_data_and_resets():
    rng = np.random.default_rng(3)
    U = rng.standard_normal((64, 256)).astype(np.float32)
    asc = oracle.ns(U, 5)
    with oracle.descending_sums():
        desc = oracle.ns(U, 5)
    assert not np.array_equal(asc, desc)           # the order really changed
    rel, mx = compare_o(desc, asc)
    assert rel <= REL_TOL and mx <= ABS_TOL          # within the contract of each other
    assert np.array_equal(oracle.ns(U, 5), asc)    # and the default order is back


def test_descending_order_keeps_the_closed_form():
    # the f64-checked closed form U p^5(s) V^T holds within the bf16 error scale
    # for either order on a well-conditioned input
    rng = np.random.default_rng(8)
    m, n = 48, 160
    Uf, _ = np.linalg.qr(rng.standard_normal((m, m)))
    Vf, _ = np.linalg.qr(rng.standard_normal((n, m)))
    s = np.linspace(0.2, 1.0, m)
    U = ((Uf * s) @ Vf.T).astype(np.float32)
    exact = oracle.ns(U.astype(np.float64), 5, mode="f64")
    with oracle.descending_sums():
        desc = oracle.ns(U, 5)
    rel, _ = compare_o(desc, exact)
    assert rel < 2.5e-2


def _tiny_spreads():
    w = wl.workload("tiny")
    inp = wl.make_inputs(w, "cpu")
    out = []
    for i in range(w.count):
        W, G, M = inp["W"][i].numpy(), inp["G"][i].numpy(), inp["M"][i].numpy()
        out.append(order_spread(lambda: oracle.muon_step(W, G, M, w.lr, w.mu, w.wd,
                                                         w_bf16=False, g_bf16=False)[2]))
    return out


def test_tiny_matrix_6_is_ill_conditioned_and_the_rest_are_not():
    spreads = _tiny_spreads()
    rel6, _ = spreads[6]
    # the two legal orders alone move O by more than the contract allows
    assert rel6 > REL_TOL
    assert not bound_for(spreads[6])[2]
    for i, sp in enumerate(spreads):
        if i != 6:
            assert bound_for(sp)[2], f"matrix {i}: spread {sp}"
