"""Where X0 is rounded is part of the parity contract.

Normalisation then Newton-Schulz ("How PyTorch Scaled a Near-1T MoE on
Europe's Public Supercomputer", section "Three optimizations that changed the
economics", FlexShard bullet: the orthogonalisation of whole matrices) is read
as X0 = bf16(U * sigma), sigma = 1 / (||U||_F + eps), then five bf16 iterations.

A cheaper front would store bf16(U) and fold sigma into the first products
instead (sigma^2 into the first Gram, sigma into the first update), which is the
same mathematics with X0 rounded at another point.  These tests show why the
CUDA path does not do that: every element of X0 then rounds differently, the
five bf16 iterations carry the difference into the small singular directions,
and O moves far beyond the 1e-2 contract, while the two legal fp32 summation
orders (the only freedom the contract leaves) stay well inside it.

The folded variant is written here in numpy as a test helper, not in the
oracle; a first test checks that the same helper without folding reproduces
the oracle within the contract, so the comparison isolates the rounding point.
"""
import numpy as np
import pytest

import oracle

A, B, C = (np.float32(x) for x in oracle.COEFFS)


def _bf16(x):
    """Round fp32 to the nearest bf16 (ties to even), returned as fp32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _ns(U, fold):
    """Five bf16 Newton-Schulz iterations of the r x k matrix U (r <= k), fp32
    products; `fold`: X0 = bf16(U) and sigma applied inside the first Gram and
    update instead of X0 = bf16(U * sigma)."""
    s = np.float32(1.0 / (np.sqrt((U.astype(np.float64) ** 2).sum()) + oracle.EPS))
    X = _bf16(U) if fold else _bf16(U * s)
    for it in range(5):
        G = X @ X.T
        if fold and it == 0:
            G = G * np.float32(s * s)
        Am = _bf16(G)
        Bm = _bf16(B * Am + C * (Am @ Am))
        V = A * X + Bm @ X
        if fold and it == 0:
            V = V * s
        X = _bf16(V)
    return X


def _full_rank(r, k, seed, lo=1e-3, hi=1.0):
    """Full-rank r x k fp32 matrix with singular values log-uniform in [lo, hi]
    (the mixed-block workload's spectrum)."""
    rng = np.random.default_rng(seed)
    Q1, R1 = np.linalg.qr(rng.standard_normal((r, r)))
    Q2, R2 = np.linalg.qr(rng.standard_normal((k, r)))
    Q1 *= np.sign(np.diag(R1))
    Q2 *= np.sign(np.diag(R2))
    s = np.exp(rng.uniform(np.log(lo), np.log(hi), r))
    return ((Q1 * s) @ Q2.T).astype(np.float32)


def _rel(x, ref):
    return float(np.linalg.norm(x - ref) / np.linalg.norm(ref))


@pytest.mark.parametrize("seed", [0, 1])
def test_numpy_helper_without_folding_reproduces_the_oracle(seed):
    U = _full_rank(128, 384, seed)
    ref = oracle.ns(U)
    assert _rel(_ns(U, fold=False), ref) <= 1e-2


@pytest.mark.parametrize("seed", [0, 1])
def test_folding_sigma_moves_o_far_beyond_the_summation_order_spread(seed):
    # measured: the two orders differ by 0.3 - 1.0 %, folding moves O by 7 - 9 %
    U = _full_rank(128, 384, seed)
    ref = oracle.ns(U)
    with oracle.descending_sums():
        spread = _rel(oracle.ns(U), ref)
    folded = _rel(_ns(U, fold=True), ref)
    assert spread <= 1e-2
    assert folded > 4e-2 and folded > 4 * spread


def test_folding_is_exact_when_sigma_is_a_power_of_two():
    # 4096 entries of +-1: ||U|| = 64 and fp32(1 / (64 + eps)) = 2^-6 exactly, so
    # scaling before or after the first rounding gives the same bits all the way
    rng = np.random.default_rng(3)
    U = np.zeros(128 * 384, dtype=np.float32)
    U[rng.choice(U.size, 4096, replace=False)] = rng.choice([-1.0, 1.0], 4096)
    U = U.reshape(128, 384)
    assert np.float32(1.0 / (64.0 + oracle.EPS)) == np.float32(2.0 ** -6)
    assert np.array_equal(_ns(U, fold=True), _ns(U, fold=False))
