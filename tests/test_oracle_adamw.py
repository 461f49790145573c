"""Pins of the oracle's AdamW (the optimizer for the parameters Muon does not
cover).  torch.optim.AdamW run in fp64 is an independent implementation of the
same update (decoupled weight decay, bias correction, eps outside the square
root); the fp32 oracle must agree with it to fp32 rounding."""
import math

import numpy as np
import pytest
import torch

import oracle

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)


def _torch_adamw_fp64(p0, grads, hp):
    p = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                            weight_decay=hp["wd"], foreach=False)
    for g in grads:
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


@pytest.mark.parametrize("hp", [HP, dict(lr=1e-2, beta1=0.8, beta2=0.999, eps=1e-6, wd=0.0)])
def test_adamw_matches_torch_fp64_over_several_steps(hp):
    rng = np.random.default_rng(51)
    n = 4000
    p = (rng.standard_normal(n) * 0.05).astype(np.float32)
    grads = [(rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 0, n)).astype(np.float32) for _ in range(4)]
    P, M, V = p.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t, g in enumerate(grads, start=1):
        P, M, V = oracle.adamw(P, g, M, V, step=t, p_bf16=False, g_bf16=False, **hp)
    # the oracle's hyper-parameters are fp32 values: give torch exactly those
    hp64 = {k: float(np.float32(v)) for k, v in hp.items()}
    rp, rm, rv = _torch_adamw_fp64(p.astype(np.float64), [g.astype(np.float64) for g in grads], hp64)
    # fp32 rounding bound: a few ulps of the sum of the absolute contributions
    T = len(grads)
    hp = hp64
    am = sum((1 - hp["beta1"]) * hp["beta1"] ** (T - t) * np.abs(g.astype(np.float64)) for t, g in enumerate(grads, 1))
    av = sum((1 - hp["beta2"]) * hp["beta2"] ** (T - t) * g.astype(np.float64) ** 2 for t, g in enumerate(grads, 1))
    assert np.all(np.abs(M - rm) <= 2.0 ** -20 * am)
    assert np.all(np.abs(V - rv) <= 2.0 ** -20 * av)
    # parameters: the update is lr-sized, so compare the change against fp32 resolution
    assert np.abs(P - rp).max() <= 1e-6 * max(1.0, np.abs(rp).max()) + 1e-3 * hp["lr"]


def test_adamw_first_step_closed_form_and_zero_gradient():
    rng = np.random.default_rng(52)
    n = 1000
    p = (rng.standard_normal(n) * 0.05).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    P, M, V = oracle.adamw(p, g, np.zeros(n, np.float32), np.zeros(n, np.float32), step=1,
                           p_bf16=False, g_bf16=False, **HP)
    # step 1: m_hat = g, v_hat = g^2 -> p' = p (1 - lr wd) - lr g / (|g| + eps)
    want = p.astype(np.float64) * (1 - HP["lr"] * HP["wd"]) - HP["lr"] * g / (np.abs(g) + HP["eps"])
    assert np.abs(P - want).max() < 1e-7
    # zero gradient and zero state: only the decay acts
    P0, M0, V0 = oracle.adamw(p, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32),
                              step=3, p_bf16=False, g_bf16=False, **HP)
    dcy = oracle.adamw_scalars(HP["lr"], HP["beta1"], HP["beta2"], HP["wd"], 3)[2]
    assert np.array_equal(P0, (dcy * p).astype(np.float32)) and not M0.any() and not V0.any()


def test_adamw_host_scalars():
    s = oracle.adamw_scalars(3e-4, 0.9, 0.95, 0.1, 7)
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.95))
    assert s[3] == np.float32(float(np.float32(3e-4)) / (1 - b1 ** 7))
    assert s[4] == np.float32(1 / math.sqrt(1 - b2 ** 7))
    assert s[0] == np.float32(1 - b1) and s[2] == np.float32(1 - float(np.float32(3e-4)) * float(np.float32(0.1)))


def test_adamw_bf16_parameters_round_once():
    rng = np.random.default_rng(53)
    n = 2000
    p32 = (rng.standard_normal(n) * 0.05).astype(np.float32)
    pb = oracle.bf16_rne(p32)
    g = oracle.bf16_rne((rng.standard_normal(n) * 1e-2).astype(np.float32))
    Pb, Mb, Vb = oracle.adamw(pb, g, np.zeros(n, np.float32), np.zeros(n, np.float32), step=2,
                              p_bf16=True, g_bf16=True, **HP)
    P32, M32, V32 = oracle.adamw(oracle.bf16_to_f32(pb), oracle.bf16_to_f32(g), np.zeros(n, np.float32),
                                 np.zeros(n, np.float32), step=2, p_bf16=False, g_bf16=False, **HP)
    assert np.array_equal(Mb, M32) and np.array_equal(Vb, V32)
    assert np.array_equal(Pb, oracle.bf16_rne(P32))      # the fp32 result rounded once to bf16
