"""Seeded random batches against the oracle.

Each case draws a ragged batch of shapes (1 .. 600 on a side, both orientations,
widths that are and are not multiples of 8), weight dtype, stacked gradient
count and hyperparameters from a fixed seed, runs one full step through the C
ABI with the default routing (small matrices on the CUDA-core path, the rest on
the tensor cores with the fused final update) and checks every matrix: the
momentum bit-exact, O within the Newton-Schulz tolerance, W bit-exact given O.
"""
import numpy as np
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
import oracle
from tests.gpu_util import assert_o_close, bits, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(3, 9))
    shapes = []
    for _ in range(n):
        a = int(rng.choice([rng.integers(1, 65), rng.integers(64, 601)]))
        b = int(rng.integers(max(1, a // 4), 601))
        shapes.append((a, b) if rng.random() < 0.5 else (b, a))
    w_dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    K = int(rng.integers(1, 4))
    lr = float(np.float32(rng.uniform(1e-3, 5e-2)))
    mu = float(np.float32(rng.uniform(0.8, 0.99)))
    wd = float(np.float32(rng.uniform(0.0, 0.2)))
    return shapes, w_dtype, K, lr, mu, wd


@pytest.mark.parametrize("seed", range(6))
def test_random_batch_against_oracle(seed, monkeypatch):
    monkeypatch.delenv("MUON_DISABLE_SMALL_NS", raising=False)
    monkeypatch.delenv("MUON_NO_FUSED_UPDATE", raising=False)
    shapes, w_dtype, K, lr, mu, wd = _case(seed)
    gen = torch.Generator(device=DEV).manual_seed(1000 + seed)
    W = [(0.02 * torch.randn(s, generator=gen, device=DEV)).to(w_dtype) for s in shapes]
    G = [torch.randn((K,) + s if K > 1 else s, generator=gen, device=DEV).to(torch.bfloat16) for s in shapes]
    M = [1e-2 * torch.randn(s, generator=gen, device=DEV) for s in shapes]
    W0 = [bits(w) if w_dtype == torch.bfloat16 else f32(w) for w in W]
    G0 = [bits(g) for g in G]
    M0 = [f32(m) for m in M]
    O = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    mg.muon_step_ex(W, G, M, lr, mu, wd, o_out=O)
    torch.cuda.synchronize()
    assert mg.muon_device_status() == 0
    wb = w_dtype == torch.bfloat16
    for i, s in enumerate(shapes):
        _, M1, Oref = oracle.muon_step(W0[i], G0[i], M0[i], lr, mu, wd, w_bf16=wb, g_bf16=True)
        assert np.array_equal(f32(M[i]).view(np.uint32), M1.view(np.uint32)), f"M {s}"
        assert_o_close(f32(O[i]), Oref, f"O {s} (seed {seed})")
        dcy, sc = oracle.update_scalars(lr, wd, *s)
        got = bits(W[i]) if wb else f32(W[i]).view(np.uint32)
        ref = oracle.weight_update(W0[i], f32(O[i]), dcy, sc, w_bf16=wb)
        assert np.array_equal(got, ref if wb else ref.view(np.uint32)), f"W {s}"
