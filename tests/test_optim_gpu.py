"""MuonAdamW (torch.optim wrapper) against direct calls of the two steps."""
import pytest
import torch

import muon_newton_schulz_step_gb300 as mg
from muon_newton_schulz_step_gb300.optim import MuonAdamW

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _params(seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    shapes = [(256, 768), (768, 256), (64, 256), (4096,), (33,), (1000, 64)]
    ps = [torch.nn.Parameter((0.02 * torch.randn(s, generator=gen, device=DEV)).to(torch.bfloat16)) for s in shapes]
    grads = [[torch.randn(s, generator=gen, device=DEV).to(torch.bfloat16) for s in shapes] for _ in range(3)]
    return ps, grads


def test_optimizer_matches_direct_calls_over_three_steps():
    ps, grads = _params(51)
    ref = [p.detach().clone() for p in ps]
    opt = MuonAdamW(ps, lr=0.02, momentum=0.95, weight_decay=0.1, adamw_lr=1e-3, betas=(0.9, 0.95),
                    eps=1e-8, adamw_weight_decay=0.01)
    M = [torch.zeros_like(r, dtype=torch.float32) for r in ref if r.ndim == 2]
    Am = [torch.zeros_like(r, dtype=torch.float32) for r in ref if r.ndim != 2]
    Av = [torch.zeros_like(r, dtype=torch.float32) for r in ref if r.ndim != 2]
    for t, g in enumerate(grads, start=1):
        for p, gi in zip(ps, g):
            p.grad = gi
        opt.step()
        Wr = [r for r in ref if r.ndim == 2]
        Gr = [gi for r, gi in zip(ref, g) if r.ndim == 2]
        mg.muon_step_ex(Wr, Gr, M, 0.02, 0.95, 0.1)
        Pr = [r for r in ref if r.ndim != 2]
        Gp = [gi for r, gi in zip(ref, g) if r.ndim != 2]
        mg.muon_adamw_step(Pr, Gp, Am, Av, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.01, step=t)
    torch.cuda.synchronize()
    for p, r in zip(ps, ref):
        assert torch.equal(p.detach().view(torch.int16), r.view(torch.int16)), tuple(p.shape)


def test_use_muon_flag_routes_a_matrix_to_adamw():
    ps, grads = _params(52)
    emb = ps[-1]                                  # an embedding-like matrix trained with AdamW
    opt = MuonAdamW([{"params": ps[:-1]}, {"params": [emb], "use_muon": False}])
    for p, gi in zip(ps, grads[0]):
        p.grad = gi
    opt.step()
    torch.cuda.synchronize()
    assert "exp_avg" in opt.state[emb] and "momentum" not in opt.state[emb]
    assert "momentum" in opt.state[ps[0]]
