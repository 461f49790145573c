"""A torch.optim.Optimizer over the library's two steps.

The recipe in "Domyn is training a 1T-parameter MoE on Europe's Jupiter
supercomputer, and published the recipe" (table "The model and the machine")
trains the weight matrices (about 99.5 % of the parameters) with Muon and the
rest -- vectors, norms, embeddings -- with AdamW.  ``MuonAdamW`` does that
split for a model's parameters: every 2-D parameter not marked otherwise goes
through one batched ``muon_step_ex`` call per dtype, everything else through
one ``muon_adamw_step`` call per dtype.  It only marshals arguments: the state
(fp32 momentum for Muon, fp32 first and second moments for AdamW) lives in
``self.state`` as CUDA tensors and every update runs in the library's kernels.
"""
from collections import defaultdict

import torch

from . import muon_adamw_step, muon_step_ex


class MuonAdamW(torch.optim.Optimizer):
    """Muon for matrices, AdamW for the rest.

    Parameter groups take ``use_muon`` (default: ``p.ndim == 2``), ``lr``,
    ``momentum``, ``weight_decay``, ``nesterov``, ``ns_steps`` (Muon) and
    ``adamw_lr``, ``betas``, ``eps``, ``adamw_weight_decay`` (AdamW).
    Parameters must be contiguous CUDA tensors in bf16 or fp32 with gradients
    of a supported dtype; those without a gradient are skipped.
    """

    def __init__(self, params, lr=0.02, momentum=0.95, weight_decay=0.1, nesterov=True, ns_steps=5,
                 adamw_lr=3e-4, betas=(0.9, 0.95), eps=1e-8, adamw_weight_decay=0.0, use_muon=None):
        defaults = dict(lr=lr, momentum=momentum, weight_decay=weight_decay, nesterov=nesterov,
                        ns_steps=ns_steps, adamw_lr=adamw_lr, betas=betas, eps=eps,
                        adamw_weight_decay=adamw_weight_decay, use_muon=use_muon)
        super().__init__(params, defaults)

    @staticmethod
    def _is_muon(group, p):
        flag = group["use_muon"]
        return (p.ndim == 2) if flag is None else bool(flag)

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for group in self.param_groups:
            muon = defaultdict(list)    # (W dtype, G dtype) -> [(p, grad, momentum)]
            adam = defaultdict(list)    # (P dtype, G dtype) -> [(p, grad, m, v, step)]
            for p in group["params"]:
                if p.grad is None:
                    continue
                st = self.state[p]
                if self._is_muon(group, p):
                    if p.ndim != 2:
                        raise ValueError("Muon parameters must be matrices")
                    if "momentum" not in st:
                        st["momentum"] = torch.zeros_like(p, dtype=torch.float32)
                    muon[(p.dtype, p.grad.dtype)].append((p, p.grad, st["momentum"]))
                else:
                    if "exp_avg" not in st:
                        st["exp_avg"] = torch.zeros_like(p, dtype=torch.float32)
                        st["exp_avg_sq"] = torch.zeros_like(p, dtype=torch.float32)
                        st["step"] = 0
                    st["step"] += 1
                    adam[(p.dtype, p.grad.dtype, st["step"])].append((p, p.grad, st["exp_avg"], st["exp_avg_sq"]))
            for items in muon.values():
                W, G, M = zip(*items)
                muon_step_ex(W, G, M, group["lr"], group["momentum"], group["weight_decay"],
                             steps=group["ns_steps"], nesterov=group["nesterov"])
            b1, b2 = group["betas"]
            for (_, _, step), items in adam.items():
                P, G, M, V = zip(*items)
                muon_adamw_step(P, G, M, V, lr=group["adamw_lr"], beta1=b1, beta2=b2, eps=group["eps"],
                                wd=group["adamw_weight_decay"], step=step)
        return loss
