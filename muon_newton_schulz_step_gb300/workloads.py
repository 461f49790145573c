"""Seeded synthetic workloads for the Muon step (inputs only, no Muon arithmetic).

Shared by the tests, the benchmark and the oracle checks: this module only
draws matrices; it holds none of the method's arithmetic.

The shapes follow the model in "How PyTorch Scaled a Near-1T MoE on Europe's
Public Supercomputer", section "Introduction" (hidden size 6,144, 384 routed
experts) with four-way expert parallelism inside a node ("The real problem
was the system balance"), i.e. 96 experts per rank whose whole matrices sit on
that rank (FlexShard bullet of "Three optimizations that changed the
economics").  The expert width 2048 and the gradient spectra are this
library's synthetic choices.  No public dataset is involved.

Every matrix i of workload w is drawn from its own generator seeded with
1_000_003 * w.seed_id + i (gradient), + 500_000_009 (weights), + 2 * 500_000_009
(momentum), so any subset of a workload can be regenerated alone.
"""
from dataclasses import dataclass, field
import math
from typing import List, Optional

import torch

SEED_STRIDE = 1_000_003
STREAM_W = 500_000_009
STREAM_M = 2 * 500_000_009


@dataclass(frozen=True)
class MatrixSpec:
    rows: int
    cols: int
    spectrum: str            # "uniform" | "loguniform" | "const" | "none"
    rank: Optional[int]      # None = full rank min(rows, cols); 0 = no low-rank part
    lo: float = 0.0
    hi: float = 0.0
    noise: float = 0.0       # std of the added Gaussian noise
    role: str = ""


@dataclass
class Workload:
    name: str
    seed_id: int
    call: str                # "step" (full Muon step) or "ns" (Newton-Schulz only)
    mats: List[MatrixSpec]
    g_dtype: torch.dtype = torch.bfloat16
    w_dtype: torch.dtype = torch.bfloat16
    lr: float = 0.02
    mu: float = 0.95
    wd: float = 0.1
    m_std: float = 1e-3      # 0 -> zeros
    w_std: float = 0.02
    on_host: bool = False    # draw on the CPU generator (small workloads)
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def count(self) -> int:
        return len(self.mats)

    def shapes(self):
        return [(s.rows, s.cols) for s in self.mats]


def nominal_ns_flops(rows: int, cols: int, steps: int = 5) -> float:
    """Nominal Newton-Schulz FLOPs of one matrix: steps * (4 r^2 k + 2 r^3),
    r = min, k = max (Gram 2r^2k + polynomial 2r^3 + update 2r^2k)."""
    r, k = min(rows, cols), max(rows, cols)
    return steps * (4.0 * r * r * k + 2.0 * r ** 3)


def _expert(rows, cols, role, spectrum="loguniform", rank=16, lo=1e-2, hi=1.0, noise=1e-3):
    return MatrixSpec(rows, cols, spectrum, rank, lo, hi, noise, role)


def workload(name: str) -> Workload:
    if name == "tiny":
        mats = [MatrixSpec(64, 256, "uniform", 4, 0.1, 10.0, 1e-3, "tiny") for _ in range(8)]
        return Workload("tiny", 1, "step", mats, g_dtype=torch.float32, w_dtype=torch.float32,
                        m_std=0.0, on_host=True,
                        description="8 x 64x256 fp32 G = rank-4 (s~U[0.1,10]) + N(0,1e-3); M = 0; "
                                    "W N(0,0.02) fp32; one Muon step")
    if name == "expert_gate":
        mats = [_expert(2048, 6144, "gate") for _ in range(96)]
        return Workload("expert_gate", 2, "ns", mats,
                        description="96 x 2048x6144 bf16, rank-16 (log-U[1e-2,1]) + N(0,1e-3); NS5 only")
    if name == "dense_attn":
        mats = [MatrixSpec(6144, 6144, "const", 32, 0.1, 0.1, 1e-3, "attn") for _ in range(4)]
        mats += [MatrixSpec(1024, 6144, "const", 32, 0.1, 0.1, 1e-3, "kv") for _ in range(2)]
        return Workload("dense_attn", 3, "step", mats,
                        description="4 x 6144^2 + 2 x 1024x6144 bf16 G = N(0,1e-3) + rank-32 spike (0.1); "
                                    "M N(0,1e-3) fp32; W N(0,0.02) bf16; full Muon step")
    if name == "moe_layer":
        mats = []
        for _ in range(96):
            mats += [_expert(2048, 6144, "gate"), _expert(2048, 6144, "up"), _expert(6144, 2048, "down")]
        return Workload("moe_layer", 4, "step", mats,
                        description="96 experts x {gate 2048x6144, up 2048x6144, down 6144x2048} = 288 "
                                    "matrices; bf16 G rank-16 + N(0,1e-3), M N(0,1e-3) fp32, W N(0,0.02) "
                                    "bf16; lr 0.02, mu 0.95, wd 0.1; full Muon step")
    if name == "mixed_block":
        mats = []
        full = dict(spectrum="loguniform", rank=None, lo=1e-3, hi=1.0, noise=0.0)
        for _ in range(96):
            mats += [_expert(2048, 6144, "gate", **full), _expert(2048, 6144, "up", **full),
                     _expert(6144, 2048, "down", **full)]
        mats += [_expert(6144, 6144, "q", **full), _expert(1024, 6144, "k", **full),
                 _expert(1024, 6144, "v", **full), _expert(6144, 6144, "o", **full)]
        mats += [_expert(2048, 6144, "shared", **full) for _ in range(3)]
        perm = torch.randperm(len(mats), generator=torch.Generator().manual_seed(0)).tolist()
        mats = [mats[i] for i in perm]
        return Workload("mixed_block", 5, "step", mats,
                        description="288 expert matrices + q,o 6144^2, k,v 1024x6144, 3 shared 2048x6144 "
                                    "(295, order shuffled with seed 0); full-rank spectra log-U[1e-3,1]")
    raise KeyError(name)


WORKLOADS = ("tiny", "expert_gate", "dense_attn", "moe_layer", "mixed_block")


def _haar(n, k, gen, device):
    a = torch.randn(n, k, generator=gen, device=device, dtype=torch.float32)
    # thin factors are orthonormalised on the host (cheap, and no device linear-algebra
    # library is needed); full-rank ones on the device
    q, r = torch.linalg.qr(a.cpu() if k <= 64 else a)
    return (q * torch.sign(torch.diagonal(r)).unsqueeze(0)).to(device)


def _spectrum(spec: MatrixSpec, k: int, gen, device):
    u = torch.rand(k, generator=gen, device=device, dtype=torch.float32)
    if spec.spectrum == "uniform":
        return spec.lo + (spec.hi - spec.lo) * u
    if spec.spectrum == "loguniform":
        return torch.exp(math.log(spec.lo) + (math.log(spec.hi) - math.log(spec.lo)) * u)
    if spec.spectrum == "const":
        return torch.full((k,), spec.lo, device=device, dtype=torch.float32)
    raise ValueError(spec.spectrum)


def gradient(w: Workload, i: int, device) -> torch.Tensor:
    """fp32 gradient of matrix i: U diag(s) V^T (+ Gaussian noise)."""
    spec = w.mats[i]
    dev = "cpu" if w.on_host else device
    gen = torch.Generator(device=dev).manual_seed(SEED_STRIDE * w.seed_id + i)
    m, n = spec.rows, spec.cols
    g = torch.zeros(m, n, device=dev, dtype=torch.float32)
    rank = min(m, n) if spec.rank is None else spec.rank
    if rank > 0 and spec.spectrum != "none":
        U = _haar(m, rank, gen, dev)
        V = _haar(n, rank, gen, dev)
        s = _spectrum(spec, rank, gen, dev)
        g += (U * s.unsqueeze(0)) @ V.T
    if spec.noise > 0:
        g += spec.noise * torch.randn(m, n, generator=gen, device=dev, dtype=torch.float32)
    return g.to(device)


def weights(w: Workload, i: int, device) -> torch.Tensor:
    spec = w.mats[i]
    dev = "cpu" if w.on_host else device
    gen = torch.Generator(device=dev).manual_seed(SEED_STRIDE * w.seed_id + i + STREAM_W)
    t = w.w_std * torch.randn(spec.rows, spec.cols, generator=gen, device=dev, dtype=torch.float32)
    return t.to(w.w_dtype).to(device)


def momentum(w: Workload, i: int, device) -> torch.Tensor:
    spec = w.mats[i]
    if w.m_std == 0.0:
        return torch.zeros(spec.rows, spec.cols, device=device, dtype=torch.float32)
    dev = "cpu" if w.on_host else device
    gen = torch.Generator(device=dev).manual_seed(SEED_STRIDE * w.seed_id + i + STREAM_M)
    t = w.m_std * torch.randn(spec.rows, spec.cols, generator=gen, device=dev, dtype=torch.float32)
    return t.to(device)


def make_inputs(w: Workload, device, indices=None):
    """Lists W, G, M for the chosen matrices (all by default).  For an "ns"
    workload only G is drawn (the matrices to orthogonalise, bf16)."""
    idx = range(w.count) if indices is None else list(indices)
    G = [gradient(w, i, device).to(w.g_dtype) for i in idx]
    if w.call == "ns":
        return {"G": G}
    W = [weights(w, i, device) for i in idx]
    M = [momentum(w, i, device) for i in idx]
    return {"W": W, "G": G, "M": M}
