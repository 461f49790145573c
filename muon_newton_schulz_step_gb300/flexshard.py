"""Whole-matrix placement of Muon work across ranks (host-side planner).

"How PyTorch Scaled a Near-1T MoE on Europe's Public Supercomputer", section
"Three optimizations that changed the economics", FlexShard bullet: Newton-
Schulz works on full matrices, so sharding every matrix across ranks forces a
gather and a scatter per step; placing whole experts on ranks instead makes
each orthogonalisation local, with no communication.

This module decides that placement.  A *group* is a set of matrices that must
stay together (one expert's gate, up and down projections); groups are
assigned to ranks greedily, largest nominal Newton-Schulz cost first, each to
the currently least-loaded rank (longest-processing-time rule), with ties
broken by the lowest rank so that every rank computes the same plan without
talking to the others.  The plan is a pure function of the shapes, so each
rank derives its own share locally; no collective is involved.
"""
from typing import List, Optional, Sequence, Tuple

from .workloads import nominal_ns_flops


def group_costs(shapes: Sequence[Tuple[int, int]], groups: Sequence[Sequence[int]], steps: int = 5):
    return [sum(nominal_ns_flops(*shapes[i], steps=steps) for i in g) for g in groups]


def assign(shapes: Sequence[Tuple[int, int]], world_size: int,
           groups: Optional[Sequence[Sequence[int]]] = None, steps: int = 5) -> List[int]:
    """Rank of every matrix.  ``groups`` defaults to one group per matrix."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    n = len(shapes)
    if groups is None:
        groups = [[i] for i in range(n)]
    seen = sorted(i for g in groups for i in g)
    if seen != list(range(n)):
        raise ValueError("groups must cover every matrix exactly once")
    costs = group_costs(shapes, groups, steps)
    order = sorted(range(len(groups)), key=lambda gi: (-costs[gi], gi))
    load = [0.0] * world_size
    owner = [-1] * n
    for gi in order:
        r = min(range(world_size), key=lambda k: (load[k], k))
        load[r] += costs[gi]
        for i in groups[gi]:
            owner[i] = r
    return owner


def local_indices(shapes, rank: int, world_size: int, groups=None, steps: int = 5) -> List[int]:
    """Indices (in input order) of the matrices rank `rank` owns."""
    owner = assign(shapes, world_size, groups, steps)
    return [i for i, r in enumerate(owner) if r == rank]


def rank_loads(shapes, world_size: int, groups=None, steps: int = 5) -> List[float]:
    owner = assign(shapes, world_size, groups, steps)
    load = [0.0] * world_size
    for i, r in enumerate(owner):
        load[r] += nominal_ns_flops(*shapes[i], steps=steps)
    return load


def expert_groups(n_experts: int, per_expert: int = 3) -> List[List[int]]:
    """Groups for matrices laid out expert by expert (gate, up, down, gate, ...)."""
    return [list(range(e * per_expert, (e + 1) * per_expert)) for e in range(n_experts)]
