"""N > 1 host logic on CPU: FlexShard-style whole-matrix placement and the
benchmark's max-over-ranks timing, run as world-size-2 gloo process groups.
The Muon step itself needs no collective (every matrix is independent)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from muon_newton_schulz_step_gb300 import flexshard
from muon_newton_schulz_step_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_assignment_is_a_partition_and_balanced():
    w = wl.workload("mixed_block")
    shapes = w.shapes()
    for world in (1, 2, 3, 4, 8):
        owner = flexshard.assign(shapes, world)
        assert sorted(set(owner)) == list(range(min(world, len(shapes))))
        loads = flexshard.rank_loads(shapes, world)
        biggest = max(wl.nominal_ns_flops(*s) for s in shapes)
        # LPT: the spread between ranks never exceeds the largest single item
        assert max(loads) - min(loads) <= biggest + 1e-6 * max(loads)
        assert abs(sum(loads) - sum(wl.nominal_ns_flops(*s) for s in shapes)) < 1e-6 * sum(loads)


def test_expert_groups_stay_together():
    w = wl.workload("moe_layer")
    shapes = w.shapes()
    groups = flexshard.expert_groups(96)
    owner = flexshard.assign(shapes, 4, groups)
    for g in groups:
        assert len({owner[i] for i in g}) == 1
    # 96 identical experts over 4 ranks: exactly 24 experts (72 matrices) each
    assert [owner.count(r) for r in range(4)] == [72, 72, 72, 72]


def test_bad_groups_rejected():
    with pytest.raises(ValueError):
        flexshard.assign([(4, 4), (4, 4)], 2, groups=[[0], [0]])
    with pytest.raises(ValueError):
        flexshard.assign([(4, 4)], 0)


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = wl.workload("mixed_block")
        shapes = w.shapes()
        mine = flexshard.local_indices(shapes, rank, world)
        # every rank derives its share locally; gather them only to check the partition
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        # the benchmark's timing reduction: the job time is the max over ranks
        t = torch.tensor([10.0 + rank], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.barrier()
        q.put((rank, gathered, float(t.item())))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_partition_and_max_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    n = wl.workload("mixed_block").count
    for rank, gathered, tmax in out:
        assert tmax == 11.0
        flat = sorted(i for part in gathered for i in part)
        assert flat == list(range(n))
        assert set(gathered[0]).isdisjoint(gathered[1])
