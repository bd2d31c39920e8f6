"""Multi-rank host logic on CPU: the unit split and the max-over-ranks timing
reduction, run as two gloo ranks (no GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from head_dim_attention_gb300.shard import max_over_ranks, shard, units


def test_shard_covers_every_unit_once():
    for batch, hkv, world in [(1, 8, 2), (2, 3, 4), (1, 1, 3), (3, 5, 1), (4, 8, 8)]:
        u = units(batch, hkv)
        parts = [shard(u, r, world) for r in range(world)]
        flat = [x for p in parts for x in p]
        assert sorted(flat) == sorted(u)
        assert len(set(flat)) == len(flat)
        sizes = [len(p) for p in parts]
        assert max(sizes) - min(sizes) <= 1


def test_shard_rejects_bad_rank():
    with pytest.raises(ValueError):
        shard(units(1, 2), 2, 2)
    with pytest.raises(ValueError):
        shard(units(1, 2), 0, 0)


def test_max_without_process_group_is_identity():
    assert max_over_ranks(3.5) == 3.5


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = shard(units(1, 8), rank, world)
        elapsed = 10.0 + rank  # each rank's own time
        out[rank] = (mine, max_over_ranks(elapsed))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert sorted(res) == [0, 1]
    got = sorted(x for r in res for x in res[r][0])
    assert got == units(1, 8)
    assert all(res[r][1] == 11.0 for r in res)  # MAX over the ranks' times
