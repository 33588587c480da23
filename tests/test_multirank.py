"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): heads
are split into disjoint contiguous ranges covering every head, with no
collective on the data path; the job time is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


@pytest.mark.parametrize("H", [1, 2, 7, 40, 56])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_head_ranges_partition_the_heads(H, world):
    seen = []
    for r in range(world):
        lo, hi = bench.head_range(H, world, r)
        assert 0 <= lo <= hi <= H
        seen.extend(range(lo, hi))
    assert seen == list(range(H))
    sizes = [bench.head_range(H, world, r)[1] - bench.head_range(H, world, r)[0] for r in range(world)]
    assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        lo, hi = bench.head_range(56, w, r)
        t = bench.max_over_ranks(10.0 + 5.0 * r, "cpu")          # rank 1 is the slow one
        heads = torch.zeros(56, dtype=torch.int64)
        heads[lo:hi] = 1
        dist.all_reduce(heads)                                  # test-side check only
        out[r] = (lo, hi, t, int(heads.min()), int(heads.max()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_heads_and_take_the_max_time():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][:2] == (0, 28) and out[1][:2] == (28, 56)
    assert out[0][2] == out[1][2] == 15.0
    assert all(v[3] == 1 and v[4] == 1 for v in out.values())   # every head on exactly one rank
