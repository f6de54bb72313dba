"""Host-side logic of the benchmark that needs no GPU: the N>1 (torchrun) path with gloo ranks on
the CPU, the weak-scaling aggregate, the reference arm's rank handling, and the traffic record."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.5 + rank, dist)        # rank r took 1.5 + r ms
        value = bench.weak_scaling_value(1000, world, slowest)
        dist.barrier()
        results[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_replica():
    world = 2
    results = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
    for r in range(world):
        slowest, value = results[r]
        assert slowest == 2.5
        assert value == pytest.approx(1000 * world / 2.5e-3)


def test_weak_scaling_value_single_rank():
    assert bench.weak_scaling_value(25165824, 1, 0.2) == pytest.approx(25165824 / 2e-4)


def test_reference_arm_only_rank0_reports():
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), rank=1, world=2) is None


def test_traffic_record_matches_sources_or_is_null():
    t = bench.committed_traffic("scan_fwd_kernel")
    assert t is None or t > 0
    assert bench.committed_traffic("no_such_kernel") is None


def test_workload_config_names_the_workload():
    import ssm_workloads as wl
    c = bench.workload_config(wl.MID)
    assert c["workload"] == wl.MID.name and c["seqlen"] == 2048 and "l2" in c


@pytest.mark.parametrize("batch,dim,world", [(8, 1536, 1), (8, 1536, 2), (8, 1536, 3), (8, 1536, 8), (1, 5120, 8),
                                             (3, 100, 4), (2, 33, 5), (1, 8, 4), (5, 200, 7)])
def test_partition_covers_every_channel_once(batch, dim, world):
    """The ranks' boxes cover every (batch, channel) exactly once, each box is a whole-row range or
    part of one row, and the shares differ by at most one 32-channel unit."""
    seen = {}
    shares = []
    for r in range(world):
        boxes = bench.partition_boxes(batch, dim, world, r)
        n = 0
        for b0, b1, d0, d1 in boxes:
            assert 0 <= b0 < b1 <= batch and 0 <= d0 < d1 <= dim
            assert (d0, d1) == (0, dim) or b1 == b0 + 1
            for b in range(b0, b1):
                for d in range(d0, d1):
                    assert (b, d) not in seen, ("overlap", b, d)
                    seen[(b, d)] = r
            n += (b1 - b0) * (d1 - d0)
        shares.append(n)
    assert len(seen) == batch * dim
    units = [-(-s // 32) for s in shares]
    assert max(shares) - min(shares) <= 32 * (1 + max(units) - min(units))
    per_row = -(-dim // 32)
    assert max(units) - min(units) <= 1 + (per_row if dim % 32 else 0)


def _partition_rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        boxes = bench.partition_boxes(8, 1536, world, rank)
        mine = sum((b1 - b0) * (d1 - d0) for b0, b1, d0, d1 in boxes)
        t = torch.tensor([mine], dtype=torch.int64)
        dist.all_reduce(t)  # test-only check of the union; the benchmark itself needs no collective
        slowest = bench.max_over_ranks(2.0 + rank, dist)
        results[rank] = (int(t.item()), slowest, bench.strong_scaling_value(8 * 1536 * 2048, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_one_workload():
    world = 2
    results = mp.Manager().dict()
    mp.spawn(_partition_rank, args=(world, _free_port(), results), nprocs=world, join=True)
    for r in range(world):
        total, slowest, value = results[r]
        assert total == 8 * 1536
        assert slowest == 3.0
        assert value == pytest.approx(8 * 1536 * 2048 / 3e-3)
