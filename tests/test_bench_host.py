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
