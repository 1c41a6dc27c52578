"""Multi-rank logic of bench.py on CPU: two gloo ranks, each timing a
different (fake) step, must agree on the slowest rank's time and report the
whole-job throughput of independent replicas (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.5, 3.0][rank]
        m = bench.max_over_ranks(ms, torch.device("cpu"))
        q.put((rank, m, bench.aggregate(3.0e12, world, m)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, agg in got:
        assert m == 3.0
        # two replicas of a 3e12-flop problem in 3 ms -> 2000 TFLOP/s
        assert agg == pytest.approx(2000.0)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(1.25, torch.device("cpu")) == 1.25
    assert bench.aggregate(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_selected_flops_matches_workload_count():
    # the bench recounts effective FLOPs from a selection held in tensors (the
    # GPU's own selection); on the seeded workloads it must equal their count
    import bench
    import workloads as W
    for cfg in (3, 4):
        w = W.make_workload(cfg)
        assert bench.selected_flops(w.q2k_idx, w.q2k_num, w.block_sizes, w.D) == W.effective_flops(w)
