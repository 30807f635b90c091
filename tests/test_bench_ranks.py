"""The whole-job aggregation of bench.py over ranks (world size 2, gloo, CPU).

Each rank reports its own time; the job's time is the slowest rank's, taken
by an all-reduce MAX, and the whole-job rate counts the units of every rank
(replicas, weak scaling).  This is the host logic of `bench.py --gpus N`
under torchrun, run here with the gloo backend instead of NCCL.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seconds, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(seconds[rank], world)
        rate = bench.job_rate(1000.0, world, t)
        out.put((rank, t, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_units_add_up():
    world = 2
    seconds = [0.5, 2.0]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, seconds, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get(timeout=5) for _ in range(world))
    for rank, t, rate in got:
        assert t == 2.0                              # the slowest rank, on every rank
        assert rate == pytest.approx(world * 1000.0 / 2.0)


def test_single_rank_is_the_identity():
    import bench

    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_rate(10.0, 1, 2.0) == 5.0


def test_recorded_traffic_matches_problems_and_sources():
    import bench

    ent = {"source_hash": "abc", "per_problem": [
        {"case": "4096,6144,16", "variant": "tc_decode:16:1:8", "dram_read": 100.0, "dram_write": 4.0},
        {"case": "4096,4096,16", "variant": "tc_decode:16:1:8", "dram_read": 60.0, "dram_write": 0.0},
    ]}
    v8 = dict(kernel="tc_decode", block_m=16, split_k=1, dq_warps=8)
    v12 = dict(v8, dq_warps=12)
    both = [(4096, 6144, 16, v8), (4096, 4096, 16, v8)]
    assert bench.recorded_traffic(ent, "abc", both) == 82
    assert bench.recorded_traffic(ent, "other", both) is None          # sources changed
    assert bench.recorded_traffic(ent, "abc", [(4096, 6144, 16, v12)]) is None   # another variant
    assert bench.recorded_traffic(ent, "abc", both + [(4096, 28672, 16, v8)]) is None  # not captured
    assert bench.recorded_traffic(ent, "abc", []) is None
