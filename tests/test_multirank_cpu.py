"""The bench's multi-rank path on CPU with gloo (world size 2): each rank
runs its own replica, the slowest rank's time sets the job time, and the
job throughput sums the ranks' work (weak scaling, no data-path
collective)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.0, 30.0][rank]                     # rank 1 is the slow one
    ms_max = bench.reduce_max(dist, ms, "cpu")
    out[rank] = (ms_max, bench.job_throughput(1e12, world, ms_max))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_aggregate():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms_max, tput = res[0]
    assert ms_max == 30.0
    assert tput == pytest.approx(2 * 1e12 / 0.030 / 1e12)


def test_single_process_identity():
    import bench
    assert bench.reduce_max(None, 7.5) == 7.5
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)


def test_both_bench_arms_report_the_same_config():
    """The reference arm's JSON line describes the same workload object as the
    library arm's, for every schedule and forward variant."""
    import argparse
    import bench
    for schedule, fwd, world in (("ring", "partials", 1), ("ring", "fused", 2), ("a2a", "partials", 1)):
        args = argparse.Namespace(schedule=schedule, fwd=fwd)
        w = bench.get_workload("large")
        cfg = bench.bench_config(w, args, world)
        assert cfg == bench.bench_config(w, args, world)
        assert cfg["workload"].startswith("large: B=64 x S=8192")
        assert cfg["forward"] == ("fused online softmax" if (fwd == "fused" or schedule == "a2a")
                                  else "ring-step partials + LSE merge")
        assert cfg["parallelism"] == ("replicas x2" if world == 2 else "1 GPU, CP emulated")


def test_kernel_attribution_splits_a_steps_work_over_its_launches():
    """A kernel launched several times a step (the dQ and dK passes of the
    backward that keeps dS: once per kv head) is credited the step's work
    divided by its launches a step; a kernel whose work is given per launch
    (the pack) keeps it."""
    import bench
    U = 3.0e12
    work = {"attn_bwd_dq": ("tensor", 3.0 * U, "step"), "thd_pack": ("hbm", 8.0e9, "launch")}
    pk = {"bf16_sustained": 1700.0, "hbm": 6800.0}
    steps = 2
    prof = [("attn_bwd_dq", 10.0)] * (8 * steps) + [("thd_pack", 2.0)] * (4 * steps)
    kernels, agg = bench.attribute_kernels(prof, work, steps, pk)
    dq = kernels["attn_bwd_dq"]
    assert dq["launches_per_step"] == 8 and dq["ms_per_launch"] == 10.0
    assert abs(dq["achieved"] - (3.0 * U / 8) / 10e-3 / 1e12) < 0.01
    assert abs(dq["frac"] - dq["achieved"] / 1700.0) < 1e-4
    pack = kernels["thd_pack"]
    assert abs(pack["achieved"] - 8.0e9 / 2e-3 / 1e9) < 0.01
    assert agg["attn_bwd_dq"] == [16, 160.0]
