"""bench.py's multi-rank host logic on CPU: two gloo ranks (world_size 2, 127.0.0.1).

Each rank times its own replica; the job's step time is the maximum over ranks and the
whole-job throughput counts every rank's tokens.  The GPU timing itself is not exercised
here (no GPU in this test)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) x the time of rank 0 on the first two timings
        mine = [10.0 * (rank + 1), 3.0 * (rank + 1), 7.0 - rank]
        got = bench.reduce_max(mine, dist, "cpu")
        tokens = 4096
        ms_step = got[0] / 5
        out[rank] = (got, bench.job_throughput(tokens, world, ms_step))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_timings_max_reduced_and_throughput_counts_all_ranks():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()        # no fork of a process that runs torch threads
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
    for rank in range(world):
        got, value = out[rank]
        assert got == [20.0, 6.0, 7.0]                 # element-wise max over the ranks
        assert value == pytest.approx(4096 * 2 / (4.0 * 1e-3))   # both replicas' tokens / slowest


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max([1.5, 2.5], None, "cpu") == [1.5, 2.5]
    assert bench.job_throughput(1000, 1, 2.0) == pytest.approx(5e5)


def test_launch_count_per_step():
    import bench
    from chunked_gated_linear_gb300 import synth
    ws = {w.name: w for w in synth.standard_workloads()}
    assert bench.launches_per_step(ws["gdn_fwd_bf16_T4096_H16_d128"]) == 3
    # the varlen prefill (64 slots x 16 heads): the fused plan, one kernel after the metadata
    assert bench.launches_per_step(ws["gdn_varlen_bf16_N32_Nmax64_Tmax65536_H16_d128"]) == 2
    assert bench.fwd_plan_of(ws["gdn_varlen_bf16_N32_Nmax64_Tmax65536_H16_d128"]) == "fused"
    assert bench.launches_per_step(ws["gdn_fwdbwd_bf16_B4_T8192_H16_d128"]) == 6
    assert bench.launches_per_step(ws["kda_fwd_bf16_T2048_H10_d128"]) == 3
    # fp32 with the fastest workspace: the CUDA-core split plan (chunk prep + chain)
    assert bench.fwd_plan_of(ws["gdn_fwd_fp32_T256_H2_d64"]) == "cuda_cores_split"
    assert bench.launches_per_step(ws["gdn_fwd_fp32_T256_H2_d64"]) == 3
    assert bench.launches_per_step(ws["kda_fwdbwd_bf16_T2048_H10_d128"]) == 5
    # one 64K-token sequence of one head: the segmented chain (on any GPU of 24 or more SMs)
    assert bench.launches_per_step(ws["gdn_fwd_bf16_T65536_H1_d128"]) == 5
    assert bench.launches_per_step(ws["kda_fwd_bf16_T65536_H1_d128"]) == 5
    # chunk size 32 runs the CUDA-core split plan; fp16 (GDN, d = 128) the transition form
    assert bench.launches_per_step(ws["gdn_fwd_f16_T4096_H16_d128"]) == 3       # fp16: tensor cores
    assert bench.launches_per_step(ws["gdn_fwd_bf16_bt32_T4096_H16_d128"]) == 3
