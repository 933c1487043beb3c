"""bench.py's multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank of a multi-GPU run times its own replica of the workload; the
reported time is the maximum over ranks and the value counts the work of
every rank. The reference arm runs on rank 0 only.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                      # rank 1 is the slowest
        bench.barrier(world)
        out[rank] = bench.max_over_ranks(mine, world)
        assert bench.dist_env()[:2] == (rank, world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_whole_job_value_counts_all_ranks():
    # 1e12 FLOP per step, 10 steps, 4 ranks, slowest rank 20 ms -> 2000 TFLOP/s
    assert bench.whole_job_value(1e12, 10, 4, 20.0) == pytest.approx(2000.0)
    assert bench.whole_job_value(1e12, 10, 1, 20.0) == pytest.approx(500.0)


def test_reference_arm_only_on_rank0(capsys):
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    from flashattention_fa_fwd_gb300.inputs import WORKLOADS

    assert bench.reference_arm(args, WORKLOADS["f32_single_head_m256_n512_d64"], 1, 2) == 0
    assert capsys.readouterr().out == ""


def test_clock_summary_and_rejection():
    rows = [["0", "2070", "2070", "700", "0x0", "Not Active", "Not Active", "Not Active", "Active"],
            ["0", "1980", "2070", "900", "0x4", "Not Active", "Not Active", "Not Active", "Active"]]
    c = bench.summarize_clocks(rows)
    assert c["sm_mhz"] == 2025.0 and c["reasons"] == ["sw_power_cap"] and not bench.clocks_rejected(c)
    rows[1][7] = "Active"
    assert bench.clocks_rejected(bench.summarize_clocks(rows))
    assert bench.clocks_rejected({"sm_mhz": 900.0, "sm_max_mhz": 2070.0, "reasons": []})
