"""Host-side logic of the benchmark and the plan builder (no GPU): replica
aggregation over ranks (world size 2 on gloo), clock-sample parsing, the
roofline arithmetic and the launch counter."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import quantized_skinny_gemm_gb300 as dg
from quantized_skinny_gemm_gb300 import plans


def test_floor_matches_the_pages_weight_read_arithmetic():
    # 1.4 GB of fp16 weights per step at 44 GB/s is about a 32 ms floor
    # ("MiniCPM-V on Orange Pi AIPro (Ascend 310B)", closing paragraph)
    assert bench.floor_seconds(1.4e9, 44) * 1e3 == pytest.approx(31.8, abs=0.1)
    # the 28-layer fp16 decoder step at the measured 6782.1 GB/s
    assert bench.floor_seconds(2620391424, 6782.1) * 1e6 == pytest.approx(386.4, abs=0.1)


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput_gbs(1e9, 10, 1, 1.0) == pytest.approx(10.0)
    assert bench.job_throughput_gbs(1e9, 10, 4, 2.0) == pytest.approx(20.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        secs = bench.max_over_ranks(1.0 + rank, dist, "cpu")
        out[rank] = secs
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_time_world2():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_clock_parsing_and_throttle_reasons():
    text = ("1965, 2070, 900.1, Not Active, Not Active, Not Active, Active\n"
            "2070, 2070, 1200.3, Not Active, Not Active, Not Active, Not Active\n"
            "1980, 2070, 1300.0, Not Active, Active, Not Active, Not Active\n"
            "[N/A], 2070, 1.0, x, x, x, x\n")
    c = bench.parse_clock_samples(text)
    assert c["samples"] == 3 and c["sm_mhz"] == 1980.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def _lin(kind, M, N, K, x, y=0, token=0, x_i8=0):
    return dg.Linear(kind=kind, M=M, N=N, K=K, group_size=32, W=0x1000, x=x, y=y or 0x9000,
                     token=token or None, x_i8=x_i8 or None, logits=0x8000 if token else None)


def test_launch_counter_matches_the_fusion_rule():
    X, Y = 0x100000, 0x200000
    layer = [_lin(0, 1, 8, 16, X), _lin(0, 1, 8, 16, X), _lin(0, 1, 8, 16, X),
             _lin(0, 1, 8, 16, Y), _lin(0, 1, 8, 16, X + 64), _lin(0, 1, 8, 16, X + 64),
             _lin(0, 1, 8, 32, X + 128)]
    assert plans.count_launches(layer) == 1                  # one persistent launch
    assert plans.count_launches(layer, persistent=False) == 4  # q|k|v, o, gate|up, down
    two = [_lin(0, 2, 8, 16, X), _lin(0, 2, 8, 16, X)]
    assert plans.count_launches(two) == 1                    # fused, per-group (M = 2)
    head = [_lin(3, 1, 8, 32, X, token=0x7000)]
    assert plans.count_launches(head, persistent=False) == 2  # lm_head + argmax pass
