"""Host-side logic of the benchmark: clock-record parsing, whole-job
throughput, and the N > 1 path (barrier + max over ranks) on two gloo ranks."""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def test_parse_clock_csv():
    text = ("0, 1950, 2032, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "0, 1890, 2032, 1100.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "0, 1920, 2032, 1050.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.parse_clock_csv(text)
    assert c["sm_mhz"] == 1920.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.parse_clock_csv("")["samples"] == 0


def test_job_throughput():
    assert bench.job_throughput(32768, 1, 0.5) == 65536.0
    assert bench.job_throughput(100, 4, 2.0) == 200.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, _ = bench.rank_info()
    bench.dist_setup(w, "gloo")
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 + r, w)
    bench.barrier(w)
    q.put((r, m, bench.job_throughput(1000, w, m)))
    torch.distributed.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    assert all(m == 2.5 for _, m, _ in res)          # slowest rank sets the time
    assert all(v == 2000 / 2.5 for _, _, v in res)   # all ranks' units / that time


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)
