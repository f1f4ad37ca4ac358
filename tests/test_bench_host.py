"""Host-side logic of the benchmark: clock-record parsing, whole-job
throughput, the N > 1 path (barrier + max over ranks) on two gloo ranks, the
per-kernel rate table and the lookup of committed DRAM-traffic figures."""

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


def test_kernel_table_rates():
    """Contractions get TFLOP/s from 2 rows d V per launch (the forward over the
    rows whose logits are formed, the backward over the valid rows); the single
    sweep's gated recompute gets a time but no rate; the cached-column pass is
    rated in GB/s from 14 K bytes per valid row."""
    ks = {"logits_fwd": (4, 40.0), "logits_bwd": (4, 0.1), "dh": (4, 36.0), "dW": (4, 38.0),
          "sweep_fix": (4, 0.2)}
    T, nv, d, V, K = 1000, 900, 64, 5000, 10
    t = bench.kernel_table(ks, 2, T, nv, d, V, K, sweep=True)
    assert t["logits_fwd"]["flops_per_launch"] == 2.0 * T * d * V * 2 / 4
    assert t["dh"]["flops_per_launch"] == 2.0 * nv * d * V * 2 / 4
    assert "tflops" not in t["logits_bwd"] and "note" in t["logits_bwd"]
    assert t["sweep_fix"]["bytes_per_launch"] == 14.0 * K * nv * 2 / 4
    split = bench.kernel_table(ks, 2, T, nv, d, V, K, sweep=False)
    assert split["logits_bwd"]["flops_per_launch"] == 2.0 * nv * d * V * 2 / 4


def test_traffic_matches_workload_and_chunk(tmp_path, monkeypatch):
    """A committed DRAM-traffic figure is reported only for the workload and
    chunk size it was captured on, and only while the device code hashes the
    same."""
    import json
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.device_source_sha256()
    (prof / "traffic.json").write_text(json.dumps({
        "dh": {"bytes_per_launch": 123, "workload": "ctx_32k", "chunk": 8192, "device_sha256": h},
        "dW": {"bytes_per_launch": 456, "workload": "ctx_32k", "chunk": 8192,
               "device_sha256": "0" * 64}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "device_source_sha256", lambda: h)
    assert bench.load_traffic("dh", "ctx_32k", 8192) == 123
    assert bench.load_traffic("dh", "ctx_32k", 4096) is None
    assert bench.load_traffic("dh", "ctx_8k", 8192) is None
    assert bench.load_traffic("dW", "ctx_32k", 8192) is None
    assert bench.load_traffic("nothing", "ctx_32k", 8192) is None
