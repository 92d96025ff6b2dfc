"""bench.py host logic on CPU: multi-rank aggregation with gloo (world size 2),
the JSON contract of the reference arm, and the clock summary parser."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
import bench
world, rank, _ = bench.dist_env()
bench.init_dist(world, "gloo")
bench.barrier(world)
secs = 1.0 + rank            # rank 1 is the slow one
m = bench.max_over_ranks(secs, world)
v = bench.aggregate(1000_000_000, 10, world, m)
if rank == 0:
    print(json.dumps({"max": m, "value": v}))
dist.destroy_process_group()
"""


def test_two_rank_max_and_aggregate(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER)
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script), ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = json.loads(outs[0][0].strip().splitlines()[-1])
    assert res["max"] == 2.0                      # the slowest rank's time
    assert res["value"] == pytest.approx(2 * 1e9 * 10 / 2.0 / 1e9)   # both ranks' bytes


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate(2e9, 5, 1, 2.0) == pytest.approx(5.0)


def test_clock_summary_parser(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    f = tmp_path / "clk.csv"
    f.write_text("0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active\n"
                 "0, 2070, 2070, 1000.2, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "0, 2070, 2070, 1000.2, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.path, c.proc = str(f), object()
    s = c.summary(0, 0)
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_workload_table_and_bytes():
    sys.path.insert(0, ROOT)
    from rmsnorm_fwd_bwd_gb300 import inputs
    w = inputs.WORKLOADS[inputs.HEADLINE]
    assert (w.M, w.N, w.dtype) == (65536, 4096, "bfloat16")
    assert w.fwd_bytes() == 1_074_012_160
    assert w.bwd_bytes() == 1_610_891_264


def test_recorded_traffic_follows_its_sources(tmp_path):
    """A traffic record counts only while the files it names hash to its digest;
    an unknown file or a stale digest gives null."""
    sys.path.insert(0, ROOT)
    import bench
    srcs = ["bwd.cu", "launch.h"]
    rec = {"k": {"dram_bytes_per_launch": 123.0, "sources": srcs,
                 "source_digest": bench.kernel_source_digest(srcs)}}
    path = tmp_path / "t.json"
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("k", path=str(path)) == 123.0
    assert bench.recorded_traffic("missing", path=str(path)) is None
    rec["k"]["source_digest"] = "0" * 16
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("k", path=str(path)) is None
    rec["k"]["sources"] = ["no_such_file.cu"]
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("k", path=str(path)) is None
    # without "sources" the digest covers every kernel file
    rec = {"k": {"dram_bytes_per_launch": 7.0, "source_digest": bench.kernel_source_digest()}}
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("k", path=str(path)) == 7.0
    # a recorded plan must match the current one
    rec["k"]["plan"] = "tma cluster=1 threads=128"
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("k", plan="tma cluster=1 threads=128", path=str(path)) == 7.0
    assert bench.recorded_traffic("k", plan="tma cluster=2 threads=128", path=str(path)) is None
