"""Host-side logic of bench.py (no GPU): algorithmic byte/FLOP accounting,
the committed-traffic lookup, the clock-sample parser, and the multi-rank
reduction over a 2-process gloo group."""
import json
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from w4a16_int4_weight_sigmoid_gb300 import workload as wl


def test_algorithmic_bytes_and_flops():
    sh = wl.EP8_DECODE
    a = bench.algorithmic(sh, touched=22, rows=73)
    w13 = 2 * 2048 * 7168 // 2 + 2 * 2048 * (7168 // 32) * 2
    assert a["gate_up"]["bytes"] == 22 * w13 + 73 * 7168 * 2 + 73 * 2048 * 2
    assert a["gate_up"]["flops"] == 2 * 73 * 4096 * 7168
    w2 = 7168 * 2048 // 2 + 7168 * (2048 // 32) * 2
    assert a["down"]["bytes"] == 22 * w2 + 73 * 2048 * 2 + 73 * 7168 * 2
    assert a["down"]["flops"] == 2 * 73 * 7168 * 2048


def test_committed_traffic_requires_matching_sources(tmp_path, monkeypatch):
    sha = bench.source_sha(bench.KERNEL_SOURCES["small"])
    rec = [{"kernel": "gate_up", "workload": "w", "path": "small", "source_sha": sha,
            "dram_bytes_per_launch": 123}]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_sha", lambda files: sha)
    assert bench.committed_traffic("gate_up", "w", "small") == 123
    assert bench.committed_traffic("gate_up", "w", "large") is None
    monkeypatch.setattr(bench, "source_sha", lambda files: "changed")
    assert bench.committed_traffic("gate_up", "w", "small") is None


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(None)
    c.out = ("0, 1965, 2070, 650.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
             "0, 2070, 2070, 700.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
             "garbage line\n")
    s = c.summary()
    assert s["samples"] == 2 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    assert s["sm_mhz"] == (1965 + 2070) / 2


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    q.put((r, bench.allreduce_max(10.0 + r, w)))
    dist.destroy_process_group()


def test_two_rank_gloo_max_over_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]
