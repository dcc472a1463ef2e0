"""Host-side logic of bench.py, without a GPU: the multi-rank aggregation
(world_size 2 over gloo on CPU) and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(values[rank], "cpu")
        out_q.put((rank, slowest, bench.aggregate_gbs(1000, slowest, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [2.5, 4.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest replica's time; throughput counts both replicas
    assert [g[1] for g in got] == [4.0, 4.0]
    assert got[0][2] == pytest.approx(2 * 1000 / 4.0e-3 / 1e9)


def test_single_process_aggregation_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.aggregate_gbs(18350080, 0.004, 1) == pytest.approx(18350080 / 4e-6 / 1e9)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "1", "--ref-seconds", "2"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["steps"] == 3 and j["warmup"] == 1
    assert j["unit"] == "GB/s" and j["higher_is_better"] is True and j["value"] > 0
    import bench
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] == bench.host_threads()
    assert j["e2e"]["h2d_bytes_per_step"] == 0
