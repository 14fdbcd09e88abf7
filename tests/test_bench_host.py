"""Host-side tests of bench.py: the multi-rank aggregation on gloo (world
size 2, CPU), and the reference arm's JSON line (the CPU oracle on bounded
samples)."""

import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank_main(rank, world, port, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 10.0 + 5.0 * rank  # the slower rank decides
        t = bench.max_over_ranks(torch, elapsed, dist, "cpu")
        v = bench.job_throughput_gbs(world, 32, 2.0 * (1 << 30), t)
        out_q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_replicas_take_max_time_and_sum_bytes():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, v in res:
        assert t == 15.0
        assert abs(v - 2 * 32 * 2.0 * (1 << 30) / 0.015 / 1e9) < 1e-6
    assert bench.max_over_ranks(torch, 3.0) == 3.0


def test_reference_arm_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-sample-log2", "16", "--ref-n", "20"], capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["warmup"] >= 3


def test_effective_bandwidth_bytes_match_the_page(golden):
    """The bench's algorithmic bytes per permutation, 2 * 2^n * elem, equal the
    byte count the transpose tutorial prints for 4096 x 4096 floats."""
    for n, elem, want in golden("effective_bandwidth.txt"):
        n, elem, want = int(n), int(elem), int(want)
        assert 2.0 * (1 << n) * elem == want
        assert bench.job_throughput_gbs(1, 1, 2.0 * (1 << n) * elem, 1.0) == want / 1e-3 / 1e9
