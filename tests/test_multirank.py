"""The N > 1 path of bench.py on the CPU: world-size-2 `gloo` ranks.

The decode path shards by sequence with no exchange, so N GPUs run N independent
replicas; the only cross-rank steps are the barrier and the max-reduction of the
step time, and rank 0 alone prints.  Both are host logic and run here."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        step_ms = [0.120, 0.135][rank]         # rank 1 is the slow one
        ms = bench.max_over_ranks(step_ms, world, "cpu")
        q.put((rank, ms, bench.job_tflops(world, 73.0e9, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, tflops in got:
        assert ms == pytest.approx(0.135)      # every rank sees the slowest rank's time
        assert tflops == pytest.approx(2 * 73.0e9 / 0.135e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(0.25, 1, "cpu") == 0.25
    assert bench.job_tflops(1, 73.0e9, 0.128) == pytest.approx(73.0e9 / 0.128e-3 / 1e12)


def test_reference_arm_on_a_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "1", "--warmup", "0"], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
