"""Host-side logic of bench.py without a GPU: the max-over-ranks timing under a real
two-rank gloo process group, the whole-job value, and the reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_step, other = bench.combine_over_ranks([1.0 + rank, 5.0 - rank], dist, "cpu")
        out.put((rank, ms_step, other, bench.whole_job_rows_per_s(256, world, ms_step)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_step, other, value in results:
        assert ms_step == 2.0 and other == 5.0          # max over ranks, same on every rank
        assert value == pytest.approx(256 * 2 / 2e-3)


def test_single_process_values_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_over_ranks([3.0, 4.5], None) == [3.0, 4.5]
    assert bench.algorithmic_bytes(R=2, V=10, W=8, B=1) == 2 * 10 * 4 + 2 * 8 * 8 + 2 * 8 + 2 * 4


def test_reference_arm_json_line_on_cpu():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, env=env,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in line, key
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
