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


def test_code_only_strips_comments_keeps_strings():
    sys.path.insert(0, ROOT)
    import bench
    src = 'int a = 1;  // note\n// whole line\nasm("x // y");  // z\n\n   \nfloat b;   \n'
    assert bench._code_only(src) == 'int a = 1;\nasm("x // y");\nfloat b;'


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    # The recorded ncu traffic stays valid across comment edits and is voided by a code edit.
    sys.path.insert(0, ROOT)
    import glob
    import shutil
    import bench
    csrc = tmp_path / "ragged_log_probs_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in glob.glob(os.path.join(ROOT, "ragged_log_probs_gb300", "csrc", "*.cuh")):
        shutil.copy(f, csrc)
    h0 = bench.kernel_source_hash()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_source_hash() == h0
    target = csrc / "lp_device.cuh"
    text = target.read_text(encoding="utf-8")
    target.write_text(text + "\n// a comment added at the end\n", encoding="utf-8")
    assert bench.kernel_source_hash() == h0
    target.write_text(text + "\nconstexpr int kUnused = 1;\n", encoding="utf-8")
    assert bench.kernel_source_hash() != h0


def test_recorded_traffic_has_a_committed_capture():
    # Every recorded ncu traffic figure is backed by a committed profile summary that states
    # the same device-code hash and the same bytes per launch (in MB, two decimals).
    sys.path.insert(0, ROOT)
    import glob
    import bench
    texts = [open(f, encoding="utf-8").read() for f in glob.glob(os.path.join(ROOT, "profiles", "*.md"))]
    for name, rec in bench.NCU_TRAFFIC.items():
        mb = f"{rec['bytes_per_launch'] / 1e6:.2f} MB"
        assert any(rec["source_hash"] in t and mb in t for t in texts), name


def test_oracle_one_core_timing_on_cpu():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    b = workloads.make_batch("tiny", "cpu")
    k, dt = bench.time_oracle_one_core(b, budget_s=0.2, max_rows=8)
    assert 1 <= k <= 8 and dt > 0
