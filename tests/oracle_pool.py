"""The fp64 oracle over every output row of a large batch, on all host cores.

Test infrastructure: a spawn pool of worker processes each scoring groups of rows
with ``oracle.score_row``. The parent streams the needed logits rows device -> host
in chunks into one memory-mapped file (in /dev/shm when it has room), so workers
receive only row indices (no pickled rows). This module imports numpy and the
oracle only (no torch), so the spawned workers start quickly.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

import oracle

_MAPS = {}


def _attach(path: str, n: int, V: int):
    m = _MAPS.get(path)
    if m is None:
        _MAPS.clear()
        m = np.memmap(path, dtype=np.float32, mode="r", shape=(n, V))
        _MAPS[path] = m
    return m


def _score_group(args):
    """Worker: score rows ``idx`` of the shared chunk ``[n, V]`` (fp32)."""
    path, n, V, idx, targets, taus, levels = args
    rows = _attach(path, n, V)
    W = oracle.out_per_token(levels)
    lp = np.empty((len(idx), W), dtype=np.float64)
    tok = np.empty((len(idx), W), dtype=np.uint64)
    for j, (i, t, tau) in enumerate(zip(idx, targets, taus)):
        lp[j], tok[j], _ = oracle.score_row(rows[i], int(t), levels, float(tau))
    return lp, tok


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:  # pragma: no cover
        return os.cpu_count() or 1


def new_pool(processes: int | None = None):
    return mp.get_context("spawn").Pool(processes or host_cores())


def _scratch_dir(nbytes: int):
    """/dev/shm when it has room for the chunk twice over, else the default temp dir."""
    try:
        st = os.statvfs("/dev/shm")
        if st.f_bavail * st.f_frsize >= 2 * nbytes:
            return "/dev/shm"
    except OSError:
        pass
    return None


def score_all_rows(pool, fetch_rows, mapping, V: int, levels: int, taus=None, chunk_rows: int = 512,
                   group: int = 8):
    """Oracle rows for every entry of ``mapping`` (``(batch, logits_row, target)`` per
    output row, as ``oracle.output_rows`` gives). ``fetch_rows(rows) -> float32 [n, V]``
    copies the listed logits rows to the host. Returns (logprobs f64 [R, W], ids u64 [R, W])."""
    R = len(mapping)
    W = oracle.out_per_token(levels)
    lp = np.empty((R, W), dtype=np.float64)
    tok = np.empty((R, W), dtype=np.uint64)
    fd, path = tempfile.mkstemp(prefix="oracle_rows", suffix=".f32", dir=_scratch_dir(chunk_rows * V * 4))
    os.close(fd)
    try:
        buf = np.memmap(path, dtype=np.float32, mode="w+", shape=(chunk_rows, V))
        for o0 in range(0, R, chunk_rows):
            part = mapping[o0:o0 + chunk_rows]
            n = len(part)
            buf[:n] = fetch_rows([r for _, r, _ in part])
            buf.flush()
            tasks = []
            for g0 in range(0, n, group):
                sel = list(range(g0, min(n, g0 + group)))
                tasks.append((path, chunk_rows, V, sel, [part[i][2] for i in sel],
                              [1.0 if taus is None else float(taus[part[i][0]]) for i in sel], levels))
            for g0, (glp, gtok) in zip(range(0, n, group), pool.map(_score_group, tasks, chunksize=1)):
                lp[o0 + g0:o0 + g0 + len(glp)] = glp
                tok[o0 + g0:o0 + g0 + len(gtok)] = gtok
        del buf
    finally:
        os.unlink(path)
    return lp, tok
