"""The exchange step of the vocab-parallel form on CPU, with two real gloo ranks: each
rank summarises its vocab columns with the oracle, packs the summaries in the
documented row-tuple layout, and ``gather_shard_tuples`` must hand every rank all
shards in rank order; unpacking and merging them must give the unsharded rows."""

import math
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LOG2E = 1.4426950408889634
PAD = 0xFFFFFFFF
HOLDS = 0x80000000


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _stride(K):
    return ((4 + 2 * K) * 4 + 15) // 16 * 16


def _pack(x_shard, base, target, K):
    """Row tuple (u32 words) of one shard's row, written from the layout description."""
    import oracle
    x = np.asarray(x_shard, dtype=np.float32)
    words = np.zeros(_stride(K) // 4, dtype=np.uint32)
    f = words.view(np.float32)
    m = float(x.max())
    c = np.float32(m * LOG2E) if m != -math.inf else np.float32(-np.inf)
    s = np.float32(sum(2.0 ** (float(v) * LOG2E - float(c)) for v in x if v != -math.inf)) if m != -math.inf \
        else np.float32(0)
    f[0], f[1] = c, s
    local = target - base
    holds = 0 <= local < x.shape[0]
    f[2] = x[local] if holds else np.float32(0)
    words[3] = (target & 0x7FFFFFFF) | (HOLDS if holds else 0)
    ids = oracle.row_top_k_ids(x, K)
    for i in range(K):
        f[4 + i] = x[int(ids[i])] if ids[i] != PAD else np.float32(-np.inf)
        words[4 + K + i] = base + int(ids[i]) if ids[i] != PAD else PAD
    return words


def _unpack(words, K):
    f = words.view(np.float32)
    lse = float(f[0]) * math.log(2) + math.log(float(f[1]))
    top = [(float(f[4 + i]), int(words[4 + K + i])) for i in range(K) if int(words[4 + K + i]) != PAD]
    xt = float(f[2]) if int(words[3]) & HOLDS else None
    return lse, top, xt, int(words[3]) & 0x7FFFFFFF


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import ragged_log_probs_gb300 as lp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(0)                    # same rows on every rank
        V, R, levels = 97, 5, 3
        K = 2 ** levels - 1
        x = (np.round(rng.standard_normal((R, V)) * 2) / 2).astype(np.float32)
        targets = rng.integers(0, V, size=R)
        bounds = [0, 41, V]                               # rank r holds [bounds[r], bounds[r+1])
        a, b = bounds[rank], bounds[rank + 1]
        local = np.concatenate([_pack(x[o, a:b], a, int(targets[o]), K) for o in range(R)])
        gathered = lp.gather_shard_tuples(torch.from_numpy(local.view(np.uint8).copy()))
        out.put((rank, gathered.numpy().copy(), x, targets, bounds))
    finally:
        dist.destroy_process_group()


def test_gather_and_merge_two_gloo_ranks():
    import oracle
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
    levels, K = 3, 7
    stride_words = _stride(K) // 4
    for rank, gathered, x, targets, bounds in results:
        assert gathered.shape[0] == 2                      # one buffer per rank, rank order
        words = gathered.view(np.uint32).reshape(2, -1, stride_words)
        R, V = x.shape
        for o in range(R):
            parts = []
            for p in range(2):
                lse, top, xt, t = _unpack(words[p, o], K)
                assert t == targets[o]
                assert all(bounds[p] <= i < bounds[p + 1] for _, i in top)   # shard p's ids sit at slot p
                parts.append((lse, top, xt))
            lp_m, tok_m, ok = oracle.merge_shard_partials(parts, int(targets[o]), V, levels)
            ref_lp, ref_tok, _ = oracle.score_row(x[o], int(targets[o]), levels)
            assert ok and tok_m.tolist() == ref_tok.tolist()
            np.testing.assert_allclose(lp_m, ref_lp, atol=1e-5, rtol=0)
