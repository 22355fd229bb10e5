"""Row-parallel split of one ragged batch (ragged_log_probs_gb300.partition), on CPU:
the oracle over every rank's slice, placed at the slice's global rows, equals the
oracle over the whole batch exactly; two gloo ranks exchange their rows and each
rebuilds the whole batch's rows."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads
from ragged_log_probs_gb300 import partition

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _oracle_slice(x, sl, levels):
    """Oracle rows of one rank's slice (its logits are the gathered global rows)."""
    _, lp, tok, _ = oracle.ragged_log_probs(x[sl.logit_rows], sl.logit_row_offsets, sl.tokens, sl.sampled_tokens,
                                            sl.echo.astype(bool), levels)
    return lp, tok


def _batches():
    yield workloads.make_batch("tiny", "cpu")
    yield workloads.make_batch("mixed", "cpu", B=9, max_len=13, V=701, seed=5)
    yield workloads.make_batch("prefill", "cpu", B=3, max_len=40, V=500, seed=6)
    yield workloads.make_next_token_batch(11, 300, levels=2, device="cpu", seed=7)


@pytest.mark.parametrize("P", [1, 2, 3, 7, 64])
def test_slices_rebuild_the_whole_batch(P):
    for b in _batches():
        off, tokens, sampled, echo = b.host()
        x = b.logits.numpy()
        _, lp_all, tok_all, _ = oracle.ragged_log_probs(x, off, tokens, sampled, echo, b.levels)
        R = lp_all.shape[0]
        slices = partition.split_rows(off, tokens, sampled, echo, P)
        assert [s.row_start for s in slices] == partition.rank_bounds(R, P)[:-1]
        assert slices[-1].row_end == R
        sizes = [s.rows for s in slices]
        assert max(sizes) - min(sizes) <= 1          # balanced: every row is V*4 bytes
        lp = np.full_like(lp_all, np.nan)
        tok = np.zeros_like(tok_all)
        for s in slices:
            if s.rows == 0:
                assert s.logit_row_offsets.tolist() == [0] and s.logit_rows.size == 0
                continue
            assert s.logit_row_offsets[-1] == s.logit_rows.size == s.tokens.size
            slp, stok = _oracle_slice(x, s, b.levels)
            assert slp.shape[0] == s.rows
            lp[s.row_start:s.row_end] = slp
            tok[s.row_start:s.row_end] = stok
        assert np.array_equal(tok, tok_all), b.name
        assert np.array_equal(lp, lp_all, equal_nan=True), b.name


def test_cut_echo_batch_scores_the_next_token():
    # One echo batch of 5 positions split over 2 ranks (3 + 2 rows): rank 0's last
    # position scores token 3, which becomes its sampled token.
    off = [0, 5]
    tokens = [10, 11, 12, 13, 14]
    s0, s1 = partition.split_rows(off, tokens, [99], [1], 2)
    assert (s0.row_start, s0.row_end, s1.row_start, s1.row_end) == (0, 2, 2, 5)
    assert s0.logit_rows.tolist() == [0, 1] and s0.tokens.tolist() == [10, 11]
    assert s0.sampled_tokens.tolist() == [12]
    assert s1.logit_rows.tolist() == [2, 3, 4] and s1.sampled_tokens.tolist() == [99]
    # a non-echo batch keeps only its last position
    s = partition.split_rows([0, 4], [1, 2, 3, 4], [7], [0], 1)[0]
    assert s.logit_rows.tolist() == [3] and s.sampled_tokens.tolist() == [7] and s.rows == 1


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle as orc
    import workloads as wl
    from ragged_log_probs_gb300 import partition as part
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        b = wl.make_batch("mixed", "cpu", B=10, max_len=15, V=900, seed=21)
        off, tokens, sampled, echo = b.host()
        x = b.logits.numpy()
        mine = part.split_rows(off, tokens, sampled, echo, world)[rank]
        _, lp, tok, _ = orc.ragged_log_probs(x[mine.logit_rows], mine.logit_row_offsets, mine.tokens,
                                             mine.sampled_tokens, mine.echo.astype(bool), b.levels)
        # all ranks' rows, padded to the largest share, gathered in rank order
        W = lp.shape[1]
        R = sum(s.rows for s in part.split_rows(off, tokens, sampled, echo, world))
        cap = max(s.rows for s in part.split_rows(off, tokens, sampled, echo, world))
        buf = torch.full((cap, 2 * W), float("nan"), dtype=torch.float64)
        buf[:mine.rows, :W] = torch.from_numpy(lp)
        buf[:mine.rows, W:] = torch.from_numpy(tok.astype(np.float64))
        gathered = [torch.empty_like(buf) for _ in range(world)]
        dist.all_gather(gathered, buf)
        rows = torch.cat([g[:s.rows] for g, s in zip(gathered, part.split_rows(off, tokens, sampled, echo, world))])
        _, lp_all, tok_all, _ = orc.ragged_log_probs(x, off, tokens, sampled, echo, b.levels)
        ok = (rows.shape[0] == R and np.array_equal(rows[:, W:].numpy().astype(np.uint64), tok_all)
              and np.array_equal(rows[:, :W].numpy(), lp_all, equal_nan=True))
        out.put((rank, bool(ok)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_rebuild_the_batch():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(out.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: True, 1: True}
