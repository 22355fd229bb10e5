"""The multi-GPU forms on one GPU: a row-range split of one batch run rank after rank,
and the composed vocab-parallel call through a one-rank NCCL group, both against the
oracle."""

import os
import socket

import numpy as np
import pytest
import torch

import ragged_log_probs_gb300 as lp
import workloads
from ragged_log_probs_gb300 import partition
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    parity.ensure_built()


def _dev_u32(a):
    return torch.from_numpy(np.asarray(a, dtype=np.uint32).view(np.int32).copy()).cuda()


@pytest.mark.parametrize("name,kw,P", [("mixed", dict(B=16, max_len=40), 3), ("prefill", dict(B=4, max_len=300), 2),
                                       ("decode", dict(), 5), ("wide", dict(B=3, max_len=30), 4),
                                       ("tiny", dict(), 8)])
def test_row_split_ranks_in_turn(name, kw, P):
    b = workloads.make_batch(name, "cuda", **kw)
    off, tokens, sampled, echo = b.host()
    slices = partition.split_rows(off, tokens, sampled, echo, P)
    R, W = slices[-1].row_end, lp.out_per_token(b.levels)
    g_lp = np.full((R, W), np.nan)
    g_tok = np.zeros((R, W), dtype=np.uint64)
    for s in slices:
        if s.rows == 0:
            continue
        x = b.logits.index_select(0, torch.as_tensor(s.logit_rows, device="cuda")).contiguous()
        echo_d = torch.from_numpy(s.echo).cuda()
        o_off, o_lp, o_tok = lp.ragged_log_probs(x, _dev_u32(s.logit_row_offsets), _dev_u32(s.tokens),
                                                 _dev_u32(s.sampled_tokens), echo_d, b.levels)
        assert o_lp.shape[0] == s.rows
        g_lp[s.row_start:s.row_end] = o_lp.cpu().numpy()
        g_tok[s.row_start:s.row_end] = o_tok.cpu().numpy().view(np.uint32)
    r_off, r_lp, r_tok, _ = parity.oracle_for(b)
    assert R == r_lp.shape[0]
    parity.compare(g_lp, g_tok, r_lp, r_tok, f"{name} split over {P} ranks")


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


@pytest.fixture(scope="module")
def nccl_one_rank():
    import torch.distributed as dist
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    yield dist
    dist.destroy_process_group()


@pytest.mark.parametrize("variant", ["plain", "variable_tau", "decode_levels6"])
def test_vocab_parallel_composed_call_one_rank(variant, nccl_one_rank):
    # ragged_log_probs_vocab_parallel end to end (plan, shard partials, the NCCL
    # all-gather of the tuples, merge, status check) with the one rank holding every column.
    if variant == "plain":
        b = workloads.make_batch("mixed", "cuda", B=8, max_len=12, V=20011, seed=31)
    elif variant == "variable_tau":
        b = workloads.with_temperatures(workloads.make_batch("mixed", "cuda", B=8, max_len=12, V=20011,
                                                             variable_extra=2, seed=32), seed=3)
    else:
        b = workloads.make_batch("decode", "cuda", B=24, levels=6, seed=33)
    out_off, out_lp, out_tok = lp.ragged_log_probs_vocab_parallel(
        b.logits, 0, b.V, b.logit_row_offsets, b.tokens, b.sampled_tokens, b.echo, b.levels,
        input_row_offsets=b.input_row_offsets, temperatures=b.temperatures)
    assert out_lp.dtype == torch.float32 and out_tok.dtype == torch.int32
    r_off, r_lp, r_tok, _ = parity.oracle_for(b)
    assert np.array_equal(out_off.cpu().numpy().view(np.uint32).astype(np.uint64), r_off)
    parity.compare(out_lp.cpu().numpy(), out_tok.cpu().numpy().view(np.uint32).astype(np.uint64), r_lp, r_tok,
                   f"vocab-parallel one rank ({variant})")
