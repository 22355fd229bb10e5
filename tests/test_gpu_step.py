"""lp_ragged_step (plan and reduction in one call, the reduction streaming while the plan
runs): its rows equal lp_ragged_plan + lp_ragged_compute(_ex) bit for bit on every row
kernel and input variant, its host copy reports R and the status of both launches, and it
writes no row when the offsets are bad or the output buffers hold fewer than R rows."""

import numpy as np
import pytest
import torch

import ragged_log_probs_gb300 as lp
import workloads
from tests import parity

pytestmark = pytest.mark.gpu

BIT_OFFSETS = 1 << 4
BIT_TOKEN_RANGE = 1 << 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    parity.ensure_built()


def run_step(b, rows=None, ws=None, sentinel=False):
    """lp.step with outputs of `rows` rows (default T); returns R, status and the outputs."""
    T = b.tokens.numel()
    W = lp.out_per_token(b.levels)
    rows = T if rows is None else rows
    ws = lp.new_workspace(b.B, T, b.V, b.levels) if ws is None else ws
    out_off = torch.empty(b.B + 1, dtype=torch.int32, device="cuda")
    out_lp = torch.full((rows, W), 123.25 if sentinel else 0.0, device="cuda")
    out_tok = torch.full((rows, W), 77 if sentinel else 0, dtype=torch.int32, device="cuda")
    host = torch.zeros(2, dtype=torch.int32).pin_memory()
    lp.step(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens, b.echo, b.levels, out_off, out_lp, out_tok,
            ws, input_row_offsets=b.input_row_offsets, temperatures=b.temperatures, host_out=host)
    torch.cuda.synchronize()
    return (int(host[0]), int(host[1]) & 0xFFFFFFFF, out_off.cpu().numpy().view(np.uint32).astype(np.uint64),
            out_lp.cpu().numpy(), out_tok.cpu().numpy().view(np.uint32).astype(np.uint64))


def check_equal(b, what):
    R, status, off, g_lp, g_tok = run_step(b)
    assert status == 0, what
    r_off, r_lp, r_tok = parity.run_gpu(b)
    assert np.array_equal(off, r_off) and R == int(r_off[-1]), what
    assert np.array_equal(g_tok[:R], r_tok), what
    assert np.array_equal(g_lp[:R], r_lp, equal_nan=True), what


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("name,kw", [("decode", dict(B=40)), ("prefill", dict(B=3, max_len=90)),
                                     ("mixed", dict(B=9, max_len=20)), ("wide", dict(B=2, max_len=12)),
                                     ("tiny", dict())])
def test_step_equals_plan_and_compute(kernel, name, kw, monkeypatch):
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    check_equal(workloads.make_batch(name, "cuda", **kw), f"{name}/{kernel}")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
def test_step_variants_and_split_rows(kernel, monkeypatch):
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    b = workloads.make_batch("mixed", "cuda", B=10, max_len=16, V=30011, variable_extra=2, seed=81)
    check_equal(workloads.with_temperatures(b, seed=3), f"tau+variable/{kernel}")
    # few rows: the row-queue kernel splits each row over several CTAs (tickets)
    check_equal(workloads.make_next_token_batch(3, 200003, levels=6, device="cuda", seed=5), f"split/{kernel}")


def test_step_full_size_decode_against_oracle():
    b = workloads.make_batch("decode", "cuda")
    R, status, off, g_lp, g_tok = run_step(b)
    assert status == 0 and R == b.B
    rows = parity.sample_rows(R, 32, seed=9)
    r_off, r_lp, r_tok, _ = parity.oracle_for(b, rows=rows)
    assert np.array_equal(off, r_off)
    parity.compare(g_lp[rows], g_tok[rows], r_lp, r_tok, "decode step")


def test_step_many_batches_offsets_not_staged():
    # B + 1 > 2048: the row kernel reads the plan's offsets after it (no early stream)
    g = torch.Generator().manual_seed(31)
    B = 2100
    x = torch.randn(B, 300, generator=g).cuda()
    b = workloads.make_custom_batch(x, [1] * B, [0] * B, 3, seed=31)
    check_equal(b, "B=2100")


def test_step_bad_offsets_write_no_row():
    x = torch.randn(6, 500).cuda()
    b = workloads.make_custom_batch(x, [3, 3], [1, 0], 3, seed=4)
    b.logit_row_offsets.copy_(torch.tensor([0, 4, 3], dtype=torch.int32))   # decreasing range
    R, status, _, g_lp, g_tok = run_step(b, sentinel=True)
    assert status & BIT_OFFSETS
    assert np.all(g_lp == 123.25) and np.all(g_tok == 77)


def test_step_output_buffer_too_small():
    b = workloads.make_batch("decode", "cuda", B=24)
    R, status, _, g_lp, g_tok = run_step(b, rows=b.B - 1, sentinel=True)
    assert R == b.B and status == BIT_OFFSETS
    assert np.all(g_lp == 123.25) and np.all(g_tok == 77)


def test_step_reports_the_reduction_status():
    g = torch.Generator().manual_seed(13)
    x = torch.randn(4, 600, generator=g).cuda()
    b = workloads.make_custom_batch(x, [4], [1], 3, seed=13, tokens=[1, 2, 600, 3], sampled=[5])
    R, status, _, g_lp, g_tok = run_step(b)
    assert R == 4 and status == BIT_TOKEN_RANGE
    assert np.isnan(g_lp[1, 7]) and g_tok[1, 7] == 600


@pytest.mark.parametrize("kernel", ["warp", "queue"])
def test_step_repeated_then_compute(kernel, monkeypatch):
    # Steps and a plain compute on one workspace: the counters the row kernels use are
    # back to zero after each launch, so every call gives the same rows.
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    b = workloads.make_next_token_batch(40, 150001, levels=3, device="cuda", seed=21)
    ws = lp.new_workspace(b.B, b.T, b.V, b.levels)
    first = run_step(b, ws=ws)
    again = run_step(b, ws=ws)
    r_off, r_lp, r_tok = parity.run_gpu(b, workspace=ws)
    for got in (first, again):
        assert got[1] == 0
        assert np.array_equal(got[4][:40], r_tok) and np.array_equal(got[3][:40], r_lp, equal_nan=True)


@pytest.mark.parametrize("B,V", [(200, 70001), (152, 128256), (40, 250007), (1, 33)])
def test_step_next_token_prefetch(B, V, monkeypatch):
    # One logits row per batch: each CTA that starts on a task of its own prefetches its
    # warps' first blocks of that row into L2 before it reads the offsets (odd V: rows not
    # 16-byte aligned; 40 rows: split pieces; 152 rows: one task per SM). A hint only:
    # the rows equal plan + compute bit for bit.
    monkeypatch.setenv("LP_RAGGED_KERNEL", "queue")
    check_equal(workloads.make_next_token_batch(B, V, levels=3, device="cuda", seed=B), f"next-token {B}x{V}")


@pytest.mark.parametrize("B", [5, 200])
def test_step_next_token_bad_offsets_write_no_row(B, monkeypatch):
    # One logits row per batch, so the row kernel streams row o for output row o before it
    # has seen any offset; with non-monotone offsets that guess is wrong, nothing is written
    # and the status says so (200 rows: more tasks than SMs, the second ones by a fixed map).
    monkeypatch.setenv("LP_RAGGED_KERNEL", "queue")
    g = torch.Generator().manual_seed(17)
    x = torch.randn(B, 70001, generator=g).cuda()
    b = workloads.make_custom_batch(x, [1] * B, [0] * B, 3, seed=17)
    off = list(range(B + 1))
    off[2], off[3] = 3, 2
    b.logit_row_offsets.copy_(torch.tensor(off, dtype=torch.int32))
    R, status, _, g_lp, g_tok = run_step(b, sentinel=True)
    assert status & BIT_OFFSETS
    assert np.all(g_lp == 123.25) and np.all(g_tok == 77)
