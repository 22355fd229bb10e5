"""The two input variants of lp_ragged_compute_ex against the oracle: per-batch
temperature (SGLang page, the sampler's softmax after temperature scaling) and
VARIABLE logits (MAX page, "echo 的前置条件：ReturnLogits 枚举"), on both row kernels,
shrunk and at full size, with their device-detected errors."""

import numpy as np
import pytest
import torch

import ragged_log_probs_gb300 as lp
import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    parity.ensure_built()


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("levels", [0, 1, 3, 5, 6])
def test_temperature_every_levels(kernel, levels, monkeypatch):
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    b = workloads.make_batch("mixed", "cuda", B=10, max_len=14, V=7001, levels=levels, seed=60 + levels)
    parity.check_batch(workloads.with_temperatures(b, seed=levels), what=f"tau/{kernel}/{levels}")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("name,kw", [("decode", dict(B=24)), ("prefill", dict(B=3, max_len=80)),
                                     ("wide", dict(B=2, max_len=10)), ("tiny", dict())])
def test_variable_logits_workloads(kernel, name, kw, monkeypatch):
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    b = workloads.make_batch(name, "cuda", variable_extra=3, **kw)
    parity.check_batch(b, what=f"variable/{name}/{kernel}")
    parity.check_batch(workloads.with_temperatures(b, seed=2), what=f"variable+tau/{name}/{kernel}")


@pytest.mark.parametrize("kernel", ["warp", "queue"])
def test_variable_mixed_echo_and_extra_rows(kernel, monkeypatch):
    # Non-echo batches with 1-4 present rows (only the last is read), echo batches with all.
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    b = workloads.make_batch("mixed", "cuda", B=16, max_len=30, variable_extra=3, seed=71)
    assert b.T < int(b.input_row_offsets[-1])
    parity.check_batch(b)


@pytest.mark.parametrize("name,n", [("decode", 40), ("prefill", 30), ("mixed", 30)])
def test_temperature_full_size_sampled_rows(name, n):
    b = workloads.with_temperatures(workloads.make_batch(name, "cuda"), seed=5)
    off = b.logit_row_offsets.cpu().numpy()
    echo = b.echo.cpu().numpy()
    R = int(sum((off[i + 1] - off[i]) if echo[i] else 1 for i in range(b.B)))
    parity.check_batch(b, rows=parity.sample_rows(R, n, seed=3), full_copy=False)
    del b
    torch.cuda.empty_cache()


def test_variable_full_size_mixed_sampled_rows():
    b = workloads.make_batch("mixed", "cuda", variable_extra=2)
    ioff = b.input_row_offsets.cpu().numpy()
    echo = b.echo.cpu().numpy()
    R = int(sum((ioff[i + 1] - ioff[i]) if echo[i] else 1 for i in range(b.B)))
    parity.check_batch(b, rows=parity.sample_rows(R, 40, seed=4), full_copy=False)
    del b
    torch.cuda.empty_cache()


def test_temperature_extremes_keep_ids():
    g = torch.Generator().manual_seed(8)
    x = (torch.randn(6, 4099, generator=g) * 3).cuda()
    base = workloads.make_custom_batch(x, [2, 4], [1, 1], 3, seed=8)
    plain = parity.run_gpu(base)
    for taus in ([1e-3, 1e4], [0.05, 50.0], [1.0, 1.0]):
        bt = workloads.with_temperatures(base, values=taus)
        parity.check_batch(bt, what=f"tau={taus}")
        got = parity.run_gpu(bt)
        assert np.array_equal(got[2], plain[2])        # ids rank the raw logits
    # tau == 1 everywhere is bit-identical to the plain entry point
    ones = parity.run_gpu(workloads.with_temperatures(base, values=[1.0, 1.0]))
    assert np.array_equal(ones[1], plain[1])


def test_ex_without_variants_is_bitwise_compute():
    b = workloads.make_batch("mixed", "cuda", B=8, max_len=20, seed=9)
    ws = lp.new_workspace(b.B, b.T, b.V, b.levels)
    out_off = lp.plan(b.logit_row_offsets, b.echo, b.T, ws)
    R = int(out_off[-1])
    outs = []
    for use_ex in (False, True):
        o_lp = torch.empty((R, 8), device="cuda")
        o_tok = torch.empty((R, 8), dtype=torch.int32, device="cuda")
        if use_ex:
            lp.compute_ex(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens, out_off, b.echo, 3,
                          o_lp, o_tok, ws)
        else:
            lp.compute(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens, out_off, b.echo, 3,
                       o_lp, o_tok, ws)
        assert lp.read_status(ws) == 0
        outs.append((o_lp.cpu().numpy(), o_tok.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0], equal_nan=True)
    assert np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("bad", [0.0, -1.0, float("nan"), float("inf")])
def test_invalid_temperature_sets_status(bad):
    g = torch.Generator().manual_seed(10)
    x = torch.randn(7, 500, generator=g).cuda()
    b = workloads.make_custom_batch(x, [3, 4], [1, 0], 3, seed=10)
    bt = workloads.with_temperatures(b, values=[0.7, bad])
    ws = lp.new_workspace(b.B, b.T, b.V, b.levels)
    out_off = lp.plan(b.logit_row_offsets, b.echo, b.T, ws)
    o_lp = torch.empty((4, 8), device="cuda")
    o_tok = torch.empty((4, 8), dtype=torch.int32, device="cuda")
    lp.compute_ex(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens, out_off, b.echo, 3, o_lp, o_tok,
                  ws, temperatures=bt.temperatures)
    assert lp.read_status(ws) == (1 << 8)
    g_lp, g_tok = o_lp.cpu().numpy(), o_tok.cpu().numpy().view(np.uint32)
    assert np.all(np.isnan(g_lp[3])) and np.all(g_tok[3] == 0xFFFFFFFF)   # batch 1's only row
    ok = workloads.with_temperatures(b, values=[0.7, 1.0])
    ref = parity.oracle_for(ok)
    parity.compare(g_lp[:3], g_tok[:3].astype(np.uint64), ref[1][:3], ref[2][:3], "valid batch")
    with pytest.raises(lp.LpError):
        lp.ragged_log_probs(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens, b.echo, 3,
                            temperatures=bt.temperatures)


def test_variable_too_few_rows_sets_status():
    # Batch 0 is echo with 3 positions but only 2 present logits rows.
    x = torch.randn(4, 300).cuda()
    loff = torch.tensor([0, 2, 4], dtype=torch.int32, device="cuda")
    ioff = torch.tensor([0, 3, 6], dtype=torch.int32, device="cuda")
    echo = torch.tensor([1, 0], dtype=torch.uint8, device="cuda")
    tokens = torch.arange(6, dtype=torch.int32, device="cuda")
    sampled = torch.tensor([7, 8], dtype=torch.int32, device="cuda")
    ws = lp.new_workspace(2, 6, 300, 2)
    out_off = lp.plan(ioff, echo, 6, ws)
    o_lp = torch.empty((4, 4), device="cuda")
    o_tok = torch.empty((4, 4), dtype=torch.int32, device="cuda")
    lp.compute_ex(x, loff, tokens, sampled, out_off, echo, 2, o_lp, o_tok, ws, input_row_offsets=ioff)
    assert lp.read_status(ws) == (1 << 4)
    g_lp, g_tok = o_lp.cpu().numpy(), o_tok.cpu().numpy().view(np.uint32)
    assert np.all(np.isnan(g_lp[:3])) and np.all(g_tok[:3] == 0xFFFFFFFF)
    # batch 1 (non-echo, last position 5 -> logits row 3, sampled token 8) is still right
    import oracle
    ref_lp, ref_tok, _ = oracle.score_row(x[3].cpu().numpy(), 8, 2)
    parity.compare(g_lp[3:], g_tok[3:].astype(np.uint64), ref_lp[None], ref_tok[None], "valid batch")


def test_variable_host_rejects_mismatched_rows():
    x = torch.randn(3, 50).cuda()
    off = torch.tensor([0, 2, 3], dtype=torch.int32, device="cuda")
    ws = lp.new_workspace(2, 3, 50, 1)
    out_off = lp.plan(off, torch.zeros(2, dtype=torch.uint8, device="cuda"), 3, ws)
    o = torch.empty((2, 2), device="cuda")
    ot = torch.empty((2, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):   # 5 tokens but 3 logits rows and no input offsets
        lp.compute_ex(x, off, torch.zeros(5, dtype=torch.int32, device="cuda"),
                      torch.zeros(2, dtype=torch.int32, device="cuda"), out_off,
                      torch.zeros(2, dtype=torch.uint8, device="cuda"), 1, o, ot, ws)
