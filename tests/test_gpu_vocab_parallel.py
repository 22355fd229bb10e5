"""Vocab-parallel form on one GPU: the ranks' column shards are run one after another
into the slices of one gathered tuple buffer (what the all-gather produces), then
merged; the rows must equal the oracle on the unsplit logits and, id for id, the
unsharded CUDA path."""

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


def _bounds(V, P, rng):
    if P == 1:
        return [0, V]
    cuts = sorted(rng.choice(np.arange(1, V), size=P - 1, replace=False).tolist())
    return [0] + cuts + [V]


def run_sharded(b, bounds, rows_capacity=None):
    """Plan, one lp_ragged_shard_partials per shard into its slice, then the merge."""
    P = len(bounds) - 1
    T = b.tokens.numel()
    ws = lp.new_workspace(b.B, T, b.V, b.levels)
    host = torch.zeros(2, dtype=torch.int32).pin_memory()
    out_off = lp.plan(b.positions_offsets, b.echo, T, ws, host_out=host)
    torch.cuda.synchronize()
    R = int(host[0])
    assert int(host[1]) == 0
    cap = R if rows_capacity is None else rows_capacity
    stride = lp.tuple_bytes(b.levels)
    gathered = torch.zeros((P, cap * stride), dtype=torch.uint8, device="cuda")
    for p in range(P):
        shard = b.logits[:, bounds[p]:bounds[p + 1]].contiguous()
        lp.shard_partials(shard, bounds[p], b.logit_row_offsets, b.tokens, b.sampled_tokens, out_off, b.echo,
                          b.levels, gathered[p], cap, ws, input_row_offsets=b.input_row_offsets,
                          temperatures=b.temperatures)
    W = lp.out_per_token(b.levels)
    out_lp = torch.empty((R, W), device="cuda")
    out_tok = torch.empty((R, W), dtype=torch.int32, device="cuda")
    lp.shard_merge(gathered, P, cap, b.V, out_off, b.levels, out_lp, out_tok, ws, temperatures=b.temperatures)
    status = lp.read_status(ws)
    return (status, out_off.cpu().numpy().view(np.uint32).astype(np.uint64), out_lp.cpu().numpy(),
            out_tok.cpu().numpy().view(np.uint32).astype(np.uint64))


def check_sharded(b, bounds, what):
    status, g_off, g_lp, g_tok = run_sharded(b, bounds)
    assert status == 0, what
    r_off, r_lp, r_tok, _ = parity.oracle_for(b)
    assert np.array_equal(g_off, r_off), what
    parity.compare(g_lp, g_tok, r_lp, r_tok, what)
    _, _, u_tok = parity.run_gpu(b)
    assert np.array_equal(g_tok, u_tok), f"{what}: ids differ from the unsharded path"


@pytest.mark.parametrize("kernel", ["warp", "queue"])
@pytest.mark.parametrize("name,kw,P", [
    ("decode", dict(B=24), 8),
    ("decode", dict(B=5), 1),
    ("mixed", dict(B=8, max_len=20, V=40003), 3),
    ("prefill", dict(B=2, max_len=70), 4),
    ("wide", dict(B=2, max_len=10), 5),
    ("tiny", dict(), 2),
])
def test_sharded_equals_oracle(kernel, name, kw, P, monkeypatch):
    monkeypatch.setenv("LP_RAGGED_KERNEL", kernel)
    b = workloads.make_batch(name, "cuda", **kw)
    rng = np.random.default_rng(P * 13 + b.V)
    check_sharded(b, _bounds(b.V, P, rng), f"{name}/P={P}/{kernel}")


@pytest.mark.parametrize("levels", [0, 1, 4, 6])
def test_sharded_every_levels_narrow_shards(levels):
    # Shards narrower than K, one-column shards, odd bases (rows start unaligned).
    b = workloads.make_batch("mixed", "cuda", B=6, max_len=10, V=301, levels=levels, seed=80 + levels)
    bounds = [0, 1, 2, 9, 40, 41, 170, 301]
    check_sharded(b, bounds, f"narrow/levels={levels}")


def test_sharded_ties_across_shard_boundaries():
    # Quantised logits: equal values on both sides of every boundary.
    g = torch.Generator().manual_seed(12)
    x = (torch.round(torch.randn(12, 5000, generator=g) * 2) / 2).cuda()
    b = workloads.make_custom_batch(x, [5, 7], [1, 1], 6, seed=12)
    check_sharded(b, [0, 1250, 2500, 3750, 5000], "ties")


def test_sharded_with_temperature_and_variable_logits():
    b = workloads.with_temperatures(workloads.make_batch("mixed", "cuda", B=10, max_len=16, V=30011,
                                                         variable_extra=2, seed=81), seed=3)
    check_sharded(b, [0, 7000, 7001, 30011], "tau+variable")


def test_sharded_full_size_decode_sampled():
    b = workloads.make_batch("decode", "cuda")
    bounds = [round(i * b.V / 8) for i in range(9)]
    status, g_off, g_lp, g_tok = run_sharded(b, bounds)
    assert status == 0
    rows = parity.sample_rows(b.B, 32, seed=5)
    r_off, r_lp, r_tok, _ = parity.oracle_for(b, rows=rows)
    parity.compare(g_lp[rows], g_tok[rows], r_lp, r_tok, "decode P=8")


def test_merge_flags_token_out_of_range():
    g = torch.Generator().manual_seed(13)
    x = torch.randn(4, 600, generator=g).cuda()
    b = workloads.make_custom_batch(x, [4], [1], 3, seed=13, tokens=[1, 2, 600, 3], sampled=[5])
    status, _, g_lp, g_tok = run_sharded(b, [0, 300, 600])
    assert status == (1 << 5)
    assert np.isnan(g_lp[1, 7]) and g_tok[1, 7] == 600
    assert not np.isnan(g_lp[0, 7])


def test_partials_refuse_small_tuple_buffer():
    b = workloads.make_batch("tiny", "cuda")
    T = b.tokens.numel()
    ws = lp.new_workspace(b.B, T, b.V, b.levels)
    out_off = lp.plan(b.logit_row_offsets, b.echo, T, ws)
    stride = lp.tuple_bytes(b.levels)
    buf = torch.full((5 * stride,), 0xAB, dtype=torch.uint8, device="cuda")   # R = 6 rows needed
    lp.shard_partials(b.logits, 0, b.logit_row_offsets, b.tokens, b.sampled_tokens, out_off, b.echo, b.levels,
                      buf, 5, ws)
    assert lp.read_status(ws) == (1 << 4)
    assert torch.all(buf == 0xAB)                 # nothing written
