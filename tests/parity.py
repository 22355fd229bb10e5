"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle on the
same inputs, compare element by element.

Tolerance: token ids and row layout bit-exact; logprobs |delta| <= 1e-4 absolute
(NaN where the oracle has NaN, -inf where it has -inf) wherever |logprob| < 2048.
From 2048 up no fp32 output can hold 1e-4: rounding the exact value to fp32 alone
moves it by up to half a spacing, 1.22e-4 at 2048. There the bound is that half
spacing plus 1e-5, the error the kernel may carry before its final rounding (its
logprob is formed in fp64 from the row's fp32 sum-exp; the sum's relative rounding
error over a row, typically a few 1e-7, is what remains, and no part of the error
grows with |logprob|)."""

from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL = 1e-4
FP32_EXACT_LIMIT = 2048.0   # |logprob| from which half an fp32 spacing exceeds ATOL
PRE_ROUNDING_ERR = 1e-5     # the kernel's error before it rounds a logprob to fp32


def tolerance(ref):
    """Per-element bound on |gpu - ref| for finite fp64 reference logprobs."""
    ref = np.asarray(ref, dtype=np.float64)
    half_spacing = 0.5 * np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return np.where(np.abs(ref) < FP32_EXACT_LIMIT, ATOL, half_spacing + PRE_ROUNDING_ERR)


def ensure_built():
    from ragged_log_probs_gb300 import _build
    _build.build()


def run_gpu(batch, workspace=None):
    import ragged_log_probs_gb300 as lp
    out_off, out_lp, out_tok = lp.ragged_log_probs(batch.logits, batch.logit_row_offsets, batch.tokens,
                                                   batch.sampled_tokens, batch.echo, batch.levels,
                                                   workspace=workspace, input_row_offsets=batch.input_row_offsets,
                                                   temperatures=batch.temperatures)
    torch.cuda.synchronize()
    return (out_off.cpu().numpy().view(np.uint32).astype(np.uint64), out_lp.cpu().numpy(),
            out_tok.cpu().numpy().view(np.uint32).astype(np.uint64))


def row_getter(logits: torch.Tensor):
    """Fetch single logits rows device -> host for the oracle (no full copy)."""
    cache = {}

    def get(r):
        if r not in cache:
            cache[r] = logits[r].cpu().numpy()
        return cache[r]
    return get


def oracle_for(batch, rows=None, full_copy=None):
    off, tokens, sampled, echo = batch.host()
    ioff, tau = batch.host_variant()
    if full_copy is None:
        full_copy = batch.logits.numel() * 4 <= (1 << 31)
    src = batch.logits.cpu().numpy() if full_copy else row_getter(batch.logits)
    return oracle.ragged_log_probs(src, off, tokens, sampled, echo, batch.levels, rows=rows, T=batch.T,
                                   temperatures=None if tau is None else [float(t) for t in tau],
                                   input_row_offsets=ioff)


def compare(gpu_lp, gpu_tok, ref_lp, ref_tok, what=""):
    assert gpu_tok.shape == ref_tok.shape, (what, gpu_tok.shape, ref_tok.shape)
    bad = np.argwhere(gpu_tok != ref_tok)
    assert bad.size == 0, f"{what}: {len(bad)} token-id mismatches, first at {bad[:5].tolist()}: " \
        f"gpu {gpu_tok[tuple(bad[0])]} ref {ref_tok[tuple(bad[0])]}"
    ref32 = ref_lp
    nan_ref = np.isnan(ref32)
    assert np.array_equal(np.isnan(gpu_lp), nan_ref), f"{what}: NaN pattern differs"
    inf_ref = np.isinf(ref32)
    assert np.array_equal(np.isinf(gpu_lp) & ~nan_ref, inf_ref), f"{what}: inf pattern differs"
    assert np.all(gpu_lp[inf_ref] == ref32[inf_ref]), f"{what}: inf signs differ"
    fin = ~(nan_ref | inf_ref)
    err = np.abs(gpu_lp[fin].astype(np.float64) - ref32[fin])
    tol = tolerance(ref32[fin])
    if err.size:
        i = int(np.argmax(err - tol))
        assert err[i] <= tol[i], f"{what}: |delta| {err[i]:.3g} > {tol[i]:.3g} at reference {ref32[fin][i]:.6g}"
    return float(err.max()) if err.size else 0.0


def check_batch(batch, rows=None, full_copy=None, what=None):
    """Run GPU + oracle; full comparison, or only the given output rows."""
    what = what or batch.name
    g_off, g_lp, g_tok = run_gpu(batch)
    r_off, r_lp, r_tok, _ = oracle_for(batch, rows=rows, full_copy=full_copy)
    assert np.array_equal(g_off, r_off), f"{what}: output_row_offsets differ"
    if rows is not None:
        g_lp, g_tok = g_lp[rows], g_tok[rows]
    return compare(g_lp, g_tok, r_lp, r_tok, what)


def sample_rows(R, n, seed=0):
    rng = np.random.default_rng(seed)
    picks = set([0, R - 1, R // 2]) | set(rng.integers(0, R, size=n).tolist())
    return sorted(p for p in picks if 0 <= p < R)
