"""The allocation-free entry point, lp_ragged_compute_noalloc, called through the C
ABI, gives the same results as lp_ragged_compute on calls in a row.

It serves callers that cannot allocate device memory (a serving engine whose HBM
pool is reserved up front and that forbids cudaMalloc on the request path, or a
binding without a device allocator): its scratch is a static device array inside
the library, shared by every call. The first call of each case raises a device
status bit (a sampled token >= V), so the valid calls after it check that the
leftovers of earlier calls (status word, arrival counters, partial tuples) do not
leak into them. Collected last so that a stop-at-first-failure run has already run
every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import ragged_log_probs_gb300 as lp
import workloads
from tests import parity

pytestmark = pytest.mark.gpu

LP_ERR_OFFSETS_BIT = 1 << 4
LP_ERR_TOKEN_RANGE_BIT = 1 << 5


def _noalloc_fn():
    parity.ensure_built()
    lib = lp.load()
    fn = lib.lp_ragged_compute_noalloc
    u32, vp = ctypes.c_uint32, ctypes.c_void_p
    fn.argtypes = [vp, u32, u32, vp, u32, vp, vp, vp, vp, u32, vp, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, b, sampled, out_off, out_lp, out_tok, host_status, stream):
    return fn(b.logits.data_ptr(), b.T, b.V, b.logit_row_offsets.data_ptr(), b.B, b.tokens.data_ptr(),
              sampled.data_ptr(), out_off.data_ptr(), b.echo.data_ptr(), b.levels, out_lp.data_ptr(),
              out_tok.data_ptr(), host_status.data_ptr(), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("case", ["split_rows_levels6", "ragged_echo_levels3", "decode_levels3"])
def test_noalloc_matches_workspace_entry_point(case):
    fn = _noalloc_fn()
    if case == "split_rows_levels6":
        b = workloads.make_next_token_batch(5, 200003, levels=6, dist="normal", scale=3.0, device="cuda", seed=17)
    elif case == "ragged_echo_levels3":
        b = workloads.make_batch("mixed", "cuda", B=12, max_len=24)
    else:
        b = workloads.make_batch("decode", "cuda")
    W = lp.out_per_token(b.levels)

    # existing entry point (caller-provided workspace)
    out_off, ref_lp, ref_tok = lp.ragged_log_probs(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens,
                                                   b.echo, b.levels)
    R = ref_lp.shape[0]
    ref_lp = ref_lp.cpu().numpy()
    ref_tok = ref_tok.cpu().numpy().view(np.uint32).astype(np.uint64)

    # call 1: one sampled token out of range, a device-detected error (no fault): the
    # status bit must come back; calls 2 and 3 are valid and must not see it
    bad_sampled = b.sampled_tokens.clone()
    bad_sampled[b.B - 1] = b.V
    stream = torch.cuda.current_stream()
    for call in range(3):
        out_lp = torch.full((R, W), 123.0, dtype=torch.float32, device="cuda")
        out_tok = torch.zeros((R, W), dtype=torch.int32, device="cuda")
        host_status = torch.full((1,), -1, dtype=torch.int32).pin_memory()
        sampled = bad_sampled if call == 0 else b.sampled_tokens
        rc = _call(fn, b, sampled, out_off, out_lp, out_tok, host_status, stream)
        assert rc == 0, f"call {call}: {lp.STATUS_NAMES.get(rc, rc)}"
        stream.synchronize()
        status = int(host_status[0]) & 0xFFFFFFFF
        if call == 0:
            assert status == LP_ERR_TOKEN_RANGE_BIT, f"call 0: device status {status:#x}"
            continue
        assert status == 0, f"call {call}: device status {status:#x}"
        parity.compare(out_lp.cpu().numpy(), out_tok.cpu().numpy().view(np.uint32).astype(np.uint64),
                       ref_lp.astype(np.float64), ref_tok, f"{case} call {call}")


def test_noalloc_reports_offsets_the_plan_rejects():
    # Decreasing input offsets: lp_ragged_plan flags them and gives the bad batch no
    # row; the allocation-free call checks the offsets itself, writes no row and
    # returns the LP_ERR_OFFSETS bit in its own status word.
    fn = _noalloc_fn()
    g = torch.Generator().manual_seed(3)
    x = torch.randn(6, 500, generator=g).cuda()
    off = torch.tensor([0, 4, 2, 6], dtype=torch.int32, device="cuda")
    echo = torch.tensor([1, 0, 1], dtype=torch.uint8, device="cuda")
    tokens = torch.zeros(6, dtype=torch.int32, device="cuda")
    sampled = torch.zeros(3, dtype=torch.int32, device="cuda")
    ws = lp.new_workspace(3, 6, 500, 3)
    host = torch.zeros(2, dtype=torch.int32).pin_memory()
    out_off = lp.plan(off, echo, 6, ws, host_out=host)
    torch.cuda.synchronize()
    assert int(host[1]) == LP_ERR_OFFSETS_BIT
    rows = max(int(host[0]), 1)
    out_lp = torch.full((rows, 8), 123.0, dtype=torch.float32, device="cuda")
    out_tok = torch.full((rows, 8), 7, dtype=torch.int32, device="cuda")
    host_status = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    b = workloads.Batch(name="decreasing offsets", logits=x, logit_row_offsets=off, tokens=tokens,
                        sampled_tokens=sampled, echo=echo, levels=3, B=3, T=6, V=500)
    stream = torch.cuda.current_stream()
    assert _call(fn, b, sampled, out_off, out_lp, out_tok, host_status, stream) == 0
    stream.synchronize()
    assert (int(host_status[0]) & 0xFFFFFFFF) == LP_ERR_OFFSETS_BIT
    assert torch.all(out_lp == 123.0) and torch.all(out_tok == 7)


def test_noalloc_host_checks():
    fn = _noalloc_fn()
    fake = 0x10000
    args = [fake, 4, 100, fake, 2, fake, fake, fake, fake, 3, fake, fake, None, None]
    bad = list(args)
    bad[0] = None
    assert fn(*bad) == 1            # LP_ERR_NULL
    bad = list(args)
    bad[9] = 7
    assert fn(*bad) == 2            # LP_ERR_LEVELS
    bad = list(args)
    bad[2] = 0
    assert fn(*bad) == 3            # LP_ERR_SHAPE, rejected before anything is enqueued
