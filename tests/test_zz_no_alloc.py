"""The allocation-free entry point, lp_ragged_compute_noalloc, called through the C
ABI, gives the same results as lp_ragged_compute on two calls in a row.

It serves callers that cannot allocate device memory (a serving engine whose HBM
pool is reserved up front and that forbids cudaMalloc on the request path, or a
binding without a device allocator): its scratch is a static device array inside
the library, shared by every call, so the second call checks that the leftovers
of the first (arrival counters, status word, partial tuples) do not leak into it.
Collected last so that a stop-at-first-failure run has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import ragged_log_probs_gb300 as lp
import workloads
from tests import parity

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    parity.ensure_built()
    lib = lp.load()
    fn = lib.lp_ragged_compute_noalloc
    u32, vp = ctypes.c_uint32, ctypes.c_void_p
    fn.argtypes = [vp, u32, u32, vp, u32, vp, vp, vp, vp, u32, vp, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("case", ["split_rows_levels6", "ragged_echo_levels3", "decode_levels3"])
def test_noalloc_matches_workspace_entry_point_twice(case):
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

    stream = torch.cuda.current_stream()
    for call in range(2):
        out_lp = torch.full((R, W), 123.0, dtype=torch.float32, device="cuda")
        out_tok = torch.zeros((R, W), dtype=torch.int32, device="cuda")
        host_status = torch.full((1,), -1, dtype=torch.int32).pin_memory()
        rc = fn(b.logits.data_ptr(), b.T, b.V, b.logit_row_offsets.data_ptr(), b.B, b.tokens.data_ptr(),
                b.sampled_tokens.data_ptr(), out_off.data_ptr(), b.echo.data_ptr(), b.levels, out_lp.data_ptr(),
                out_tok.data_ptr(), host_status.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, f"call {call}: {lp.STATUS_NAMES.get(rc, rc)}"
        stream.synchronize()
        assert int(host_status[0]) == 0, f"call {call}: device status {int(host_status[0])}"
        parity.compare(out_lp.cpu().numpy(), out_tok.cpu().numpy().view(np.uint32).astype(np.uint64),
                       ref_lp.astype(np.float64), ref_tok, f"{case} call {call}")


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
