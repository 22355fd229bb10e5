"""CUDA path vs the fp64 oracle on the five workloads (shrunk: every output row;
full size: sampled rows) and on the FlashInfer sampling-test shape grid."""

import numpy as np
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    parity.ensure_built()


def test_tiny_full():
    b = workloads.make_batch("tiny", "cuda")
    parity.check_batch(b)


@pytest.mark.parametrize("name,kw", [
    ("prefill", dict(B=6, max_len=70)),
    ("mixed", dict(B=12, max_len=24)),
    ("wide", dict(B=3, max_len=40)),
    ("decode", dict()),
])
def test_workload_shrunk_every_row(name, kw):
    b = workloads.make_batch(name, "cuda", **kw)
    parity.check_batch(b)


@pytest.mark.parametrize("name,n", [("prefill", 40), ("mixed", 40), ("wide", 24)])
def test_workload_full_size_sampled_rows(name, n):
    b = workloads.make_batch(name, "cuda")
    off, _, _, echo = b.host()
    R = int(sum((off[i + 1] - off[i]) if echo[i] else 1 for i in range(b.B)))
    rows = parity.sample_rows(R, n, seed=11)
    parity.check_batch(b, rows=rows, full_copy=False)
    del b
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dist", ["normal", "gumbel"])
@pytest.mark.parametrize("B", [1, 99, 989])
@pytest.mark.parametrize("V", [111, 32000, 128256])
def test_flashinfer_shape_grid(dist, B, V):
    b = workloads.make_next_token_batch(B, V, levels=3, dist=dist, scale=2.0, device="cuda", seed=B * 7 + V)
    rows = None if B * V <= 99 * 32000 else parity.sample_rows(B, 24, seed=B)
    parity.check_batch(b, rows=rows)


@pytest.mark.parametrize("levels", [0, 1, 2, 3, 4, 5, 6])
def test_every_levels(levels):
    b = workloads.make_batch("mixed", "cuda", B=10, max_len=12, V=5003, levels=levels, seed=40 + levels)
    parity.check_batch(b)


def test_host_assembly_from_gpu_rows():
    # The user-facing result (MAX page, "compute_top 的结果组装") from the GPU rows vs the
    # oracle's rows: per-batch None pattern, dict keys exact, values within tolerance.
    import oracle
    import ragged_log_probs_gb300 as lp
    b = workloads.make_batch("mixed", "cuda", B=10, max_len=16)
    out_off, out_lp, out_tok = lp.ragged_log_probs(b.logits, b.logit_row_offsets, b.tokens, b.sampled_tokens,
                                                   b.echo, b.levels)
    top_n = np.random.default_rng(3).integers(0, 8, size=b.B)
    got = lp.assemble(out_off, out_lp, out_tok, top_n, b.V)
    r_off, r_lp, r_tok, _ = parity.oracle_for(b)
    want = oracle.assemble(r_off, r_lp, r_tok, top_n, b.V)
    for g, w in zip(got, want):
        if w is None:
            assert g is None
            continue
        assert [set(d) for d in g.top_log_probabilities] == [set(d) for d in w[1]]
        for dg, dw in zip(g.top_log_probabilities, w[1]):
            for k in dw:
                assert abs(dg[k] - dw[k]) <= 1e-4 or dg[k] == dw[k]
        np.testing.assert_allclose(g.token_log_probabilities, w[0], atol=1e-4)
