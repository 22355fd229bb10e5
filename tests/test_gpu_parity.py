"""CUDA path vs the fp64 oracle on the five workloads (every output row, at full size
and shrunk) and on the FlashInfer sampling-test shape grid."""

import warnings

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import oracle_pool, parity

pytestmark = pytest.mark.gpu


class ParityReport(UserWarning):
    """A full-size comparison's summary, shown in pytest's warnings summary."""


@pytest.fixture(scope="module", autouse=True)
def _built():
    parity.ensure_built()


@pytest.fixture(scope="module")
def pool():
    p = oracle_pool.new_pool()
    yield p
    p.terminate()
    p.join()


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
    # decode with no overrides is the full-size decode workload
    b = workloads.make_batch(name, "cuda", **kw)
    err = parity.check_batch(b)
    if not kw:
        warnings.warn(ParityReport(f"{name} at full size: all rows match the oracle (ids exact), "
                                   f"max |dlogprob| = {err:.3e}"))


@pytest.mark.parametrize("name", ["prefill", "mixed", "wide"])
def test_workload_full_size_every_row(name, pool):
    # The three large workloads at full size (the tiny and decode ones run whole above):
    # every output row against the oracle, run on all host cores.
    b = workloads.make_batch(name, "cuda")
    g_off, g_lp, g_tok = parity.run_gpu(b)
    off, tokens, sampled, echo = b.host()
    ioff, tau = b.host_variant()
    mapping = oracle.output_rows(off, echo, tokens, sampled, input_row_offsets=ioff)
    assert np.array_equal(g_off, oracle.output_row_offsets(off if ioff is None else ioff, echo)), name

    def fetch(rows):
        idx = torch.as_tensor(rows, dtype=torch.long, device=b.logits.device)
        return b.logits.index_select(0, idx).cpu().numpy()

    r_lp, r_tok = oracle_pool.score_all_rows(pool, fetch, mapping, b.V, b.levels, taus=tau)
    err = parity.compare(g_lp, g_tok, r_lp, r_tok, f"{name} full size, every row")
    warnings.warn(ParityReport(f"{name} at full size: all {len(mapping)} rows x {g_lp.shape[1]} columns match "
                               f"the oracle (ids exact), max |dlogprob| = {err:.3e}"))
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
