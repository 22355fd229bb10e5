"""The package's host-side result assembly against the oracle's, on synthetic output
rows (no GPU): same None pattern, same dicts, same token logprobs."""

import numpy as np
import pytest

import oracle
from ragged_log_probs_gb300 import results


def _rows(rng, R, W, V):
    K = W - 1
    tok = np.empty((R, W), dtype=np.uint64)
    lp = np.empty((R, W), dtype=np.float64)
    for r in range(R):
        n_real = int(rng.integers(0, K + 1))
        ids = rng.choice(V, size=n_real, replace=False)
        vals = np.sort(rng.standard_normal(n_real) * 3 - 2)[::-1]
        tok[r, :n_real] = ids
        lp[r, :n_real] = vals
        tok[r, n_real:K] = oracle.PAD_ID
        lp[r, n_real:K] = -np.inf
        tok[r, K] = ids[0] if (n_real and rng.random() < 0.3) else rng.integers(0, V)
        lp[r, K] = lp[r, 0] if (n_real and tok[r, K] == ids[0]) else -rng.random() * 10
    return tok, lp


@pytest.mark.parametrize("levels", [1, 2, 3, 6])
def test_assemble_matches_oracle(levels):
    rng = np.random.default_rng(levels)
    W = 2 ** levels
    lengths = rng.integers(1, 6, size=9)
    off = np.concatenate([[0], np.cumsum(lengths)])
    V = 2 * W + 10
    tok, lp = _rows(rng, int(off[-1]), W, V=V)
    top_n = rng.integers(0, W, size=9)
    want = oracle.assemble(off, lp, tok, top_n, vocab_size=V)
    got = results.assemble(off.astype(np.uint32), lp.astype(np.float32), tok.astype(np.uint32), top_n, V)
    assert len(got) == len(want)
    for g, w in zip(got, want):
        if w is None:
            assert g is None
            continue
        np.testing.assert_allclose(g.token_log_probabilities, w[0], rtol=1e-6)
        assert [set(d) for d in g.top_log_probabilities] == [set(d) for d in w[1]]
        for dg, dw in zip(g.top_log_probabilities, w[1]):
            for k in dw:
                assert dg[k] == pytest.approx(dw[k], rel=1e-6, abs=1e-6) or (np.isinf(dg[k]) and np.isinf(dw[k]))


def test_assemble_rejects_out_of_range_top_n():
    off = np.array([0, 1], dtype=np.uint32)
    lp = np.zeros((1, 8), dtype=np.float32)
    tok = np.zeros((1, 8), dtype=np.uint32)
    with pytest.raises(ValueError):
        results.assemble(off, lp, tok, [8], 10)
    with pytest.raises(ValueError):
        results.assemble(off, lp, tok, [-1], 10)
    assert results.assemble(off, lp, tok, [0], 10) == [None]
