"""Host-side test helpers checked on CPU: the parity tolerance and the pooled oracle
that the full-size GPU tests compare every row against."""

import numpy as np

import oracle
import workloads
from tests import oracle_pool, parity


def test_tolerance_is_the_pages_bound_below_2048():
    # 1e-4 absolute wherever fp32 can hold it: half its spacing is 6.1e-5 just below 2048
    ref = np.array([0.0, -1.0, -1023.9, -2047.99])
    assert np.all(parity.tolerance(ref) == 1e-4)


def test_tolerance_above_2048_is_half_a_spacing_plus_the_pre_rounding_error():
    # fp32 spacing is 2^-12 on [2048, 4096) and 2^-11 on [4096, 8192)
    ref = np.array([-2048.0, -3000.0, -5000.0])
    want = np.array([2.0 ** -13, 2.0 ** -13, 2.0 ** -12]) + 1e-5
    np.testing.assert_allclose(parity.tolerance(ref), want, rtol=0, atol=1e-12)
    # a correctly rounded fp32 result always passes
    for v in (-2048.3, -3000.7, -6000.2, -4095.99987):
        assert abs(float(np.float32(v)) - v) <= parity.tolerance(np.array([v]))[0]


def test_pooled_oracle_equals_the_plain_oracle():
    b = workloads.make_batch("mixed", "cpu", B=6, max_len=9, V=3001)
    off, tokens, sampled, echo = b.host()
    mapping = oracle.output_rows(off, echo, tokens, sampled)
    x = b.logits.numpy()
    pool = oracle_pool.new_pool(2)
    try:
        lp, tok = oracle_pool.score_all_rows(pool, lambda rows: x[rows], mapping, b.V, b.levels, chunk_rows=7,
                                             group=3)
    finally:
        pool.terminate()
        pool.join()
    _, rlp, rtok, _ = oracle.ragged_log_probs(x, off, tokens, sampled, echo, b.levels)
    assert np.array_equal(tok, rtok)
    assert np.array_equal(lp, rlp, equal_nan=True)
