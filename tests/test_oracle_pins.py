"""Pins that tie the fp64 oracle to what the pages and the mathematics fix.

None of these re-type the oracle's formulas: they use values printed on the pages,
closed forms (dyadic distributions, uniform rows), an independent library routine
(scipy's log_softmax), and brute force by pairwise counting on tiny rows.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import PAD_ID

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --- worked constants (MAX page: API contract, max top-n) -------------------------

def test_levels_worked_values():
    g = _golden("page_constants.json")
    for top_n, levels in g["levels_examples"]["top_n_to_levels"]:
        assert oracle.levels_for_top_n(top_n) == levels
    for levels, w in g["levels_examples"]["levels_to_out_per_token"]:
        assert oracle.out_per_token(levels) == w
    assert oracle.top_k_capacity(g["max_top_n"]["levels"]) == g["max_top_n"]["max_top_n"]


def test_levels_relation_all():
    for levels in range(0, 7):
        k = oracle.top_k_capacity(levels)
        assert oracle.out_per_token(levels) == k + 1
        assert oracle.levels_for_top_n(k) == levels
        if levels:
            assert oracle.levels_for_top_n(k + 1) == levels + 1
    assert oracle.top_k_capacity(6) == 63
    with pytest.raises(ValueError):
        oracle.levels_for_top_n(-1)


# --- layout (MAX page: ragged data layout) ----------------------------------------

def test_tiny_layout_golden():
    g = _golden("tiny_layout.json")
    off = np.concatenate([[0], np.cumsum(g["lengths"])])
    got = oracle.output_row_offsets(off, g["echo"])
    assert got.tolist() == g["output_row_offsets"]
    assert np.diff(got).tolist() == g["output_counts"]
    rows = oracle.output_rows(off, g["echo"], tokens=np.zeros(off[-1], int), sampled_tokens=[0] * 4)
    assert [r for (_, r, _) in rows] == g["logit_rows_scored"]


def test_next_token_layout_is_arange():
    B = 9
    off = np.arange(B + 1)
    got = oracle.output_row_offsets(off, [False] * B)
    assert got.tolist() == list(range(B + 1))
    rows = oracle.output_rows(off, [False] * B, tokens=np.arange(B), sampled_tokens=np.arange(100, 100 + B))
    assert [(b, r, t) for (b, r, t) in rows] == [(b, b, 100 + b) for b in range(B)]


def test_target_is_next_input_token_then_sampled():
    # SGLang page, "input logprob 和 output logprob 来自哪里": a prompt position
    # scores the following prompt token; the final position scores the sampled one.
    off = [0, 3, 5]
    tokens = [10, 11, 12, 20, 21]
    rows = oracle.output_rows(off, [True, False], tokens, [99, 98])
    assert rows == [(0, 0, 11), (0, 1, 12), (0, 2, 99), (1, 4, 98)]
    rows = oracle.output_rows(off, [False, True], tokens, [99, 98])
    assert rows == [(0, 2, 99), (1, 3, 21), (1, 4, 98)]


def test_invalid_offsets_rejected():
    with pytest.raises(ValueError):
        oracle.validate_offsets([0, 2, 2, 5], 5)      # empty batch
    with pytest.raises(ValueError):
        oracle.validate_offsets([0, 3, 2], 5)         # decreasing
    with pytest.raises(ValueError):
        oracle.validate_offsets([0, 3, 7], 5)         # past T
    oracle.validate_offsets([0, 3, 5], 5)


# --- values (SGLang page: logprob numeric form) -----------------------------------

def test_dyadic_row_closed_form_and_tie_order():
    p = np.array([0.5, 0.25, 0.125, 0.125])
    x = np.log(p).astype(np.float32)
    lp, tok, ok = oracle.score_row(x, target=3, levels=2)
    assert ok
    assert tok.tolist() == [0, 1, 2, 3]        # ids 2 and 3 tie: lower id first
    np.testing.assert_allclose(lp, np.log(p[[0, 1, 2, 3]]), atol=1e-7)
    # fp32 logits of exact powers of two: ln(2^-k) rounded to fp32 differs from the
    # fp64 value by < 1e-7; the dyadic sum itself is exact.


def test_page_probability_examples():
    g = _golden("page_constants.json")["probability_examples"]
    for lp_print, pct in g["logprob_to_percent"]:
        assert round(100 * math.exp(lp_print)) == pct
    # A three-token distribution with those probabilities, shifted by an arbitrary
    # constant (softmax is shift-invariant): natural-log logprobs come back.
    probs = np.array([0.154, 0.122, 0.724])
    x = (np.log(probs) + 7.5).astype(np.float32)
    lp, tok, _ = oracle.score_row(x, target=0, levels=2)
    assert tok[:3].tolist() == [2, 0, 1]
    assert round(lp[1], 2) == -1.87 and round(lp[2], 2) == -2.10
    assert round(lp[3], 2) == -1.87


def test_uniform_row_is_minus_log_v():
    V = 1000
    x = np.full(V, 3.25, dtype=np.float32)
    lp, tok, _ = oracle.score_row(x, target=17, levels=3)
    assert tok[:7].tolist() == list(range(7))
    np.testing.assert_allclose(lp, -math.log(V), atol=1e-12, rtol=0)


def test_full_vocab_columns_sum_to_one():
    rng = np.random.default_rng(5)
    for V in (1, 2, 5, 7):
        x = (rng.standard_normal(V) * 4).astype(np.float32)
        lp, tok, _ = oracle.score_row(x, target=0, levels=3)
        real = lp[:V]
        assert abs(scipy.special.logsumexp(real)) < 1e-12
        assert sorted(tok[:V].tolist()) == list(range(V))
        assert all(t == PAD_ID for t in tok[V:7])
        assert all(v == -math.inf for v in lp[V:7])


def test_matches_scipy_log_softmax():
    rng = np.random.default_rng(6)
    for V in (3, 40, 63):
        x = (rng.standard_normal(V) * 3).astype(np.float32)
        ref = scipy.special.log_softmax(x.astype(np.float64))
        for target in (0, V - 1):
            lp, tok, _ = oracle.score_row(x, target=target, levels=6)
            for c in range(min(V, 63)):
                assert abs(lp[c] - ref[int(tok[c])]) < 1e-12
            assert abs(lp[63] - ref[target]) < 1e-12


def test_brute_force_rank_and_pairwise_values():
    """Tiny rows with many exact ties, every levels: ids by pairwise rank counting,
    values by lp_i = -log(sum_j exp(x_j - x_i)) summed with math.fsum."""
    rng = np.random.default_rng(7)
    for trial in range(40):
        V = int(rng.integers(1, 65))
        x = (np.round(rng.standard_normal(V) * 4) / 4).astype(np.float32)
        if trial % 5 == 0:
            x[rng.integers(0, V, size=max(1, V // 4))] = -np.inf
        if np.all(np.isneginf(x)):
            x[0] = 0.0
        better = lambda j, i: (x[j] > x[i]) or (x[j] == x[i] and j < i)
        rank = [sum(better(j, i) for j in range(V)) for i in range(V)]
        by_rank = [None] * V
        for i, r in enumerate(rank):
            by_rank[r] = i
        xs = [float(v) for v in x]
        def brute_lp(i):
            if xs[i] == -math.inf:
                return -math.inf
            return -math.log(math.fsum(math.exp(xj - xs[i]) for xj in xs if xj != -math.inf))
        for levels in range(0, 7):
            K = oracle.top_k_capacity(levels)
            t = int(rng.integers(0, V))
            lp, tok, ok = oracle.score_row(x, target=t, levels=levels)
            assert ok and tok[K] == t
            assert abs(lp[K] - brute_lp(t)) < 1e-9 or (lp[K] == brute_lp(t) == -math.inf)
            for c in range(K):
                if c < V:
                    assert tok[c] == by_rank[c]
                    want = brute_lp(by_rank[c])
                    assert (lp[c] == want == -math.inf) or abs(lp[c] - want) < 1e-9
                else:
                    assert tok[c] == PAD_ID and lp[c] == -math.inf


def test_lexsort_cross_check_large_row():
    rng = np.random.default_rng(8)
    V = 5000
    x = (np.round(rng.standard_normal(V) * 16) / 16).astype(np.float32)
    top = oracle.row_top_k_ids(x, 63)
    # independent: python's sort on (-x, id) tuples
    want = sorted(range(V), key=lambda i: (-float(x[i]), i))[:63]
    assert top.tolist() == want


# --- special values and invariants -------------------------------------------------

def test_neg_inf_entries_rank_last():
    x = np.array([-np.inf, 1.0, -np.inf, 0.5, -np.inf], dtype=np.float32)
    lp, tok, _ = oracle.score_row(x, target=2, levels=3)
    assert tok[:5].tolist() == [1, 3, 0, 2, 4]
    assert lp[2] == -np.inf and lp[3] == -np.inf and lp[4] == -np.inf
    assert lp[7] == -np.inf and tok[7] == 2
    assert abs(np.logaddexp(lp[0], lp[1])) < 1e-12


def test_all_neg_inf_row_is_nan_by_reading():
    x = np.full(10, -np.inf, dtype=np.float32)
    lp, tok, _ = oracle.score_row(x, target=4, levels=2)
    assert tok.tolist() == [0, 1, 2, 4]
    assert np.all(np.isnan(lp))


def test_target_out_of_range_flags_nan():
    x = np.zeros(8, dtype=np.float32)
    lp, tok, ok = oracle.score_row(x, target=8, levels=1)
    assert not ok and tok[1] == 8 and math.isnan(lp[1])


def test_invariants_on_tiny_workload():
    import workloads
    b = workloads.make_batch("tiny", "cpu")
    off, tok_in, sampled, echo = b.host()
    out_off, lp, tok, ok = oracle.ragged_log_probs(b.logits.numpy(), off, tok_in, sampled, echo, b.levels)
    assert ok
    assert out_off.tolist() == _golden("tiny_layout.json")["output_row_offsets"]
    assert lp.shape == (6, 8)
    assert np.all(lp <= 0)
    x = b.logits.numpy()
    rows = oracle.output_rows(off, echo, tok_in, sampled)
    for o, (_, r, t) in enumerate(rows):
        # top-k is sorted: non-increasing logit, ascending id within a tie
        keys = [(-float(x[r, i]), int(i)) for i in tok[o, :7]]
        assert keys == sorted(keys)
        # the actual-token column equals the top-k entry when the id coincides
        for c in range(7):
            if tok[o, c] == t:
                assert lp[o, c] == lp[o, 7]
    # row 0 of the tiny workload holds two exactly tied maxima, lower id first
    r0 = x[0]
    ties = np.flatnonzero(r0 == r0.max())
    assert len(ties) == 2
    assert tok[0, :2].tolist() == sorted(ties.tolist())


def test_assemble_hand_example():
    # MAX page, "compute_top 的结果组装": padding ids dropped, candidates ordered by logprob
    # and cut to top_n, the last column's token forced in (replacing an equal key),
    # top_n == 0 -> None, top_n outside [0, W-1] -> error. Worked by hand for W = 4.
    PAD = oracle.PAD_ID
    off = np.array([0, 2, 3])
    tok = np.array([[5, 2, PAD, 7], [3, 4, 5, 3], [1, 2, 3, 9]], dtype=np.uint64)
    lp = np.array([[-0.1, -1.0, -np.inf, -3.0], [-0.5, -0.7, -2.0, -0.5], [-0.2, -0.3, -4.0, -6.0]])
    res = oracle.assemble(off, lp, tok, batch_top_n=[2, 0], vocab_size=10)
    assert res[1] is None
    token_lps, tops = res[0]
    assert token_lps == [-3.0, -0.5]
    assert tops[0] == {5: -0.1, 2: -1.0, 7: -3.0}
    assert tops[1] == {3: -0.5, 4: -0.7}
    res = oracle.assemble(off, lp, tok, batch_top_n=[1, 3], vocab_size=10)
    assert res[0][1][1] == {3: -0.5}
    assert res[1][1][0] == {1: -0.2, 2: -0.3, 3: -4.0, 9: -6.0}
    with pytest.raises(ValueError):
        oracle.assemble(off, lp, tok, batch_top_n=[4, 1], vocab_size=10)
    with pytest.raises(ValueError):
        oracle.assemble(off, lp, tok, batch_top_n=[-1, 1], vocab_size=10)


# --- temperature (SGLang page: the sampler's softmax after temperature scaling) ---------

def _one_row(x, target, levels, tau):
    off, lp, tok, ok = oracle.ragged_log_probs(np.asarray(x, dtype=np.float32)[None, :], [0, 1], [0], [target],
                                               [False], levels, temperatures=[tau])
    return lp[0], tok[0], ok


def test_temperature_two_token_closed_form():
    # Two logits a > b at temperature tau: p(a) = 1 / (1 + e^{(b - a)/tau}), the logistic
    # function, so log p(a) = -log1p(e^{(b-a)/tau}) and log p(b) = -log1p(e^{(a-b)/tau}).
    a, b = 1.75, -0.5
    for tau in (0.25, 0.5, 1.0, 2.0, 3.0, 10.0):
        lp, tok, ok = _one_row([b, a], target=0, levels=1, tau=tau)
        assert ok and tok.tolist() == [1, 0]
        assert abs(lp[0] - (-math.log1p(math.exp((b - a) / tau)))) < 1e-14
        assert abs(lp[1] - (-math.log1p(math.exp((a - b) / tau)))) < 1e-14


def test_temperature_matches_scipy_of_scaled_row():
    rng = np.random.default_rng(21)
    for V, tau in ((50, 0.6), (63, 1.7), (200, 0.05)):
        x = (rng.standard_normal(V) * 3).astype(np.float32)
        ref = scipy.special.log_softmax(x.astype(np.float64) / tau)
        lp, tok, _ = _one_row(x, target=V - 1, levels=6, tau=tau)
        for c in range(63):
            if tok[c] != PAD_ID:
                assert abs(lp[c] - ref[int(tok[c])]) < 1e-11
        assert abs(lp[63] - ref[V - 1]) < 1e-11


def test_temperature_limits():
    rng = np.random.default_rng(22)
    V = 100
    x = (rng.standard_normal(V) * 2).astype(np.float32)
    # tau -> infinity: the distribution flattens to uniform, every logprob -> -log V
    lp, _, _ = _one_row(x, target=3, levels=3, tau=1e7)
    np.testing.assert_allclose(lp, -math.log(V), atol=1e-5, rtol=0)
    # tau -> 0: all mass on the largest logit (gap to the runner-up >= 0.05 here)
    x[7] = x.max() + 0.25
    lp, tok, _ = _one_row(x, target=3, levels=3, tau=1e-3)
    assert tok[0] == 7 and lp[0] > -1e-15 and lp[1] < -40


def test_temperature_keeps_ids_and_one_is_plain():
    import workloads
    b = workloads.make_batch("tiny", "cpu")
    off, tok_in, sampled, echo = b.host()
    x = b.logits.numpy()
    plain = oracle.ragged_log_probs(x, off, tok_in, sampled, echo, b.levels)
    ones = oracle.ragged_log_probs(x, off, tok_in, sampled, echo, b.levels, temperatures=[1.0] * b.B)
    assert np.array_equal(plain[1], ones[1]) and np.array_equal(plain[2], ones[2])
    for taus in ([0.3, 2.0, 7.0, 0.9], [5.0] * 4):
        hot = oracle.ragged_log_probs(x, off, tok_in, sampled, echo, b.levels, temperatures=taus)
        assert np.array_equal(hot[2], plain[2])          # ids rank the raw logits
        for o in range(hot[1].shape[0]):
            # each row stays a log-distribution: top-k + rest sums to at most 1
            assert scipy.special.logsumexp(hot[1][o, :7]) <= 1e-12


def test_temperature_rejects_non_positive():
    x = np.zeros((1, 4), dtype=np.float32)
    for tau in (0.0, -1.0, math.nan, math.inf):
        with pytest.raises(ValueError):
            oracle.ragged_log_probs(x, [0, 1], [0], [0], [False], 1, temperatures=[tau])


# --- VARIABLE logits (MAX page: "echo 的前置条件：ReturnLogits 枚举") ---------------------

def test_variable_hand_mapping():
    # Tiny layout, lengths {3,5,1,7}, echo {T,F,T,F}; logits present for the last
    # {3,2,1,1} positions of each sequence, so loff = [0,3,5,6,7]. Worked by hand:
    # batch 0 scores positions 0,1,2 from logits rows 0,1,2 (targets tokens[1], tokens[2],
    # sampled[0]); batch 1 scores its last position 7 from row 4 (its last present row);
    # batch 2 position 8 from row 5; batch 3 position 15 from row 6.
    ioff = [0, 3, 8, 9, 16]
    loff = [0, 3, 5, 6, 7]
    tokens = list(range(100, 116))
    sampled = [900, 901, 902, 903]
    rows = oracle.output_rows(loff, [True, False, True, False], tokens, sampled, input_row_offsets=ioff)
    assert rows == [(0, 0, 101), (0, 1, 102), (0, 2, 900), (1, 4, 901), (2, 5, 902), (3, 6, 903)]
    assert oracle.output_row_offsets(ioff, [True, False, True, False]).tolist() == [0, 3, 4, 5, 6]


def test_variable_equals_all_mode_on_gathered_rows():
    import workloads
    b = workloads.make_batch("tiny", "cpu")
    off, tok_in, sampled, echo = b.host()
    x = b.logits.numpy()
    full = oracle.ragged_log_probs(x, off, tok_in, sampled, echo, b.levels)
    # same offsets for both: VARIABLE with every position present is ALL mode
    same = oracle.ragged_log_probs(x, off, tok_in, sampled, echo, b.levels, input_row_offsets=off)
    assert np.array_equal(full[1], same[1]) and np.array_equal(full[2], same[2])
    # keep only the rows the output needs (hand-listed for lengths {3,5,1,7}, echo {T,F,T,F})
    keep = [0, 1, 2, 7, 8, 15]
    compact = oracle.ragged_log_probs(x[keep], [0, 3, 4, 5, 6], tok_in, sampled, echo, b.levels,
                                      input_row_offsets=off)
    assert np.array_equal(full[0], compact[0])
    assert np.array_equal(full[1], compact[1]) and np.array_equal(full[2], compact[2])


def test_variable_too_few_rows_rejected():
    x = np.zeros((4, 8), dtype=np.float32)
    with pytest.raises(ValueError):   # echo batch of 3 positions with 2 logits rows
        oracle.ragged_log_probs(x, [0, 2, 4], list(range(5)), [0, 0], [True, False], 1,
                                input_row_offsets=[0, 3, 5])


# --- vocab-parallel form (lm_head split by vocabulary across tensor-parallel ranks) -------

def _split(V, cuts):
    edges = [0] + sorted(cuts) + [V]
    return [(a, b) for a, b in zip(edges[:-1], edges[1:]) if b > a]


def test_shard_merge_hand_example():
    # Row [1, 3, 2 | 3, 0, 2] split after column 3, K = 3, target id 4. Worked by hand:
    # the two 3's tie across the boundary (id 1 before id 3), then the two 2's (id 2
    # before id 5): top = ids 1, 3, 2; the target's logit 0 lives in shard 1.
    x = np.array([1, 3, 2, 3, 0, 2], dtype=np.float32)
    parts = [oracle.shard_partial(x[0:3], 0, 4, 3), oracle.shard_partial(x[3:6], 3, 4, 3)]
    assert parts[0][1] == [(3.0, 1), (2.0, 2), (1.0, 0)] and parts[0][2] is None
    assert parts[1][1] == [(3.0, 3), (2.0, 5), (0.0, 4)] and parts[1][2] == 0.0
    lp, tok, ok = oracle.merge_shard_partials(parts, 4, 6, 2)
    assert ok and tok.tolist() == [1, 3, 2, 4]
    z = math.log(math.fsum(math.exp(v) for v in (1, 3, 2, 3, 0, 2)))
    np.testing.assert_allclose(lp, [3 - z, 3 - z, 2 - z, 0 - z], atol=1e-14, rtol=0)


def test_shard_merge_equals_unsharded_row():
    rng = np.random.default_rng(31)
    for trial in range(60):
        V = int(rng.integers(1, 300))
        x = (np.round(rng.standard_normal(V) * 3) / 2).astype(np.float32)   # many ties
        if trial % 7 == 0:
            x[rng.integers(0, V, size=max(1, V // 5))] = -np.inf
        if np.all(np.isneginf(x)):
            x[0] = 1.0
        n_cuts = int(rng.integers(0, min(8, V)))
        shards = _split(V, rng.choice(np.arange(1, V), size=n_cuts, replace=False).tolist() if n_cuts else [])
        levels = int(rng.integers(0, 7))
        K = oracle.top_k_capacity(levels)
        t = int(rng.integers(0, V))
        tau = [1.0, 0.6, 1.9][trial % 3]
        parts = [oracle.shard_partial(x[a:b], a, t, K, tau) for a, b in shards]
        lp, tok, ok = oracle.merge_shard_partials(parts, t, V, levels, tau)
        ref_lp, ref_tok, ref_ok = oracle.score_row(x, t, levels, tau)
        assert ok == ref_ok
        assert tok.tolist() == ref_tok.tolist(), (trial, shards)
        fin = np.isfinite(ref_lp)
        assert np.array_equal(np.isneginf(lp), np.isneginf(ref_lp))
        np.testing.assert_allclose(lp[fin], ref_lp[fin], atol=1e-11, rtol=0)


def test_shard_target_outside_every_shard_is_nan():
    x = np.zeros(8, dtype=np.float32)
    parts = [oracle.shard_partial(x[0:4], 0, 8, 1), oracle.shard_partial(x[4:8], 4, 8, 1)]
    lp, tok, ok = oracle.merge_shard_partials(parts, 8, 8, 1)
    assert not ok and tok[1] == 8 and math.isnan(lp[1])
