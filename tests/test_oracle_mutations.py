"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch
each one: a pin set that lets a wrong oracle pass proves nothing."""

import math

import numpy as np
import pytest

import oracle
import oracle.ragged_oracle as ro
from tests import test_oracle_pins as pins

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _lse_without_log(x32):
    x = np.asarray(x32, dtype=np.float64)
    m = x.max()
    return float(m + np.sum(np.exp(x - m)))


def _lse_without_shift_back(x32):
    x = np.asarray(x32, dtype=np.float64)
    m = x.max()
    return float(np.log(np.sum(np.exp(x - m))))


def _top_k_ties_reversed(x32, k):
    x = np.asarray(x32, dtype=np.float32)
    ids = np.arange(x.shape[0])
    order = np.lexsort((-ids, -x.astype(np.float64)))
    top = order[:k].astype(np.uint64)
    if top.shape[0] < k:
        top = np.concatenate([top, np.full(k - top.shape[0], oracle.PAD_ID, dtype=np.uint64)])
    return top


def _rows_target_same_position(off, echo, tokens, sampled):
    rows = []
    for b in range(len(off) - 1):
        s, e = int(off[b]), int(off[b + 1])
        cnt = (e - s) if echo[b] else 1
        for j in range(cnt):
            r = e - cnt + j
            rows.append((b, r, int(tokens[r]) if r + 1 < e else int(sampled[b])))
    return rows


def _rows_first_position(off, echo, tokens, sampled):
    rows = []
    for b in range(len(off) - 1):
        s, e = int(off[b]), int(off[b + 1])
        cnt = (e - s) if echo[b] else 1
        for j in range(cnt):
            r = s + j
            rows.append((b, r, int(tokens[r + 1]) if r + 1 < e else int(sampled[b])))
    return rows


def _offsets_short_count(off, echo):
    out = [0]
    for b in range(len(off) - 1):
        out.append(out[-1] + ((int(off[b + 1]) - int(off[b]) - 1) if echo[b] else 1))
    return np.asarray(out, dtype=np.uint64)


def _score_row_sign_flipped(x32, target, levels):
    lp, tok, ok = _orig_score_row(x32, target, levels)
    return -lp, tok, ok


def _assemble_without_forced_token(out_offsets, logprobs, token_ids, batch_top_n, vocab_size):
    W = logprobs.shape[1]
    res = []
    for b, top_n in enumerate(batch_top_n):
        if int(top_n) == 0:
            res.append(None)
            continue
        tops, lps = [], []
        for o in range(int(out_offsets[b]), int(out_offsets[b + 1])):
            pairs = [(int(token_ids[o, c]), float(logprobs[o, c])) for c in range(W - 1)
                     if int(token_ids[o, c]) < vocab_size]
            tops.append(dict(sorted(pairs, key=lambda p: -p[1])[:int(top_n)]))
            lps.append(float(logprobs[o, W - 1]))
        res.append((lps, tops))
    return res


def _score_row_multiplies_temperature(x32, target, levels, temperature=1.0):
    return _orig_score_row(x32, target, levels, 1.0 / temperature)


def _score_row_lse_unscaled(x32, target, levels, temperature=1.0):
    lp, tok, ok = _orig_score_row(x32, target, levels, temperature)
    shift = ro.row_logsumexp(x32, temperature) - ro.row_logsumexp(x32, 1.0)
    return lp + shift, tok, ok


def _rows_variable_reads_first_present(logit_row_offsets, echo, tokens, sampled, input_row_offsets=None):
    rows = _orig_output_rows(logit_row_offsets, echo, tokens, sampled, input_row_offsets)
    if input_row_offsets is None:
        return rows
    out, j, prev = [], 0, None
    for (b, r, t) in rows:
        j = j + 1 if b == prev else 0
        prev = b
        out.append((b, int(logit_row_offsets[b]) + j, t))
    return out


def _shard_partial_local_ids(x32_shard, vocab_base, target, k, temperature=1.0):
    return _orig_shard_partial(x32_shard, 0, target - vocab_base, k, temperature)


def _merge_ties_by_shard_last(partials, target, vocab_size, levels, temperature=1.0):
    # pools the later shards first and sorts by logit only: ties go to the later shard
    K = ro.top_k_capacity(levels)
    W = ro.out_per_token(levels)
    lses = np.asarray([p[0] for p in partials], dtype=np.float64)
    m = lses.max()
    lse = float(m + np.log(np.sum(np.exp(lses - m))))
    pool = [pair for p in reversed(partials) for pair in p[1]]
    pool.sort(key=lambda xi: -xi[0])
    lp = np.full(W, -math.inf)
    tok = np.full(W, oracle.PAD_ID, dtype=np.uint64)
    for c in range(min(K, len(pool))):
        tok[c] = pool[c][1]
        lp[c] = pool[c][0] / temperature - lse
    holders = [p[2] for p in partials if p[2] is not None]
    ok = 0 <= target < vocab_size and len(holders) == 1
    tok[K] = target
    lp[K] = holders[0] / temperature - lse if ok else math.nan
    return lp, tok, ok


def _out_per_token_no_slot(levels):
    return 2 ** levels - 1 if levels > 0 else 1


_orig_score_row = ro.score_row
_orig_output_rows = ro.output_rows
_orig_shard_partial = ro.shard_partial
_orig_merge = ro.merge_shard_partials

MUTATIONS = {
    "lse_drops_log": ("row_logsumexp", _lse_without_log),
    "lse_drops_max": ("row_logsumexp", _lse_without_shift_back),
    "ties_by_higher_id": ("row_top_k_ids", _top_k_ties_reversed),
    "target_off_by_one": ("output_rows", _rows_target_same_position),
    "non_echo_reads_first_row": ("output_rows", _rows_first_position),
    "echo_count_short": ("output_row_offsets", _offsets_short_count),
    "logprob_sign_flipped": ("score_row", _score_row_sign_flipped),
    "no_sampled_slot": ("out_per_token", _out_per_token_no_slot),
    "assembly_drops_actual_token": ("assemble", _assemble_without_forced_token),
    "temperature_multiplies": ("score_row", _score_row_multiplies_temperature),
    "temperature_lse_unscaled": ("score_row", _score_row_lse_unscaled),
    "variable_reads_first_present_rows": ("output_rows", _rows_variable_reads_first_present),
    "shard_ids_not_offset": ("shard_partial", _shard_partial_local_ids),
    "shard_merge_ties_by_later_shard": ("merge_shard_partials", _merge_ties_by_shard_last),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(ro, attr, fn)
    monkeypatch.setattr(oracle, attr, fn, raising=False)
    failures = 0
    for t in PIN_TESTS:
        try:
            t()
        except (AssertionError, ValueError, IndexError, TypeError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name!r}"
