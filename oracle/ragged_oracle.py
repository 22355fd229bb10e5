"""Plain fp64 CPU oracle for ragged batched log-probabilities.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or
run this module.  It shares no code with the CUDA path (``ragged_log_probs_gb300``)
and imports nothing from it.

What it computes (the plain definition, written out, slow on purpose):

* Output layout — "MAX Python SDK 中 log_probabilities 模块解析", section
  "ragged 数据编排：从输入缓冲到 kernel 调用": batch ``b`` owns logits rows
  ``[off[b], off[b+1])``; it emits ``len_b`` output rows when echo is on and one
  row otherwise; the output offsets are ``[0]`` followed by the running sum of
  those counts.
* Columns — same page, sections "两个核心函数的 API 契约" and "top-k 语义：堆式
  kernel 与「采样 token 兜底」": ``out_per_token = 2**levels`` (1 when
  ``levels == 0``); the first ``2**levels - 1`` columns hold the top candidates,
  the last column holds the actual (for the last position: sampled) token.
* Value — "logprob、finish reason 与 output processing", section "logprob 的数值
  形态": a logprob is the natural log of the softmax probability, ``x_v - lse``.
* Which token a row scores — same SGLang page, section "input logprob 和 output
  logprob 来自哪里": a prompt position scores the next prompt token; the decode
  step scores the sampled token.

Readings taken where the pages are silent:

* Non-echo batches read the LAST logits row of their sequence (for next-token
  logits with ``off = arange(B+1)`` that row is the only one).
* Top-k order: fp32 logit descending, ties by ascending token id; padding columns
  (vocab smaller than k) carry id ``0xFFFFFFFF`` and logprob ``-inf``.
* ``-inf`` logits are valid tokens with probability 0; a row of only ``-inf``
  has ``lse = NaN`` semantics (``-inf - -inf``), so all its logprobs are NaN.
* A target token ``>= V`` gets logprob NaN and is reported as an error.
* Raw logits unless per-batch temperatures are given. With temperature ``tau_b``
  (the sampler's scaling on the SGLang page, "第二步：采样层选出 token_id，同时计算
  logprob": the logprobs reuse the softmax taken after temperature scaling) the
  values are ``x_v / tau_b - logsumexp(x / tau_b)``; the top-k ranking stays on the
  raw fp32 logits, which is the same order because ``tau_b > 0``.
* Vocab-parallel form (the SGLang page runs the forward pass on "TP worker"s; with the
  lm_head split by vocabulary each rank holds a contiguous column range): a shard
  summarises a row as (logsumexp of its columns, its top-k with global ids, the target
  logit if it holds the target); merging the shards' summaries gives exactly the
  unsharded row, because logsumexp and "k best under (logit desc, id asc)" both
  decompose over a partition of the columns.
* VARIABLE logits (MAX page, "echo 的前置条件：ReturnLogits 枚举"): when the input
  positions are given separately, batch ``b``'s logits rows
  ``[loff[b], loff[b+1])`` hold its LAST ``loff[b+1] - loff[b]`` positions, which
  must cover the positions it scores.

Every function here has a pin in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math
from typing import Callable, Sequence, Union

import numpy as np

PAD_ID = 0xFFFFFFFF

RowSource = Union[np.ndarray, Callable[[int], np.ndarray]]


def out_per_token(levels: int) -> int:
    """Columns per output row: ``2**levels``, or 1 when ``levels == 0``.

    "MAX Python SDK 中 log_probabilities 模块解析", section "两个核心函数的 API 契约".
    """
    if levels < 0:
        raise ValueError("levels must be >= 0")
    return 2 ** levels if levels > 0 else 1


def top_k_capacity(levels: int) -> int:
    """Largest top-n a graph built with ``levels`` can return: ``2**levels - 1``.

    Same page, section "图支持的最大 top-n" (``levels=3`` gives 7); the extra
    column of ``out_per_token`` is reserved for the sampled token.
    """
    return out_per_token(levels) - 1


def levels_for_top_n(top_n: int) -> int:
    """Smallest ``levels`` whose capacity ``2**levels - 1`` covers ``top_n``.

    Same page, section "两个核心函数的 API 契约": ``logprobs=5`` needs ``levels=3``.
    """
    if top_n < 0:
        raise ValueError("top_n must be >= 0")
    levels = 0
    while 2 ** levels - 1 < top_n:
        levels += 1
    return levels


def validate_offsets(logit_row_offsets: Sequence[int], T: int) -> None:
    """Offsets must be non-empty per batch and stay inside the ``T`` logits rows.

    Batch ``n`` owns rows ``[off[n], off[n+1])`` (same page, section "两个核心函数
    的 API 契约"); an empty range is rejected because a non-echo batch would then
    read another batch's row.
    """
    off = [int(v) for v in logit_row_offsets]
    if len(off) < 2:
        raise ValueError("need at least one batch")
    for b in range(len(off) - 1):
        if off[b + 1] <= off[b]:
            raise ValueError(f"batch {b} has an empty or decreasing row range")
    if off[-1] > T:
        raise ValueError("offsets run past the logits rows")


def output_row_offsets(logit_row_offsets: Sequence[int], echo: Sequence[bool]) -> np.ndarray:
    """``[0] ++ cumsum(count_b)``, ``count_b = len_b`` if echo else 1.

    Same page, section "ragged 数据编排：从输入缓冲到 kernel 调用".
    """
    off = [int(v) for v in logit_row_offsets]
    B = len(off) - 1
    if len(echo) != B:
        raise ValueError("echo must have one flag per batch")
    out = [0]
    for b in range(B):
        count = (off[b + 1] - off[b]) if bool(echo[b]) else 1
        out.append(out[-1] + count)
    return np.asarray(out, dtype=np.uint64)


def output_rows(logit_row_offsets: Sequence[int], echo: Sequence[bool],
                tokens: Sequence[int], sampled_tokens: Sequence[int],
                input_row_offsets: Sequence[int] | None = None) -> list[tuple[int, int, int]]:
    """For every output row in order: ``(batch, logits_row, target_token)``.

    Echo batches emit one row per input position, non-echo batches one row for
    their last position; the row of position ``i`` scores token ``i + 1`` of the
    same sequence, and the last position scores the batch's sampled token.
    ("input logprob 和 output logprob 来自哪里" on the SGLang page; sampled-token
    slot in "compute_top 的结果组装" on the MAX page.)

    With ``input_row_offsets`` (VARIABLE logits) positions and tokens follow those
    offsets, and position ``p`` of batch ``b`` reads logits row
    ``loff[b+1] - (ioff[b+1] - p)``: the present rows are the batch's last ones.
    A batch whose present rows do not cover its scored positions is an error.
    """
    loff = [int(v) for v in logit_row_offsets]
    ioff = loff if input_row_offsets is None else [int(v) for v in input_row_offsets]
    if len(ioff) != len(loff):
        raise ValueError("input and logits offsets must both have B+1 entries")
    rows = []
    for b in range(len(ioff) - 1):
        start, end = ioff[b], ioff[b + 1]
        count = (end - start) if bool(echo[b]) else 1
        present = loff[b + 1] - loff[b]
        if present < count:
            raise ValueError(f"batch {b} has {present} logits rows but scores {count} positions")
        for j in range(count):
            p = end - count + j
            t = int(tokens[p + 1]) if p + 1 < end else int(sampled_tokens[b])
            rows.append((b, loff[b + 1] - (end - p), t))
    return rows


def row_logsumexp(x32: np.ndarray, temperature: float = 1.0) -> float:
    """``log(sum(exp(x / temperature)))`` of one fp32 row, in fp64 with the max shift."""
    x = np.asarray(x32, dtype=np.float64) / np.float64(temperature)
    m = x.max()
    return float(m + np.log(np.sum(np.exp(x - m))))


def row_top_k_ids(x32: np.ndarray, k: int) -> np.ndarray:
    """The ``k`` best ids of a row under (fp32 logit desc, id asc), padded with PAD_ID.

    A full stable sort of the whole row — no selection tricks.
    """
    x = np.asarray(x32, dtype=np.float32)
    ids = np.arange(x.shape[0], dtype=np.int64)
    order = np.lexsort((ids, -x.astype(np.float64)))  # primary: -x ascending; secondary: id ascending
    top = order[:k].astype(np.uint64)
    if top.shape[0] < k:
        top = np.concatenate([top, np.full(k - top.shape[0], PAD_ID, dtype=np.uint64)])
    return top


def _get_row(logits: RowSource, r: int) -> np.ndarray:
    if callable(logits):
        return np.asarray(logits(r), dtype=np.float32)
    return np.asarray(logits[r], dtype=np.float32)


def score_row(x32: np.ndarray, target: int, levels: int,
              temperature: float = 1.0) -> tuple[np.ndarray, np.ndarray, bool]:
    """One output row: ``W`` logprobs (fp64) and ids; flag says the target was in range.

    Values are log-softmax of ``x / temperature``; ids rank the raw fp32 logits."""
    V = x32.shape[0]
    K = top_k_capacity(levels)
    W = out_per_token(levels)
    x = np.asarray(x32, dtype=np.float64) / np.float64(temperature)
    lse = row_logsumexp(x32, temperature)
    lp = np.empty(W, dtype=np.float64)
    tok = np.empty(W, dtype=np.uint64)
    if K > 0:
        top = row_top_k_ids(x32, K)
        for c in range(K):
            tok[c] = top[c]
            lp[c] = (x[int(top[c])] - lse) if top[c] != PAD_ID else -math.inf
    in_range = 0 <= target < V
    tok[K] = target
    lp[K] = (x[target] - lse) if in_range else math.nan
    return lp, tok, in_range


def shard_partial(x32_shard: np.ndarray, vocab_base: int, target: int, k: int, temperature: float = 1.0):
    """Summary of one row over the columns ``[vocab_base, vocab_base + V_s)`` it holds.

    Returns ``(lse_s, top, xt)``: the fp64 logsumexp of ``x / temperature`` over the
    shard, the shard's ``k`` best ``(fp32 logit, global id)`` pairs under (logit desc,
    id asc) without padding, and the target's fp32 logit or None when the target is
    not in the shard."""
    x = np.asarray(x32_shard, dtype=np.float32)
    lse_s = row_logsumexp(x, temperature)
    ids = row_top_k_ids(x, min(k, x.shape[0]))
    top = [(float(x[int(i)]), vocab_base + int(i)) for i in ids if int(i) != PAD_ID]
    local = target - vocab_base
    xt = float(x[local]) if 0 <= local < x.shape[0] else None
    return lse_s, top, xt


def merge_shard_partials(partials, target: int, vocab_size: int, levels: int, temperature: float = 1.0):
    """One output row from the shards' summaries (same layout as ``score_row``).

    lse = log(sum_s exp(lse_s)) (fp64, max-shifted); the top-k is the k best of the
    union of the shards' lists under (logit desc, global id asc); the target column
    takes the holder's logit."""
    K = top_k_capacity(levels)
    W = out_per_token(levels)
    lses = np.asarray([p[0] for p in partials], dtype=np.float64)
    m = lses.max()
    lse = float(m + np.log(np.sum(np.exp(lses - m))))
    pool = [pair for p in partials for pair in p[1]]
    pool.sort(key=lambda xi: (-xi[0], xi[1]))
    lp = np.empty(W, dtype=np.float64)
    tok = np.empty(W, dtype=np.uint64)
    for c in range(K):
        if c < len(pool):
            tok[c] = pool[c][1]
            lp[c] = np.float64(pool[c][0]) / np.float64(temperature) - lse
        else:
            tok[c] = PAD_ID
            lp[c] = -math.inf
    holders = [p[2] for p in partials if p[2] is not None]
    in_range = 0 <= target < vocab_size and len(holders) == 1
    tok[K] = target
    lp[K] = (np.float64(holders[0]) / np.float64(temperature) - lse) if in_range else math.nan
    return lp, tok, in_range


def ragged_log_probs(logits: RowSource, logit_row_offsets: Sequence[int], tokens: Sequence[int],
                     sampled_tokens: Sequence[int], echo: Sequence[bool], levels: int,
                     rows: Sequence[int] | None = None, T: int | None = None,
                     temperatures: Sequence[float] | None = None,
                     input_row_offsets: Sequence[int] | None = None):
    """Reference result of the whole path.

    ``logits`` is a 2-D fp32 array ``[T, V]`` or a callable ``r -> row``.
    ``temperatures`` (one positive value per batch) scales the logits before the
    softmax; ``input_row_offsets`` switches to VARIABLE logits (see ``output_rows``).
    Returns ``(out_offsets u64[B+1], logprobs f64[R', W], token_ids u64[R', W],
    all_targets_in_range)`` where ``R'`` is every output row, or only ``rows``
    (output-row indices) when given.
    """
    if T is None:
        T = int(logits.shape[0]) if not callable(logits) else int(logit_row_offsets[-1])
    validate_offsets(logit_row_offsets, T)
    pos_off = logit_row_offsets
    if input_row_offsets is not None:
        validate_offsets(input_row_offsets, int(input_row_offsets[-1]))
        pos_off = input_row_offsets
    if levels < 0:
        raise ValueError("levels must be >= 0")
    B = len(pos_off) - 1
    if temperatures is not None:
        if len(temperatures) != B:
            raise ValueError("one temperature per batch")
        for tau in temperatures:
            if not (math.isfinite(float(tau)) and float(tau) > 0.0):
                raise ValueError("temperatures must be finite and > 0")
    out_off = output_row_offsets(pos_off, echo)
    mapping = output_rows(logit_row_offsets, echo, tokens, sampled_tokens, input_row_offsets)
    wanted = range(len(mapping)) if rows is None else [int(o) for o in rows]
    W = out_per_token(levels)
    lp = np.empty((len(wanted), W), dtype=np.float64)
    tok = np.empty((len(wanted), W), dtype=np.uint64)
    ok = True
    for i, o in enumerate(wanted):
        b, r, t = mapping[o]
        tau = 1.0 if temperatures is None else float(temperatures[b])
        lp[i], tok[i], in_range = score_row(_get_row(logits, r), t, levels, tau)
        ok = ok and in_range
    return out_off, lp, tok, ok


def assemble(out_offsets, logprobs, token_ids, batch_top_n, vocab_size):
    """Per-batch result objects from the output rows, as the MAX page's host step does
    ("compute_top 的结果组装"): ``top_n == 0`` gives None; ``top_n`` outside
    ``[0, W-1]`` is an error; each row's candidate columns (all but the last) drop
    padding ids (>= vocab_size), are ordered by logprob descending and cut to
    ``top_n``; the last column's (actual or sampled) token is then written into the
    row's dict, replacing an equal key. Returns ``[None | (token_logprobs, top_dicts)]``.
    """
    W = logprobs.shape[1]
    results = []
    for b, top_n in enumerate(batch_top_n):
        top_n = int(top_n)
        if top_n < 0:
            raise ValueError("top_n must be >= 0")
        if top_n > W - 1:
            raise ValueError("top_n exceeds the candidates kept per row; build with more levels")
        if top_n == 0:
            results.append(None)
            continue
        token_lps, tops = [], []
        for o in range(int(out_offsets[b]), int(out_offsets[b + 1])):
            pairs = [(int(token_ids[o, c]), float(logprobs[o, c])) for c in range(W - 1)
                     if int(token_ids[o, c]) < vocab_size]
            pairs = sorted(pairs, key=lambda p: -p[1])[:top_n]
            d = dict(pairs)
            d[int(token_ids[o, W - 1])] = float(logprobs[o, W - 1])
            tops.append(d)
            token_lps.append(float(logprobs[o, W - 1]))
        results.append((token_lps, tops))
    return results
