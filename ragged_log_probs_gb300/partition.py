"""Row-parallel split of one ragged batch over P ranks (host logic, no device work).

Output rows are independent: each one reads one logits row and scores one token
("MAX Python SDK 中 log_probabilities 模块解析", section "ragged 数据编排：从输入缓冲
到 kernel 调用"). When a serving step's logits come off several GPUs' workers (the
SGLang page "logprob、finish reason 与 output processing", section "第一步：
ModelRunner.forward() 输出 logits"), the rows of one batch can be divided: rank k
scores the contiguous global output rows [row_start_k, row_end_k). Every output row
moves the same V*4 bytes of logits, so equal row counts are equal bytes.

A rank's share is expressed as an ordinary ragged batch the library takes as is:

* an echo batch cut inside its positions keeps its echo flag; the part before the
  cut scores, at its last position, the first token after the cut, which becomes
  that sub-batch's sampled token (the part after the cut keeps the real one);
* a non-echo batch contributes only its last position (the one row it scores).

``split_rows`` returns, per rank, the global logits rows to gather (in order), the
rebased offsets, tokens, sampled tokens and echo flags, and where its rows land in
the global output.
"""

from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass
class RankSlice:
    """Rank k's share: a ragged batch over ``logit_rows`` (global logits row indices,
    one per local position) whose output rows are global rows [row_start, row_end)."""
    logit_rows: np.ndarray          # int64 [T_k]: gather these rows of the global logits
    logit_row_offsets: np.ndarray   # uint32 [B_k + 1]
    tokens: np.ndarray              # uint32 [T_k]
    sampled_tokens: np.ndarray      # uint32 [B_k]
    echo: np.ndarray                # uint8 [B_k]
    row_start: int
    row_end: int
    batches: np.ndarray             # int64 [B_k]: the global batch of each local batch

    @property
    def rows(self) -> int:
        return self.row_end - self.row_start


def output_rows_per_batch(logit_row_offsets, echo) -> np.ndarray:
    off = np.asarray(logit_row_offsets, dtype=np.int64)
    lengths = off[1:] - off[:-1]
    if np.any(lengths <= 0):
        raise ValueError("every batch needs at least one position")
    return np.where(np.asarray(echo).astype(bool), lengths, 1)


def rank_bounds(R: int, P: int) -> list[int]:
    """Contiguous, balanced global output-row ranges: rank k gets [b[k], b[k+1])."""
    if P < 1:
        raise ValueError("P must be >= 1")
    return [(k * R) // P for k in range(P + 1)]


def split_rows(logit_row_offsets, tokens, sampled_tokens, echo, P: int) -> list[RankSlice]:
    off = np.asarray(logit_row_offsets, dtype=np.int64)
    tok = np.asarray(tokens).astype(np.uint32)
    smp = np.asarray(sampled_tokens).astype(np.uint32)
    ech = np.asarray(echo).astype(bool)
    B = off.shape[0] - 1
    counts = output_rows_per_batch(off, ech)
    out_off = np.concatenate([[0], np.cumsum(counts)])
    R = int(out_off[-1])
    bounds = rank_bounds(R, P)
    slices = []
    for k in range(P):
        lo, hi = bounds[k], bounds[k + 1]
        rows, loff, ltok, lsmp, lech, lbat = [], [0], [], [], [], []
        if hi > lo:
            b = int(np.searchsorted(out_off, lo, side="right") - 1)
            while b < B and out_off[b] < hi:
                s, e = int(off[b]), int(off[b + 1])
                if ech[b]:
                    # output row out_off[b] + j scores position s + j; keep positions [p0, p1)
                    p0 = s + max(lo, int(out_off[b])) - int(out_off[b])
                    p1 = s + min(hi, int(out_off[b + 1])) - int(out_off[b])
                    # the last kept position scores token p1 (inside the sequence) or the sampled one
                    last_target = int(tok[p1]) if p1 < e else int(smp[b])
                else:
                    p0, p1 = e - 1, e
                    last_target = int(smp[b])
                rows.extend(range(p0, p1))
                ltok.extend(tok[p0:p1].tolist())
                loff.append(loff[-1] + (p1 - p0))
                lsmp.append(last_target)
                lech.append(1 if ech[b] else 0)
                lbat.append(b)
                b += 1
        slices.append(RankSlice(logit_rows=np.asarray(rows, dtype=np.int64),
                                logit_row_offsets=np.asarray(loff, dtype=np.uint32),
                                tokens=np.asarray(ltok, dtype=np.uint32),
                                sampled_tokens=np.asarray(lsmp, dtype=np.uint32),
                                echo=np.asarray(lech, dtype=np.uint8), row_start=lo, row_end=hi,
                                batches=np.asarray(lbat, dtype=np.int64)))
    return slices
