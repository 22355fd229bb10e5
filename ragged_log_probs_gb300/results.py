"""Host-side result assembly (the user-facing form of the output rows).

Follows the host step of "MAX Python SDK 中 log_probabilities 模块解析", section
"compute_top 的结果组装", and the result type of section "数据结构：可序列化的
LogProbabilities": per batch item, the actual/sampled token's logprob for every
output row, and per row a dict of the ``top_n`` best tokens (padding ids dropped)
with the actual/sampled token always present. ``top_n == 0`` gives None.

Host code by design (as on the page): the rows are already sorted on the device by
(logit descending, id ascending), so the assembly only cuts and formats them.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np


@dataclasses.dataclass
class LogProbabilities:
    token_log_probabilities: List[float]
    top_log_probabilities: List[dict]


def _host(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a)


def assemble(output_row_offsets, out_logprobs, out_tokens, batch_top_n: Sequence[int],
             vocab_size: int) -> List[Optional[LogProbabilities]]:
    """Build one ``LogProbabilities`` (or None) per batch item from the device outputs.

    ``top_n`` must lie in ``[0, W-1]`` (W = 2**levels): a larger request needs a larger
    ``levels``, exactly as on the page."""
    off = _host(output_row_offsets).astype(np.int64) & 0xFFFFFFFF
    lp = _host(out_logprobs).astype(np.float64)
    tok = _host(out_tokens).view(np.uint32).astype(np.int64) if _host(out_tokens).dtype != np.uint32 \
        else _host(out_tokens).astype(np.int64)
    W = lp.shape[1]
    if len(batch_top_n) != len(off) - 1:
        raise ValueError("one top_n per batch item")
    out: List[Optional[LogProbabilities]] = []
    for b, top_n in enumerate(batch_top_n):
        top_n = int(top_n)
        if top_n < 0:
            raise ValueError(f"top_n must be >= 0, got {top_n}")
        if top_n > W - 1:
            raise ValueError(f"top_n {top_n} exceeds the {W - 1} candidates per row; use more levels")
        if top_n == 0:
            out.append(None)
            continue
        rows = slice(int(off[b]), int(off[b + 1]))
        lp_b, tok_b = lp[rows], tok[rows]
        tops = []
        for r in range(lp_b.shape[0]):
            keep = [c for c in range(W - 1) if tok_b[r, c] < vocab_size][:top_n]  # already sorted
            d = {int(tok_b[r, c]): float(lp_b[r, c]) for c in keep}
            d[int(tok_b[r, W - 1])] = float(lp_b[r, W - 1])
            tops.append(d)
        out.append(LogProbabilities(token_log_probabilities=[float(v) for v in lp_b[:, W - 1]],
                                    top_log_probabilities=tops))
    return out
