"""fp64 CPU oracle for ragged batched log-probabilities.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py``; never by the ``ragged_log_probs_gb300`` package.
"""

from .ragged_oracle import (  # noqa: F401
    PAD_ID,
    assemble,
    levels_for_top_n,
    merge_shard_partials,
    out_per_token,
    output_row_offsets,
    output_rows,
    ragged_log_probs,
    row_logsumexp,
    row_top_k_ids,
    score_row,
    shard_partial,
    top_k_capacity,
    validate_offsets,
)
