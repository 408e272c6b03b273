"""CPU oracle for exact top-k / top-p candidate-set selection (test infrastructure).

This package is test infrastructure only. It may be imported by ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``; the product path (``top_selection_row_gb300``) never
imports it and shares no code with it.
"""

from .qrita_oracle import (  # noqa: F401
    AMBIGUITY_REL,
    RowResult,
    accepts,
    bf16_bits_to_f64,
    select_batch,
    select_row,
)
from .qrita_outputs import SAMPLE_BAND, candidates, sample, topk_ids  # noqa: F401
