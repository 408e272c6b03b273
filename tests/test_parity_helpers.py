"""The pooled row-by-row comparison the full-size GPU tests use, checked on
the CPU: masks the oracle itself produced pass, and a planted error in one
row (a dropped token, a swapped tie, a top-p prefix cut short) is caught in
exactly that row."""

import numpy as np

from oracle import select_batch
from parity_helpers import compare_rows_pooled
from workloads import generate


def _oracle_masks(logits, dtype, k, p):
    ref = select_batch(logits, dtype, k, p)
    return np.stack([res.mask for _, res in ref]), ref


def test_pooled_comparison_passes_the_definition_and_catches_planted_errors():
    logits, k, p = generate(4, rows=6)  # bf16, ties, top-k then top-p
    masks, ref = _oracle_masks(logits, "bf16", k, p)
    st = np.zeros(6, np.int32)
    fails, flagged, bad = compare_rows_pooled(logits, "bf16", k, p, masks, st, workers=3)
    assert fails == [] and bad == []
    assert flagged == sum(1 for _, r in ref if r.ambiguous)

    planted = masks.copy()
    # row 1: drop the last kept token in id order
    kept1 = np.nonzero(planted[1])[0]
    planted[1, kept1[-1]] = 0
    # row 4: keep a dropped token whose value equals the boundary instead of a kept one (ties by id)
    x4 = (logits[4].astype(np.uint32) << 16).view(np.float32)
    kept4 = np.nonzero(planted[4])[0]
    b = x4[kept4].min()
    tie_dropped = np.nonzero((x4 == b) & (planted[4] == 0))[0]
    tie_kept = np.nonzero((x4 == b) & (planted[4] == 1))[0]
    assert tie_dropped.size and tie_kept.size
    planted[4, tie_kept[0]] = 0
    planted[4, tie_dropped[-1]] = 1
    fails, _, bad = compare_rows_pooled(logits, "bf16", k, p, planted, st, workers=2)
    assert sorted({f[0] for f in fails}) == [1, 4]
    assert {b[0] for b in bad} <= {1, 4} and 4 in {b[0] for b in bad}


def test_pooled_mass_invariant_catches_a_short_top_p_prefix():
    logits, k, p = generate(3, rows=3)  # fp32, top-p only
    masks, ref = _oracle_masks(logits, "f32", k, p)
    st = np.zeros(3, np.int32)
    x = logits[2].astype(np.float64)
    order = np.argsort(-x, kind="stable")
    n = int(masks[2].sum())
    cut = masks.copy()
    cut[2, order[n // 2: n]] = 0  # keep only the first half of the prefix
    fails, _, bad = compare_rows_pooled(logits, "f32", k, p, cut, st, workers=2)
    assert [f[0] for f in fails] == [2]
    assert [b[0] for b in bad] == [2] and "below p" in bad[0][1][0]
