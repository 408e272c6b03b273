"""Pins of the output oracle (oracle/qrita_outputs.py) to things fixed apart
from its code: brute-force stable orders on tiny rows, exact rational
probabilities (logits ln 1, ln 2, ln 4 weigh 1, 2, 4), the draw's boundaries
worked out by hand, and stratified draws whose frequencies must equal the
probabilities. Planted mistakes in the oracle (ties to the higher id, the
sampled order sorted instead of by id, >= instead of >, no renormalisation
over the mask, a wrong softmax shift) each fail at least one pin."""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle.qrita_outputs as O

L2, L4 = math.log(2.0), math.log(4.0)


def brute_order(vals):
    """Lexicographically smallest permutation whose values do not increase."""
    best = None
    for perm in itertools.permutations(range(len(vals))):
        if all(vals[perm[i]] >= vals[perm[i + 1]] for i in range(len(vals) - 1)):
            if best is None or perm < best:
                best = perm
    return list(best)


def test_topk_ids_equal_the_brute_force_order_on_every_tiny_row():
    alphabet = [-1.0, 0.0, 2.5]
    for V in range(1, 6):
        for row in itertools.product(alphabet, repeat=V):
            order = brute_order(row)
            for k in range(0, V + 2):
                assert O.topk_ids(row, k) == order[: max(0, min(k, V))], (row, k)


def test_topk_ids_handworked():
    assert O.topk_ids([3.0, 1.0, 3.0, 2.0], 2) == [0, 2]
    assert O.topk_ids([3.0, 1.0, 3.0, 2.0], 3) == [0, 2, 3]
    assert O.topk_ids([0.0, -0.0, 0.0], 2) == [0, 1]  # -0 == +0: ids in order
    assert O.topk_ids([-np.inf, 1.0, -np.inf], 3) == [1, 0, 2]
    assert O.topk_ids([1.0, np.nan], 1) == []
    assert O.topk_ids([1.0, np.inf], 1) == []
    assert O.topk_ids([5.0, 7.0], 0) == []


def _exact_probs(a, keep):
    # logits a_i ln 2: weights 2^(a_i), exact
    w = [Fraction(2) ** ai for ai, kk in zip(a, keep) if kk]
    z = sum(w)
    return [wi / z for wi in w]


def test_candidates_exact_rational_probabilities():
    a = [1, 0, 2, 1, 0, 2]
    x = [ai * L2 for ai in a]
    for keep in itertools.product([0, 1], repeat=len(a)):
        if not any(keep):
            ids, probs = O.candidates(x, keep)
            assert ids.size == 0
            continue
        ids, probs = O.candidates(x, keep)
        assert ids.tolist() == [i for i, kk in enumerate(keep) if kk]
        want = _exact_probs(a, keep)
        assert np.allclose(probs, [float(f) for f in want], rtol=1e-14, atol=0)


def test_sample_boundaries_by_hand():
    # kept logits ln2, 0, ln4, ln2 (ids 0..3): probabilities 2/9, 1/9, 4/9, 2/9,
    # cumulative 2/9, 3/9, 7/9, 1 in id order
    x = [L2, 0.0, L4, L2]
    mask = [1, 1, 1, 1]
    cases = [(0.0, 0), (0.2, 0), (2 / 9 - 1e-9, 0), (2 / 9 + 1e-9, 1), (0.3, 1), (0.34, 2), (0.7, 2),
             (0.78, 3), (0.999999, 3)]
    for u, tok in cases:
        got, _ = O.sample(x, mask, u)
        assert got == tok, (u, got, tok)
    # exactly on a cumulative boundary the next token is drawn ("exceeds"), flagged
    got, amb = O.sample(x, mask, 2 / 9)
    assert amb
    # renormalised over the mask: ids 0, 2, 3 weigh 2, 4, 2 -> cumulative 1/4, 3/4, 1
    sub = [1, 0, 1, 1]
    assert O.sample(x, sub, 0.2)[0] == 0
    assert O.sample(x, sub, 0.3)[0] == 2
    assert O.sample(x, sub, 0.8)[0] == 3
    assert O.sample(x, [0, 0, 0, 0], 0.5) == (-1, False)


def test_stratified_draws_reproduce_the_probabilities():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(40) * 2
    mask = (rng.random(40) < 0.5).astype(np.uint8)
    mask[7] = 1
    ids, probs = O.candidates(x, mask)
    N = 20000
    counts = {int(i): 0 for i in ids}
    for j in range(N):
        tok, _ = O.sample(x, mask, (j + 0.5) / N)
        counts[tok] += 1
    freq = np.array([counts[int(i)] for i in ids]) / N
    assert np.abs(freq - probs).max() <= 1.0 / N + 1e-12


def test_shift_invariance_and_huge_logits():
    x = np.array([1000.0, 999.0, 1000.0, -np.inf])
    ids, probs = O.candidates(x, [1, 1, 1, 1])
    e = math.exp(-1.0)
    assert np.allclose(probs, [1 / (2 + e), e / (2 + e), 1 / (2 + e), 0.0], rtol=1e-14)


# --------------------------------------------------------------------------
# Planted mistakes: each mutant of the oracle fails one of the pins above
# --------------------------------------------------------------------------
def _mut_topk_high_id(x, k):
    x = np.asarray(x, np.float64)
    if k < 1 or not O._valid(x):
        return []
    order = sorted(range(x.shape[0]), key=lambda i: (-x[i], -i))  # ties to the higher id
    return order[: min(k, x.shape[0])]


def _mut_sample_ge(x, mask, u):
    ids, probs = O.candidates(x, mask)
    c = np.cumsum(probs)
    hits = np.nonzero(c >= u)[0]
    return int(ids[hits[0]]), False


def _mut_sample_sorted(x, mask, u):
    ids, probs = O.candidates(x, mask)
    order = np.argsort(-probs, kind="stable")
    c = np.cumsum(probs[order])
    return int(ids[order][np.nonzero(c > u)[0][0]]), False


def _mut_candidates_no_renorm(x, mask):
    x = np.asarray(x, np.float64)
    ids = np.nonzero(np.asarray(mask))[0]
    w = np.exp(x - x.max())
    return ids.astype(np.int64), w[ids] / w.sum()


def _pins_fail(monkeypatch, name, fn, tests):
    monkeypatch.setattr(O, name, fn)
    failed = 0
    for t in tests:
        try:
            t()
        except AssertionError:
            failed += 1
    return failed


def test_planted_mistakes_fail_the_pins(monkeypatch):
    pins = [test_topk_ids_equal_the_brute_force_order_on_every_tiny_row, test_topk_ids_handworked,
            test_candidates_exact_rational_probabilities, test_sample_boundaries_by_hand,
            test_stratified_draws_reproduce_the_probabilities]
    with monkeypatch.context() as m:
        assert _pins_fail(m, "topk_ids", _mut_topk_high_id, pins) >= 1
    with monkeypatch.context() as m:
        m.setattr(O, "sample", _mut_sample_sorted)
        assert _pins_fail(m, "sample", _mut_sample_sorted, pins) >= 1
    with monkeypatch.context() as m:
        assert _pins_fail(m, "candidates", _mut_candidates_no_renorm, pins) >= 1
    # >= instead of >: only a draw exactly on a boundary tells them apart
    x = [L2, 0.0, L4, L2]
    assert _mut_sample_ge(x, [1, 1, 1, 1], 2 / 9)[0] != O.sample(x, [1, 1, 1, 1], 2 / 9)[0]
