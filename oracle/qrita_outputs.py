"""CPU oracle for the candidate-set outputs beyond the keep-mask.

TEST INFRASTRUCTURE ONLY, like qrita_oracle: nothing on the product path
imports it, and it shares no code with the CUDA library.

Qrita technical summary (gist.science, paper 2602.01518), "Problem
statement": the full candidate set, not one sampled token, is what
speculative-decoding verification and reinforcement learning consume, and
the sort-based methods produce it exactly. The steps right after the mask
are written out here in their plain definitions:

* ``topk_ids(x, k)``: the first min(k, V) token ids of the stable
  descending order (equal logits: lower id first; -0 == +0; -inf last), in
  that order: the ids a drafter keeps for its top-k (e.g. k = 512);
* ``candidates(x, mask)``: the kept ids in increasing id order with their
  probabilities renormalised over the kept set, p_i = exp(x_i - m) / sum over
  the kept ids of exp(x_j - m), m their largest logit (a kept logit equal to
  m weighs exactly 1), in fp64;
* ``sample(x, mask, u)``: one token drawn from those probabilities by the
  inverse distribution function with a caller-supplied uniform u in [0, 1):
  walking the kept ids in increasing id order, the first one whose
  cumulative probability exceeds u. The pages fix no order for the draw; any
  fixed order draws from the same distribution, and id order needs no sort.

A row holding NaN or +inf has no candidates (the mask is all zero there).
``sample`` flags a draw as ambiguous when u lies within 1e-6 of the
cumulative probability at the chosen token or at the one before it: there
an fp32 computation may pick the neighbour.

Pins: tests/test_oracle_outputs.py (exact rational probabilities, brute-force
orders on tiny rows, stratified draws against the probabilities, planted
mistakes).
"""

from __future__ import annotations

import numpy as np

SAMPLE_BAND = 1e-6


def _valid(x: np.ndarray) -> bool:
    return not (np.isnan(x).any() or np.isposinf(x).any())


def topk_ids(x, k: int) -> list[int]:
    """The first min(k, V) ids of the stable descending order of row x
    (fp64 values); [] for k < 1 or a row holding NaN / +inf."""
    x = np.asarray(x, dtype=np.float64)
    if k < 1 or not _valid(x):
        return []
    order = np.argsort(-x, kind="stable")  # -0.0 == +0.0: ties keep id order
    return [int(i) for i in order[: min(k, x.shape[0])]]


def candidates(x, mask):
    """(ids, probs): the kept ids in increasing order and their fp64
    probabilities renormalised over the kept set."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.nonzero(np.asarray(mask))[0]
    if ids.size == 0 or not _valid(x):
        return np.zeros(0, np.int64), np.zeros(0, np.float64)
    xs = x[ids]
    m = xs.max()
    with np.errstate(invalid="ignore", over="ignore"):
        w = np.where(xs == m, 1.0, np.exp(xs - m))
    return ids.astype(np.int64), w / w.sum()


def sample(x, mask, u: float):
    """(token, ambiguous): the first kept id, in increasing id order, whose
    cumulative probability exceeds u; -1 when nothing is kept."""
    ids, probs = candidates(x, mask)
    if ids.size == 0:
        return -1, False
    c = np.cumsum(probs)
    hits = np.nonzero(c > u)[0]
    j = int(hits[0]) if hits.size else ids.size - 1  # rounding can leave c[-1] just below 1
    near = abs(c[j] - u) <= SAMPLE_BAND or (j > 0 and abs(c[j - 1] - u) <= SAMPLE_BAND)
    return int(ids[j]), bool(near)
