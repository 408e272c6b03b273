"""Plain, slow, obviously correct CPU oracle for exact top-k / top-p selection.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module;
the CUDA library shares no code, table or helper with it.

What it computes, and where the pages fix it
--------------------------------------------
Qrita technical summary (gist.science, paper 2602.01518), section "Problem
statement": sort-based top-k/top-p (as in vLLM) is exact and deterministic
but sorts the whole vocabulary; the goal is the *full candidate set* with the
exact top-k / top-p semantics. Section "Results": Qrita's output matches the
sort-based algorithms. So the oracle is the sort-based definition itself,
written out in fp64, not Qrita's steps:

1. widen the row to fp64 (exact for fp32 and bf16);
2. pi = stable sort of token ids by descending logit; ties keep the lower
   token id first; -0 and +0 are equal; -inf sorts last;
3. top-k: S_k = pi[0:k] when 1 <= k < V, else the whole row;
4. softmax over S_k in fp64 with the row max m as shift,
   w_i = exp(x_i - m) (w_i = 1 where x_i == m, which also covers a row whose
   max is -inf: equal logits give equal probability);
5. c_j = (w_{pi[0]} + ... + w_{pi[j]}) / Z_k for j < |S_k|;
6. top-p: keep pi[0..j*], j* = the smallest j with c_j >= p (the last index
   if rounding leaves every c_j below p); p >= 1 or NaN disables top-p;
7. the mask is 1 on the kept tokens.

Top-k is applied before top-p, and top-p renormalises over S_k; the pages
name both filters but not their order, and this is the reading taken.
A row holding NaN or +inf is invalid: its mask is all zero.

Boundary-band flag: when top-p is active the row is flagged ambiguous if
|c_{j*} - p| <= 1e-6 * p or |c_{j*-1} - p| <= 1e-6 * p. On such rows any
prefix of the stable order is accepted whose end the band cannot tell from
the boundary: the count n with c_{n-1} >= p - 1e-6 p (it reaches p within
the band) and c_{n-2} < p + 1e-6 p (one token fewer falls short within the
band). On short rows that is the oracle's prefix or one token more or less;
on rows of millions of logits, whose tokens each carry far less than 1e-6 of
the mass, it can be several.

Pins (tests/test_oracle_pins.py, tests/golden/): brute-force permutation
enumeration on tiny rows with exact rational weights, hand-worked tie-heavy
rows, closed forms (k = 1 is the lowest-index argmax, p -> 0 keeps one token,
equal rows keep ceil(p*V) tokens), cross-checks of the sort step against two
independent stable sorts, and invariants on random rows.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Relative width of the top-p boundary band (see module docstring).
AMBIGUITY_REL = 1e-6

STATUS_OK = 0
STATUS_NONFINITE = 1  # NaN or +inf in the row


@dataclass
class RowResult:
    """Per-row outcome of the definition.

    mask       uint8[V], 1 on kept tokens
    status     STATUS_OK or STATUS_NONFINITE
    kept       number of kept tokens
    boundary   value of the last kept token in sort order (None when invalid)
    n_boundary how many tokens equal to ``boundary`` are kept
    ambiguous  top-p boundary within the relative band of p
    alt_masks  masks of the neighbouring prefixes (only when ambiguous)
    band_kept  (smallest, largest) accepted count of kept tokens
    band_order the order of S_k (only when ambiguous), for accepts()
    """

    mask: np.ndarray
    status: int
    kept: int
    boundary: float | None
    n_boundary: int
    ambiguous: bool
    alt_masks: tuple
    band_kept: tuple = (0, 0)
    band_order: np.ndarray | None = None


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) exactly: bf16 is the top half of fp32."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def _stable_descending_order(x: np.ndarray) -> np.ndarray:
    # Negation is exact in fp64; numpy's 'stable' sort keeps equal keys in
    # input order, and -0.0 == +0.0 compare equal, so ties go to the lower id.
    return np.argsort(-x, kind="stable")


def _softmax_weights(xs: np.ndarray, m: float) -> np.ndarray:
    # w = exp(x - m); a token equal to the max weighs exactly 1, which also
    # defines the all -inf row (equal logits, equal probability).
    with np.errstate(invalid="ignore", over="ignore"):
        return np.where(xs == m, 1.0, np.exp(xs - m))


def _first_reaching(c: np.ndarray, p: float) -> int:
    # Smallest j with c_j >= p; the last index if rounding keeps all below p.
    hits = np.nonzero(c >= p)[0]
    return int(hits[0]) if hits.size else c.shape[0] - 1


def _mask_from_prefix(V: int, order: np.ndarray, count: int) -> np.ndarray:
    mask = np.zeros(V, dtype=np.uint8)
    mask[order[:count]] = 1
    return mask


def select_row(x, k: int | None, p: float | None) -> RowResult:
    """Apply the sort-based definition to one row of logits.

    ``x`` is any real array (fp32 / fp64 values, or already-widened bf16).
    ``k`` <= 0, ``k`` >= V or None disables top-k. ``p`` >= 1, NaN or None
    disables top-p; ``p`` <= 0 keeps exactly one token (c_0 >= p always).
    """
    x = np.asarray(x, dtype=np.float64)
    V = x.shape[0]
    if np.isnan(x).any() or np.isposinf(x).any():
        return RowResult(np.zeros(V, np.uint8), STATUS_NONFINITE, 0, None, 0, False, ())

    order = _stable_descending_order(x)

    # Step 3: top-k prefix of the stable order.
    if k is not None and 1 <= k < V:
        s_k = order[:k]
    else:
        s_k = order

    top_p = p is not None and not np.isnan(p) and p < 1.0
    ambiguous = False
    alts: tuple = ()
    band_kept = None
    if not top_p:
        n_keep = s_k.shape[0]
    else:
        # Step 4: softmax over S_k, shifted by the row max m = x[pi[0]].
        xs = x[s_k]
        m = x[order[0]]
        w = _softmax_weights(xs, m)
        z_k = w.sum()
        # Step 5: cumulative mass in sort order.
        c = np.cumsum(w) / z_k
        # Step 6: the smallest prefix whose mass reaches p.
        j = _first_reaching(c, p)
        n_keep = j + 1
        band = AMBIGUITY_REL * abs(p)
        near_here = abs(c[j] - p) <= band
        near_prev = j > 0 and abs(c[j - 1] - p) <= band
        ambiguous = bool(near_here or near_prev)
        if ambiguous:
            alts = tuple(
                _mask_from_prefix(V, s_k, n)
                for n in (n_keep - 1, n_keep + 1)
                if 1 <= n <= s_k.shape[0]
            )
            # every count whose prefix end the band cannot tell apart
            n_lo = _first_reaching(c, p - band) + 1
            n_hi = _first_reaching(c, p + band) + 1
            band_kept = (min(n_lo, n_keep - 1 if n_keep > 1 else 1), max(n_hi, n_keep + 1))

    mask = _mask_from_prefix(V, s_k, n_keep)
    boundary = float(x[s_k[n_keep - 1]])
    kept_vals = x[s_k[:n_keep]]
    n_boundary = int(np.count_nonzero(kept_vals == boundary))
    if band_kept is None:
        return RowResult(mask, STATUS_OK, int(n_keep), boundary, n_boundary, ambiguous, alts, (int(n_keep), int(n_keep)))
    return RowResult(mask, STATUS_OK, int(n_keep), boundary, n_boundary, ambiguous, alts,
                     (int(band_kept[0]), int(min(band_kept[1], s_k.shape[0]))), s_k)


def accepts(res: RowResult, got: np.ndarray) -> bool:
    """Whether a mask ``got`` (uint8 / bool [V]) is an accepted result for
    the row: the definition's mask, or on a flagged row any prefix of the
    stable order whose count lies in ``band_kept``."""
    g = np.asarray(got).astype(np.uint8)
    if np.array_equal(g, res.mask):
        return True
    if not res.ambiguous or res.band_order is None:
        return False
    n = int(g.sum())
    if not (res.band_kept[0] <= n <= res.band_kept[1]):
        return False
    return np.array_equal(g, _mask_from_prefix(g.shape[0], res.band_order, n))


def select_batch(logits: np.ndarray, dtype: str, k=None, p=None, rows=None):
    """Run :func:`select_row` over the rows of a [B, V] batch.

    ``dtype`` is "f32" (``logits`` float32/float64) or "bf16" (``logits``
    uint16 raw bits). ``k`` / ``p`` are per-row sequences or None.
    ``rows`` optionally restricts the work to a subset of row ids.
    Returns a list of (row id, RowResult).
    """
    if dtype == "bf16":
        widen = bf16_bits_to_f64
    elif dtype == "f32":
        def widen(a):
            return np.asarray(a, dtype=np.float64)
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    B = logits.shape[0]
    ids = range(B) if rows is None else rows
    out = []
    for r in ids:
        kr = None if k is None else int(k[r])
        pr = None if p is None else float(p[r])
        out.append((r, select_row(widen(logits[r]), kr, pr)))
    return out
