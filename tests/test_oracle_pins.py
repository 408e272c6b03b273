"""Pins that tie the CPU oracle to the definition, not to itself.

The oracle restates the sort-based definition (Qrita technical summary,
gist.science paper 2602.01518, "Problem statement" and "Results": Qrita's
candidate set equals the sort-based top-k / top-p result). These tests check
it against things fixed independently of its code:

* hand-worked rows (tests/golden/handworked_rows.txt);
* brute force on every row of tiny vocabularies: the stable descending order
  found by enumerating permutations, masses in exact rationals (weights
  1, 2, 4) or 50-digit arithmetic;
* closed forms: k = 1 is the lowest-index argmax, p -> 0 keeps one token,
  equal logits keep ceil(p * V) tokens under top-p;
* the sort step against two independent stable sorts (torch, numpy lexsort);
* invariants on random tie-heavy rows.

Each plausible mistake planted in the oracle (ties to the higher id, the
reverse order, c > p instead of c >= p, a sign error in the softmax shift, an
off-by-one prefix) must make at least one of these fail.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle.qrita_oracle as O

P_GRID = [-0.5, 0.0, 1e-9, 0.1, 0.25, 1 / 3, 0.5, 0.6, 0.75, 0.9, 0.999, 1.0, float("nan")]


# --------------------------------------------------------------------------
# Independent restatements used only as pins
# --------------------------------------------------------------------------

def brute_stable_order(vals):
    """Lexicographically smallest permutation whose values do not increase."""
    V = len(vals)
    best = None
    for perm in itertools.permutations(range(V)):
        if all(vals[perm[i]] >= vals[perm[i + 1]] for i in range(V - 1)):
            if best is None or perm < best:
                best = perm
    return list(best)


def brute_kept(vals, k, p, exact_weights):
    """Kept ids and the expected boundary-band flag, by enumeration.

    exact_weights(vals_in_S, m) returns exact masses (Fraction or mpf). The
    flag is set when the exact prefix mass at j* or j*-1 lies within
    1e-6 * |p| of p, the band the oracle documents.
    """
    V = len(vals)
    order = brute_stable_order(vals)
    s_k = order[:k] if (k is not None and 1 <= k < V) else order
    if p is None or math.isnan(p) or p >= 1.0:
        return set(s_k), False
    m = vals[order[0]]
    w = exact_weights([vals[i] for i in s_k], m)
    z = sum(w[1:], w[0])
    exact = isinstance(w[0], Fraction)
    pe = Fraction(p) if exact else p
    band = Fraction(1, 10**6) * abs(pe) if exact else 1e-6 * abs(p)
    cs = []
    acc = w[0] * 0
    for wj in w:
        acc = acc + wj
        cs.append(acc / z)
    j_star = next((j for j, c in enumerate(cs) if c >= pe), len(cs) - 1)
    near = abs(cs[j_star] - pe) <= band or (j_star > 0 and abs(cs[j_star - 1] - pe) <= band)
    return set(s_k[: j_star + 1]), bool(near)


def rational_weights(xs, m):
    # values are a*ln2 with a in {0,1,2}; w = 2^(a - a_max) exactly
    am = round(m / math.log(2))
    return [Fraction(2) ** (round(x / math.log(2)) - am) for x in xs]


def mp_weights(xs, m):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    if m == -math.inf:
        return [mpmath.mpf(1) for _ in xs]
    return [mpmath.mpf(0) if x == -math.inf else mpmath.exp(mpmath.mpf(x) - mpmath.mpf(m)) for x in xs]


# --------------------------------------------------------------------------
# Pin suites (return failure lists so the mutation tests can reuse them)
# --------------------------------------------------------------------------

def golden_failures(cases):
    fails = []
    for c in cases:
        res = O.select_row(np.array(c["x"]), c["k"], c["p"])
        kept = sorted(np.nonzero(res.mask)[0].tolist())
        status = "ok" if res.status == O.STATUS_OK else "nonfinite"
        if kept != c["kept"] or status != c["status"] or res.ambiguous != c["ambiguous"]:
            fails.append((c["name"], kept, status, res.ambiguous))
    return fails


def brute_failures(alphabet, weights, max_v, ks_extra=(-1, 0)):
    fails = []
    for V in range(1, max_v + 1):
        for row in itertools.product(alphabet, repeat=V):
            vals = list(row)
            ks = sorted(set(list(ks_extra) + list(range(1, V + 2))))
            for k in ks:
                for p in P_GRID:
                    want, near = brute_kept(vals, k, p, weights)
                    res = O.select_row(np.array(vals), k, p)
                    got = set(np.nonzero(res.mask)[0].tolist())
                    if near:
                        # exact mass within the band: the oracle must flag the
                        # row, and its prefix may differ from the exact one by
                        # one token
                        alts = [set(np.nonzero(a)[0].tolist()) for a in res.alt_masks]
                        if not res.ambiguous or (got != want and want not in alts):
                            fails.append((vals, k, p, sorted(got), sorted(want), "band"))
                    elif got != want or res.ambiguous:
                        fails.append((vals, k, p, sorted(got), sorted(want)))
    return fails


def closed_form_failures(seed=7, rows=40):
    rng = np.random.default_rng(seed)
    fails = []
    for _ in range(rows):
        V = int(rng.integers(1, 300))
        x = np.round(rng.standard_normal(V) * 2) / 2  # many ties
        # k = 1: the lowest-index argmax (np.argmax returns the first maximum)
        r = O.select_row(x, 1, 1.0)
        if np.nonzero(r.mask)[0].tolist() != [int(np.argmax(x))]:
            fails.append(("k1", V))
        # p -> 0+: one token, the same lowest-index argmax
        r = O.select_row(x, 0, 1e-30)
        if np.nonzero(r.mask)[0].tolist() != [int(np.argmax(x))]:
            fails.append(("p0", V))
        # equal logits: top-p keeps the ceil(p V) lowest ids (p*V kept off integers)
        pv = float(rng.uniform(0.05, 0.95))
        if abs(pv * V - round(pv * V)) < 1e-3:
            pv += 0.3 / V
            pv = min(pv, 0.999)
        r = O.select_row(np.full(V, 0.25), 0, pv)
        n = math.ceil(pv * V)
        if np.nonzero(r.mask)[0].tolist() != list(range(n)):
            fails.append(("equal", V, pv))
        # both filters off: all kept
        if O.select_row(x, 0, 1.0).kept != V:
            fails.append(("all", V))
    return fails


# --------------------------------------------------------------------------
# Tests
# --------------------------------------------------------------------------

def test_golden_handworked_rows(golden_rows):
    assert len(golden_rows) >= 20
    assert golden_failures(golden_rows) == []


def test_brute_force_rational_weights():
    alphabet = [0.0, math.log(2), 2 * math.log(2)]
    assert brute_failures(alphabet, rational_weights, 5) == []


def test_brute_force_high_precision_with_neg_inf():
    pytest.importorskip("mpmath")
    alphabet = [-math.inf, 0.0, 1.0, 2.0]
    assert brute_failures(alphabet, mp_weights, 4) == []


def test_closed_forms():
    assert closed_form_failures() == []


def test_sort_step_matches_two_independent_stable_sorts():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    for _ in range(20):
        V = int(rng.integers(1, 5000))
        x = np.round(rng.standard_normal(V) * 4) / 4
        x[rng.random(V) < 0.05] = -np.inf
        x[rng.random(V) < 0.05] = -0.0
        ours = O._stable_descending_order(x)
        t = torch.sort(torch.from_numpy(x), descending=True, stable=True).indices.numpy()
        lex = np.lexsort((np.arange(V), -x))  # primary key -x, then id
        assert np.array_equal(ours, t)
        assert np.array_equal(ours, lex)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x4049], np.uint16)
    want = [1.0, -1.0, 0.0, -0.0, math.inf, -math.inf, 2.0 ** -133, 3.140625]
    got = O.bf16_bits_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w and math.copysign(1, g) == math.copysign(1, w)


def test_invariants_on_random_tie_heavy_rows():
    rng = np.random.default_rng(11)
    for _ in range(60):
        V = int(rng.integers(2, 3000))
        x = np.round(rng.standard_normal(V) * rng.choice([1, 4, 16])) / 8
        k = int(rng.integers(-2, V + 2))
        p = float(rng.choice([rng.uniform(0.01, 0.999), 1.0]))
        r = O.select_row(x, k, p)
        kept = np.nonzero(r.mask)[0]
        dropped = np.nonzero(r.mask == 0)[0]
        k_on = 1 <= k < V
        assert kept.size >= 1
        if p >= 1.0:
            assert kept.size == (k if k_on else V)
        if dropped.size:
            assert x[kept].min() >= x[dropped].max()
            b = x[kept].min()
            kb = kept[x[kept] == b]
            db = dropped[x[dropped] == b]
            if db.size:
                assert kb.max() < db.min()
        # top-p kept is a subset of top-k kept
        rk = O.select_row(x, k, 1.0)
        assert np.all(rk.mask[kept] == 1)
        if p < 1.0:
            sk = np.nonzero(rk.mask)[0]
            m = x.max()
            w_all = np.exp(x - m)
            z = math.fsum(w_all[sk])
            mass = math.fsum(w_all[kept])
            assert mass >= p * z * (1 - 1e-12)
            # removing the last kept token in sort order drops below p
            order = np.lexsort((np.arange(V), -x))
            last = [i for i in order if r.mask[i]][-1]
            if kept.size > 1 and not r.ambiguous:
                assert mass - w_all[last] < p * z


# --------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin suite
# --------------------------------------------------------------------------

def _pin_failures(golden_rows):
    f = golden_failures(golden_rows)
    f += brute_failures([0.0, math.log(2), 2 * math.log(2)], rational_weights, 4)
    f += closed_form_failures(rows=10)
    return f


@pytest.mark.parametrize(
    "name,attr,mutant",
    [
        ("ties_to_higher_id", "_stable_descending_order",
         lambda x: np.lexsort((-np.arange(len(x)), -x))),
        ("ascending_order", "_stable_descending_order",
         lambda x: np.argsort(x, kind="stable")),
        ("exclusive_p", "_first_reaching",
         lambda c, p: (int(np.nonzero(c > p)[0][0]) if np.any(c > p) else c.shape[0] - 1)),
        ("shift_sign", "_softmax_weights",
         lambda xs, m: np.where(xs == m, 1.0, np.exp(np.clip(m - xs, -700, 700)))),
        ("prefix_off_by_one", "_mask_from_prefix",
         lambda V, order, count: np.isin(np.arange(V), order[: count + 1]).astype(np.uint8)),
    ],
)
def test_planted_mistakes_are_caught(monkeypatch, golden_rows, name, attr, mutant):
    monkeypatch.setattr(O, attr, mutant)
    assert _pin_failures(golden_rows), f"mutant {name} slipped through every pin"


def test_band_accepts_every_prefix_the_band_cannot_tell_apart():
    """On a row of millions of equal logits each token carries 1/V of the
    mass, so the 1e-6 relative band around p covers several prefix ends:
    c_n = n / V exactly, and for p = 1/2 the band holds counts
    V/2 - 3 .. V/2 + 3 (1e-6 * 0.5 * 6e6 = 3). Exactly those prefixes are
    accepted; a longer or shorter one, or a non-prefix of an accepted count,
    is not."""
    from oracle import accepts, select_row

    V = 6_000_000
    res = select_row(np.zeros(V), None, 0.5)
    half = V // 2
    assert res.ambiguous and res.kept == half
    assert res.band_kept == (half - 3, half + 3)

    def prefix(n):
        m = np.zeros(V, np.uint8)
        m[:n] = 1
        return m

    for n in range(half - 3, half + 4):
        assert accepts(res, prefix(n)), n
    for n in (half - 4, half + 4):
        assert not accepts(res, prefix(n)), n
    bad = prefix(half + 1)
    bad[half] = 0
    bad[V - 1] = 1
    assert not accepts(res, bad)
