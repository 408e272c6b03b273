"""The truncation tables the kernel receives, pinned to an independent normal
quantile (Qrita technical summary, "Methodology", part 1: delta comes from
tables precomputed from the normal quantile function, keyed on k or p).

The library builds its tables on the host by bisection on the C library's
erfc; these tests read them back through qrita_delta_table (no device is
touched) and compare every entry with scipy's ndtri in fp64. A wrong key
(an index off by one, the wrong power of two), a wrong sign or the upper
tail taken for the lower one moves some entry far beyond float rounding.
"""

import math

import numpy as np
import pytest

scipy_special = pytest.importorskip("scipy.special")


@pytest.fixture(scope="module")
def q():
    import os

    from top_selection_row_gb300.build import LIB_PATH, build_library

    if not os.path.exists(LIB_PATH):
        build_library()
    import top_selection_row_gb300 as q

    q.lib()
    return q


def _close(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    same_inf = np.isinf(want) & (got == want)
    # float32 rounding of an fp64 value, plus the bisection's 1e-13 bracket
    tol = np.abs(want) * 2.0**-23 + 1e-9
    with np.errstate(invalid="ignore"):  # inf - inf where both are infinite
        return same_inf | (np.abs(got - want) <= tol)


def test_top_k_table_is_the_upper_normal_quantile(q):
    lut = q.delta_table(0)
    assert lut.shape == (128,)
    i = np.arange(lut.shape[0], dtype=np.float64)
    u = np.exp2(-i / 4.0)
    # Phi^-1(1 - u), computed in the accurate tail as -Phi^-1(u)
    want = -scipy_special.ndtri(u)
    ok = _close(lut, want)
    assert ok.all(), np.nonzero(~ok)[0][:5]
    assert lut[0] == -np.inf  # u = 1: no truncation threshold below every logit
    assert np.all(np.diff(lut) > 0)  # smaller u, higher threshold


def test_top_p_table_is_the_normal_quantile_of_one_minus_p(q):
    lut = q.delta_table(1)
    assert lut.shape == (64,)
    i = np.arange(lut.shape[0], dtype=np.float64)
    qv = np.exp2(-i / 4.0)
    want = scipy_special.ndtri(qv)
    ok = _close(lut, want)
    assert ok.all(), np.nonzero(~ok)[0][:5]
    assert lut[0] == np.inf
    assert np.all(np.diff(lut) < 0)


def test_tables_against_a_second_quantile_route(q):
    """The same entries from the complementary error function's inverse:
    Phi^-1(y) = -sqrt(2) erfcinv(2 y)."""
    for which, sign in ((0, -1.0), (1, 1.0)):
        lut = q.delta_table(which).astype(np.float64)
        for i in range(1, lut.shape[0]):
            y = 2.0 ** (-i / 4.0)
            want = sign * (-math.sqrt(2.0) * scipy_special.erfcinv(2.0 * y))
            assert abs(lut[i] - want) <= abs(want) * 2.0**-23 + 1e-9, (which, i, lut[i], want)


def test_unknown_table_is_refused(q):
    assert q.lib().qrita_delta_table(2, None, 0) == -1
    with pytest.raises(ValueError):
        q.delta_table(5)
