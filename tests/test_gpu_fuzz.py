"""Seeded random parity cases: the CUDA path through the C ABI against the
CPU oracle over random row lengths, value distributions, per-row k / p and
forced paths.

Each case draws V (half the cases log-uniformly in [1, 400000], half
uniformly in [20000, 400000]), a batch of rows from one of
several value families (Gaussian at a random temperature, Gaussian with
outliers, quantised values with many ties, uniform, heavy-tailed, bimodal, a
few distinct values, sorted rows, constant rows, rows mostly masked to -inf),
and per-row k and p that include the edges (0, 1, V - 1, V, above V; p of 0,
tiny, near 1, 1). A quarter of the cases also force a path (cluster size,
fallback, key pivots, second truncation, missed histogram bracket). The pass
rule is the oracle's: bit-exact, except flagged top-p rows, which must lie in
the oracle's band.
"""

import math

import numpy as np
import pytest

from parity_helpers import check_against_oracle

pytestmark = pytest.mark.gpu

N_CASES = 160
MAX_ELEMS = 1_500_000  # per case, so the oracle finishes each in about a second
FAMILIES = ("normal", "outliers", "quantised", "uniform", "heavy", "bimodal", "few", "sorted", "constant",
            "masked")


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_selection_row_gb300 as q

    q.lib()  # must load: no fallback exists
    return torch.device("cuda", 0)


def _rows(rng, family, B, V):
    if family == "normal":
        x = rng.standard_normal((B, V)) * rng.uniform(0.2, 3.0) + rng.uniform(-5, 5)
    elif family == "outliers":
        x = rng.standard_normal((B, V))
        n_out = min(V, int(rng.integers(1, 65)))
        for r in range(B):
            pos = rng.choice(V, n_out, replace=False)
            x[r, pos] = rng.uniform(4, 12, n_out)
    elif family == "quantised":
        q = float(rng.choice([1.0, 2.0, 8.0]))
        x = np.round(rng.standard_normal((B, V)) * q) / q
    elif family == "uniform":
        a = rng.uniform(-3, 3)
        x = rng.uniform(a, a + rng.uniform(0.01, 4.0), (B, V))
    elif family == "heavy":
        x = rng.gumbel(size=(B, V)) * rng.uniform(0.5, 2.0)
    elif family == "bimodal":
        x = rng.standard_normal((B, V)) * 0.5 + np.where(rng.random((B, V)) < 0.1, 4.0, 0.0)
    elif family == "few":
        vals = rng.standard_normal(3) * 2
        x = vals[rng.integers(0, 3, (B, V))]
    elif family == "sorted":
        x = np.sort(rng.standard_normal((B, V)), axis=1)
        x[1::2] = x[1::2, ::-1]
    elif family == "constant":
        x = np.full((B, V), rng.uniform(-2, 2))
    else:  # masked: most logits -inf, as constrained decoding leaves them
        x = rng.standard_normal((B, V))
        x[rng.random((B, V)) < rng.uniform(0.5, 0.999)] = -np.inf
        x[:, int(rng.integers(0, V))] = 1.0  # at least one finite logit
    return x.astype(np.float32)


def _k_values(rng, V, B):
    choices = [0, 1, 2, V - 1, V, V + 5, max(1, V // 2)]
    k = np.empty(B, np.int64)
    for r in range(B):
        u = rng.random()
        if u < 0.4:
            k[r] = choices[int(rng.integers(0, len(choices)))]
        elif u < 0.7:
            k[r] = int(rng.integers(1, min(V, 64) + 1))
        else:
            k[r] = int(rng.integers(1, V + 1))
    return k.astype(np.int32)


def _p_values(rng, B):
    choices = [1.0, 1.0, 0.0, 1e-4, 0.5, 0.9, 0.99, 0.999999]
    p = np.empty(B, np.float32)
    for r in range(B):
        p[r] = choices[int(rng.integers(0, len(choices)))] if rng.random() < 0.5 else rng.uniform(0.0, 1.0)
    return p


def _flags(rng):
    import top_selection_row_gb300 as q

    if rng.random() >= 0.25:
        return 0
    pick = [
        q.flag_cluster(1),
        q.flag_cluster(2),
        q.flag_cluster(8),
        q.flag_cluster(16),
        q.FLAG_FORCE_FALLBACK,
        q.FLAG_KEY_PIVOTS,
        q.FLAG_NO_TRUNCATION,
        q.FLAG_FORCE_RETRY,
        q.FLAG_HIST_MISS,
        q.FLAG_FORCE_FALLBACK | q.FLAG_KEY_PIVOTS,
    ]
    return pick[int(rng.integers(0, len(pick)))]


def _case(i):
    rng = np.random.default_rng(10_000 + i)
    if rng.random() < 0.5:
        V = max(1, int(math.exp(rng.uniform(0.0, math.log(400_000)))))
    else:
        V = int(rng.integers(20_000, 400_001))
    B = int(rng.integers(1, 13))
    B = max(1, min(B, MAX_ELEMS // V))
    dtype = "bf16" if rng.random() < 0.4 else "f32"
    family = FAMILIES[int(rng.integers(0, len(FAMILIES)))]
    x = _rows(rng, family, B, V)
    if dtype == "bf16":
        from workloads import f32_to_bf16_bits

        x = f32_to_bf16_bits(x)
    return dtype, family, x, _k_values(rng, V, B), _p_values(rng, B), rng


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(dev, i):
    dtype, family, x, k, p, rng = _case(i)
    flags = _flags(rng)
    fails, flagged, got, st, info = check_against_oracle(x, dtype, k, p, dev, flags=flags)
    assert fails == [], (i, dtype, family, x.shape, hex(flags), fails[:4])
