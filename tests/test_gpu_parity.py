"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Pass rule (the oracle's): top-k masks and top-p masks of unflagged rows are
bit-exact; rows whose boundary mass lies within 1e-6 relative of p may keep
one token more or fewer. Workloads are the seeded synthetic batches of
``workloads``; small cases run the oracle on every row, full-size cases on
sampled rows plus invariants on every row.
"""

import math

import numpy as np
import pytest

from oracle import select_batch, select_row
from parity_helpers import (check_against_oracle, compare_rows, compare_rows_pooled, invariant_failures, run_gpu,
                            to_device, widen)
from workloads import WORKLOADS, f32_to_bf16_bits, generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_selection_row_gb300 as q

    q.lib()  # must load: no fallback exists
    return torch.device("cuda", 0)


_cache = {}


def workload(n, rows=None):
    key = (n, rows)
    if key not in _cache:
        _cache[key] = generate(n, rows=rows)
    return _cache[key]


# ---------------------------------------------------------------------------
# Workloads: leading rows at full V, every row against the oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_workload_leading_rows(dev, n):
    w = WORKLOADS[n]
    rows = min(w.B, 24)
    logits, k, p = workload(n, rows)
    fails, flagged, got, st, info = check_against_oracle(logits, w.dtype, k, p, dev)
    assert fails == [], fails[:5]


# ---------------------------------------------------------------------------
# Workloads at full size, launched exactly as the bench launches them: every
# row against the oracle (spread over the host cores) and the invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_workload_full_size(dev, n, record_flagged):
    w = WORKLOADS[n]
    logits, k, p = workload(n)
    got, st, info = run_gpu(logits, w.dtype, k, p, dev)
    assert (st == 0).all()
    fails, flagged, bad = compare_rows_pooled(logits, w.dtype, k, p, got, st)
    record_flagged(f"workload {n} {w.name}", flagged, w.B)
    assert fails == [], fails[:5]
    assert bad == [], bad[:5]
    # diagnostics agree with the mask
    assert np.array_equal(info["kept"], got.sum(axis=1).astype(np.uint32))


def test_multi_wave_batch_every_row(dev, record_flagged):
    """A batch of 700 one-CTA rows (more than the device holds at once), half
    of them top-p only, so the launch reorders rows heavy-first across waves;
    every row is compared with the oracle."""
    import top_selection_row_gb300 as q

    rng = np.random.default_rng(700)
    B, V = 700, 32000
    T = rng.uniform(0.5, 1.5, size=(B, 1))
    x = (rng.standard_normal((B, V)) / T).astype(np.float32)
    for r in range(B):
        pos = rng.choice(V, size=16, replace=False)
        x[r, pos] = (rng.uniform(4.0, 10.0, size=16) / T[r, 0]).astype(np.float32)
    p_only = rng.permutation(B) < B // 2
    k = np.where(p_only, V, rng.integers(1, 1000, size=B)).astype(np.int32)
    p = np.where(p_only, rng.uniform(0.5, 0.99, size=B),
                 np.where(rng.random(B) < 0.5, 1.0, rng.uniform(0.8, 1.0, size=B))).astype(np.float32)
    got, st, info = run_gpu(x, "f32", k, p, dev)
    assert (st == 0).all()
    fails, flagged, bad = compare_rows_pooled(x, "f32", k, p, got, st)
    record_flagged("multi-wave b700_v32000_f32_mixed", flagged, B)
    assert fails == [], fails[:5]
    assert bad == [], bad[:5]
    assert ((info["path"] & q.PATH_TOPP) != 0).sum() >= B // 2


@pytest.mark.parametrize("case", ["w2_c16", "w5_c16", "w2_c1", "w3_c2", "w4_c1"])
def test_copy_wait_give_up_voids_only_its_row(dev, case):
    """A bounded wait for a bulk copy that gives up (forced by a test flag on
    the first wait of row 0's first CTA) voids that row: status
    QRITA_ROW_TIMEOUT and an all-zero mask. The copy it gave up on still
    lands and is waited for before the CTA exits, and every other row of the
    batch is still exact against the oracle."""
    import top_selection_row_gb300 as q

    n = int(case[1])
    cl = {"c16": 0, "c1": q.flag_cluster(1), "c2": q.flag_cluster(2)}[case.split("_")[1]]
    w = WORKLOADS[n]
    logits, k, p = workload(n, 8)
    got, st, info = run_gpu(logits, w.dtype, k, p, dev, flags=q.FLAG_TEST_GIVE_UP | cl)
    assert st[0] == q.ROW_TIMEOUT
    assert not got[0].any()
    assert info["status"][0] == q.ROW_TIMEOUT and info["kept"][0] == 0
    ref = select_batch(logits, w.dtype, k, p, rows=list(range(1, 8)))
    fails, _ = compare_rows(got, st, ref)
    assert fails == [], fails[:5]
    # the flag leaves a batch without row 0's CTA untouched: the next call is clean
    again, st2, _ = run_gpu(logits, w.dtype, k, p, dev, flags=cl)
    assert (st2 == 0).all()
    assert np.array_equal(again[1:], got[1:])


# ---------------------------------------------------------------------------
# Hand-worked rows
# ---------------------------------------------------------------------------
def test_golden_rows(dev, golden_rows):
    for c in golden_rows:
        x = np.array([c["x"]], np.float32)
        got, st, _ = run_gpu(x, "f32", np.array([c["k"]]), np.array([c["p"]]), dev)
        kept = sorted(np.nonzero(got[0])[0].tolist())
        if c["status"] == "nonfinite":
            assert st[0] == 1 and kept == [], c["name"]
        elif c["ambiguous"]:
            res = select_row(np.array(c["x"]), c["k"], c["p"])
            ok = [sorted(np.nonzero(a)[0].tolist()) for a in (res.mask,) + res.alt_masks]
            assert kept in ok, (c["name"], kept)
        else:
            assert st[0] == 0 and kept == c["kept"], (c["name"], kept, c["kept"])


# ---------------------------------------------------------------------------
# Edge cases: tiny and ragged V, every k / p corner, tie-heavy values
# ---------------------------------------------------------------------------
def _edge_batch(rng, V, B, dtype, kind):
    if kind == "ties":
        x = np.round(rng.standard_normal((B, V)) * 2) / 4
    elif kind == "equal":
        x = np.full((B, V), 0.5)
    elif kind == "wide":
        x = rng.standard_normal((B, V)) * 30
    else:
        x = rng.standard_normal((B, V))
    x = x.astype(np.float32)
    if dtype == "bf16":
        from workloads import f32_to_bf16_bits

        return f32_to_bf16_bits(x)
    return x


@pytest.mark.parametrize("dtype,V,kind", [("f32", 3_000_017, "normal"), ("bf16", (1 << 24) + 3, "normal"),
                                          ("f32", 3_000_017, "flat")])
def test_very_long_rows(dev, dtype, V, kind):
    """Rows of millions of logits (up to 2^24 + 3): the launch spreads a row
    over up to 16 CTAs; top-k small and large, top-p over flat and peaked
    rows."""
    rng = np.random.default_rng(V + (dtype == "bf16"))
    x = rng.standard_normal((4, V)).astype(np.float32)
    if kind == "flat":
        x *= np.float32(0.3)
    if dtype == "bf16":
        from workloads import f32_to_bf16_bits

        logits = f32_to_bf16_bits(x)
    else:
        logits = x
    k = np.array([1, 5000, V, V], np.int32)
    p = np.array([1.0, 0.9, 0.95, 0.5], np.float32)
    fails, flagged, got, st, info = check_against_oracle(logits, dtype, k, p, dev)
    assert fails == [], fails[:5]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 3, 5, 7, 15, 16, 17, 31, 33, 100, 1000, 4097, 40000])
def test_edge_sizes_and_parameters(dev, dtype, V):
    rng = np.random.default_rng(V * 7 + (dtype == "bf16"))
    ks = sorted({-3, 0, 1, 2, V // 2, V - 1, V, V + 1})
    ps = [float("nan"), -1.0, 0.0, 1e-9, 0.3, 0.9, 0.999999, 1.0]
    for kind in ("normal", "ties", "equal", "wide"):
        combos = [(kk, pp) for kk in ks for pp in ps]
        B = len(combos)
        logits = _edge_batch(rng, V, B, dtype, kind)
        k = np.array([c[0] for c in combos], np.int32)
        p = np.array([c[1] for c in combos], np.float32)
        fails, flagged, got, st, info = check_against_oracle(logits, dtype, k, p, dev)
        assert fails == [], (kind, fails[:5])


def test_special_values(dev):
    V = 3000
    rng = np.random.default_rng(5)
    rows = []
    base = rng.standard_normal(V).astype(np.float32)
    r = base.copy(); r[17] = np.nan; rows.append(r)                      # NaN
    r = base.copy(); r[2999] = np.inf; rows.append(r)                    # +inf
    r = base.copy(); r[::3] = -np.inf; rows.append(r)                    # many -inf
    rows.append(np.full(V, -np.inf, np.float32))                         # all -inf
    r = np.zeros(V, np.float32); r[::2] = -0.0; rows.append(r)           # +-0 ties
    r = (rng.integers(-3, 4, V) * np.float32(1.4e-45)).astype(np.float32); rows.append(r)  # subnormals
    r = base.copy(); r[:5] = 1e30; rows.append(r)                        # huge finite
    r = base.copy(); r[5:] = -3.0e38; rows.append(r)                     # float-lowest masking
    r = np.full(V, 7.0, np.float32); rows.append(r)                      # constant
    logits = np.stack(rows)
    B = logits.shape[0]
    for k_val, p_val in ((1, 1.0), (5, 1.0), (1500, 1.0), (0, 0.5), (0, 0.999), (10, 0.7), (2999, 0.2), (0, 1.0)):
        k = np.full(B, k_val, np.int32)
        p = np.full(B, p_val, np.float32)
        fails, flagged, got, st, info = check_against_oracle(logits, "f32", k, p, dev)
        assert fails == [], (k_val, p_val, fails[:5])
        assert st[0] == 1 and st[1] == 1 and not got[0].any() and not got[1].any()


def test_misaligned_rows(dev):
    """Row starts off the 16-byte grid exercise the head / tail element paths."""
    import torch

    import top_selection_row_gb300 as q

    rng = np.random.default_rng(9)
    for dtype, V in (("f32", 1001), ("f32", 4099), ("bf16", 1003), ("bf16", 8191)):
        B = 6
        full = _edge_batch(rng, V + 3, B, dtype, "ties")
        k = np.array([1, 7, 100, 0, 500, 3], np.int32)
        p = np.array([1.0, 0.8, 1.0, 0.6, 0.95, 0.3], np.float32)
        for off in (1, 2, 3):
            sub = np.ascontiguousarray(full[:, off : off + V])
            # a contiguous [B, V] view starting `off` elements into a buffer
            buf = torch.empty(B * V + off, dtype=torch.float32 if dtype == "f32" else torch.bfloat16, device=dev)
            buf[off:] = to_device(sub.reshape(-1), dtype, dev)
            x = buf[off:].view(B, V)
            mask, st, _ = q.qrita_select_ex(x, torch.from_numpy(k).to(dev), torch.from_numpy(p).to(dev), row_status=True)
            torch.cuda.synchronize()
            got = mask.cpu().numpy().astype(np.uint8)
            ref = select_batch(sub, dtype, k, p)
            fails, _ = compare_rows(got, st.cpu().numpy(), ref)
            assert fails == [], (dtype, V, off, fails[:3])


# ---------------------------------------------------------------------------
# Every path gives the same answer
# ---------------------------------------------------------------------------
def _mixed_batch():
    parts = []
    for n, rows in ((2, 6), (3, 6), (4, 8), (5, 8)):
        logits, k, p = workload(n, rows)
        parts.append((n, logits, k, p))
    return parts


@pytest.mark.parametrize(
    "flags",
    ["none", "no_trunc", "fallback", "key_pivots", "c1", "c2", "c4", "c8", "c16", "fallback_key_c16",
     "retry", "retry_c1", "retry_c16", "retry_key", "hist_miss", "hist_miss_c16", "no_key_hist",
     "no_key_hist_c1", "no_key_hist_c4", "quaternary", "binary", "fallback_quaternary", "fallback_binary_c4",
     "no_trunc_quaternary_c1", "key_pivots_binary"],
)
def test_forced_paths_match_oracle(dev, flags):
    import top_selection_row_gb300 as q

    f = {
        "none": 0,
        "no_trunc": q.FLAG_NO_TRUNCATION,
        "fallback": q.FLAG_FORCE_FALLBACK,
        "key_pivots": q.FLAG_KEY_PIVOTS,
        "c1": q.flag_cluster(1),
        "c2": q.flag_cluster(2),
        "c4": q.flag_cluster(4),
        "c8": q.flag_cluster(8),
        "c16": q.flag_cluster(16),
        "fallback_key_c16": q.FLAG_FORCE_FALLBACK | q.FLAG_KEY_PIVOTS | q.flag_cluster(16),
        "retry": q.FLAG_FORCE_RETRY,
        "retry_c1": q.FLAG_FORCE_RETRY | q.flag_cluster(1),
        "retry_c16": q.FLAG_FORCE_RETRY | q.flag_cluster(16),
        "retry_key": q.FLAG_FORCE_RETRY | q.FLAG_KEY_PIVOTS,
        "hist_miss": q.FLAG_HIST_MISS,
        "hist_miss_c16": q.FLAG_HIST_MISS | q.flag_cluster(16),
        "no_key_hist": q.FLAG_NO_KEY_HIST,
        "no_key_hist_c1": q.FLAG_NO_KEY_HIST | q.flag_cluster(1),
        "no_key_hist_c4": q.FLAG_NO_KEY_HIST | q.flag_cluster(4),
        "quaternary": q.FLAG_SEARCH_QUATERNARY | q.FLAG_NO_KEY_HIST,
        "binary": q.FLAG_SEARCH_BINARY | q.FLAG_NO_KEY_HIST,
        "fallback_quaternary": q.FLAG_FORCE_FALLBACK | q.FLAG_SEARCH_QUATERNARY | q.FLAG_NO_KEY_HIST,
        "fallback_binary_c4": q.FLAG_FORCE_FALLBACK | q.FLAG_SEARCH_BINARY | q.FLAG_NO_KEY_HIST | q.flag_cluster(4),
        "no_trunc_quaternary_c1": q.FLAG_NO_TRUNCATION | q.FLAG_SEARCH_QUATERNARY | q.flag_cluster(1),
        "key_pivots_binary": q.FLAG_KEY_PIVOTS | q.FLAG_SEARCH_BINARY | q.FLAG_NO_KEY_HIST,
    }[flags]
    for n, logits, k, p in _mixed_batch():
        w = WORKLOADS[n]
        fails, flagged, got, st, info = check_against_oracle(logits, w.dtype, k, p, dev, flags=f)
        assert fails == [], (n, fails[:5])
        if flags.startswith("retry"):
            top_k = (k >= 1) & (k < w.V)
            assert ((info["path"][top_k] & q.PATH_RETRY) != 0).all()
        if flags.startswith("hist_miss"):
            assert ((info["path"] & q.PATH_HIST) == 0).all()
        if flags.startswith("no_key_hist"):
            assert ((info["path"] & q.PATH_KEYHIST) == 0).all()


@pytest.mark.parametrize("n,cl", [(4, 0), (5, 0), (4, 16), (5, 2)])
def test_key_histogram_places_bf16_boundaries(dev, n, cl):
    """bf16 rows whose truncation hit place both boundaries with one
    histogram of the survivors' 16-bit keys (merged over the cluster when a
    row spans several CTAs)."""
    import top_selection_row_gb300 as q

    w = WORKLOADS[n]
    logits, k, p = workload(n, 32)
    flags = q.flag_cluster(cl) if cl else 0
    fails, flagged, got, st, info = check_against_oracle(logits, w.dtype, k, p, dev, flags=flags)
    assert fails == [], fails[:5]
    topk = (info["path"] & q.PATH_TOPK) != 0
    hit = ((info["path"] & q.PATH_HIT) != 0) & topk
    kh = (info["path"] & q.PATH_KEYHIST) != 0
    assert hit.sum() >= 8
    assert (kh[topk] == hit[topk]).all()


@pytest.mark.parametrize("cl", [0, 1, 2, 4])
def test_key_window_places_bf16_top_p_rows(dev, cl):
    """bf16 rows whose top-p runs alone over far more survivors than the lists
    hold count a window of 16-bit keys in the streaming pass and place the
    boundary from those exact bins (no extraction pass, no search rounds)."""
    import top_selection_row_gb300 as q

    w = WORKLOADS[5]
    logits, k, p = workload(5, 48)
    flags = q.flag_cluster(cl) if cl else 0
    fails, flagged, got, st, info = check_against_oracle(logits, w.dtype, k, p, dev, flags=flags)
    assert fails == [], fails[:5]
    p_only = (k >= w.V) & (p < 1.0)
    assert p_only.sum() >= 4
    kw = (info["path"] & q.PATH_KEYHIST) != 0
    assert kw[p_only].all()
    assert (info["passes"][p_only] == 1).all()
    # |Z_t|, read off the window's bins and the rare logits, is the count of
    # logits >= t
    for r in np.nonzero(p_only)[0]:
        x = widen(logits[r], w.dtype)
        assert info["survivors"][r] == int(np.count_nonzero(x >= np.float32(info["threshold"][r]))), r


@pytest.mark.parametrize("case", ["above_window", "huge_tie_group", "negative_logits"])
def test_key_window_gives_way(dev, case):
    """Rows the key window cannot settle are still exact: a boundary among
    outliers far above the window, a tie group at the boundary larger than
    the emission collects, rows of negative logits only."""
    import top_selection_row_gb300 as q
    from workloads import f32_to_bf16_bits

    rng = np.random.default_rng({"above_window": 1, "huge_tie_group": 2, "negative_logits": 3}[case])
    B, V = 6, 60000
    if case == "above_window":
        x = rng.standard_normal((B, V)).astype(np.float32)
        for r in range(B):
            x[r, rng.choice(V, 4, replace=False)] = np.float32(60.0 + r)
        p = np.array([0.3, 0.5, 0.9, 0.99, 0.2, 0.7], np.float32)
    elif case == "huge_tie_group":
        x = (np.round(rng.standard_normal((B, V)) * 2) / 2).astype(np.float32)
        p = np.array([0.3, 0.5, 0.6, 0.7, 0.8, 0.95], np.float32)
    else:
        x = (rng.standard_normal((B, V)) - 40.0).astype(np.float32)
        p = np.array([0.5, 0.8, 0.9, 0.95, 0.99, 0.6], np.float32)
    logits = f32_to_bf16_bits(x)
    k = np.full(B, V, np.int32)
    for flags in (q.flag_cluster(1), q.flag_cluster(2)):
        fails, flagged, got, st, info = check_against_oracle(logits, "bf16", k, p, dev, flags=flags)
        assert fails == [], (case, flags, fails[:5])


def test_key_histogram_gives_way_on_wide_bf16_rows(dev):
    """A far outlier widens the survivors' key range beyond the histogram:
    those rows take the pivot rounds, with the same results."""
    import top_selection_row_gb300 as q
    from workloads import f32_to_bf16_bits

    rng = np.random.default_rng(17)
    B, V = 12, 50000
    x = rng.standard_normal((B, V)).astype(np.float32)
    x[:, 123] = np.float32(3e30)     # far above: tens of thousands of keys away
    x[::2, 4567] = np.float32(-1e25)
    logits = f32_to_bf16_bits(x)
    k = np.array([1, 2, 10, 100, 1000, 5000, 1, 50, 700, 3, 20000, 60], np.int32)
    p = np.array([1.0, 0.5, 0.9, 1.0, 0.99, 1.0, 0.3, 1.0, 0.95, 1.0, 0.7, 1.0], np.float32)
    fails, flagged, got, st, info = check_against_oracle(logits, "bf16", k, p, dev)
    assert fails == [], fails[:5]
    assert ((info["path"] & q.PATH_KEYHIST) == 0).all()


def test_first_pass_bins_place_flat_top_p_rows(dev):
    """Top-p rows whose survivors far exceed the lists (flat rows: high
    temperature) take their boundary's bins from the streaming pass, so one
    more pass extracts them and no narrowing pass runs."""
    import top_selection_row_gb300 as q

    w = WORKLOADS[3]
    logits, k, p = workload(3, 48)
    for flags in (0, q.flag_cluster(1), q.flag_cluster(8)):
        fails, flagged, got, st, info = check_against_oracle(logits, w.dtype, k, p, dev, flags=flags)
        assert fails == [], (flags, fails[:5])
        hist = (info["path"] & q.PATH_HIST) != 0
        assert hist.sum() >= 8, (flags, int(hist.sum()))
        assert (info["passes"][hist] == 1).all()


def test_sample_threshold_rescues_uniform_rows(dev):
    """Uniform rows defeat the Gaussian threshold (it lies above their max):
    the sample contradicts it, and an order statistic of the sample becomes
    the threshold, so the first pass keeps the candidates."""
    import top_selection_row_gb300 as q

    w = WORKLOADS[4]
    logits, k, p = workload(4, 64)
    x = widen(logits, w.dtype)
    uniform = np.abs(x).max(axis=1) <= 1.0
    assert uniform.any()
    fails, flagged, got, st, info = check_against_oracle(logits, w.dtype, k, p, dev)
    assert fails == [], fails[:5]
    path = info["path"][uniform]
    assert ((path & q.PATH_SAMPLE_T) != 0).mean() >= 0.75
    assert ((path & (q.PATH_FALLBACK | q.PATH_RETRY)) == 0).mean() >= 0.75


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_light_tails_take_the_sample_threshold_at_small_k(dev, dtype):
    """Small k on rows bounded below the Gaussian tail: the sample expects
    fewer than two values above the k-th logit, so it cannot test the
    Gaussian threshold itself; its tail lighter than the Gaussian's
    (hardly any value above mu + 2 sigma) sends the row to the sample's
    order statistic, not to a second pass. Gaussian rows keep their
    threshold."""
    import top_selection_row_gb300 as q

    rng = np.random.default_rng(41)
    B, V = 24, 201088
    x = rng.uniform(-1.0, 1.0, (B, V)).astype(np.float32)
    x[B // 2:] = rng.standard_normal((B - B // 2, V)).astype(np.float32)
    k = np.array([1, 2, 5, 20, 50, 97, 113, 200, 300, 1, 60, 150] * 2, np.int32)
    p = np.where(np.arange(B) % 3 == 0, np.float32(0.9), np.float32(1.0)).astype(np.float32)
    logits = f32_to_bf16_bits(x) if dtype == "bf16" else x
    fails, flagged, got, st, info = check_against_oracle(logits, dtype, k, p, dev)
    assert fails == [], fails[:5]
    path = info["path"].astype(np.int64)
    uni, gau = path[: B // 2], path[B // 2:]
    assert ((uni & q.PATH_SAMPLE_T) != 0).all(), [hex(v) for v in uni]
    assert ((uni & (q.PATH_RETRY | q.PATH_FALLBACK)) == 0).all(), [hex(v) for v in uni]
    assert ((gau & q.PATH_SAMPLE_T) == 0).all(), [hex(v) for v in gau]


def test_second_truncation_rescues_uniform_rows(dev):
    """With the first threshold forced to miss, the second truncation at an
    order statistic of a larger sample finds the uniform rows' candidates
    without a full-row search."""
    import top_selection_row_gb300 as q

    w = WORKLOADS[4]
    logits, k, p = workload(4, 64)
    x = widen(logits, w.dtype)
    uniform = np.abs(x).max(axis=1) <= 1.0
    assert uniform.any()
    fails, flagged, got, st, info = check_against_oracle(logits, w.dtype, k, p, dev, flags=q.FLAG_FORCE_RETRY)
    assert fails == [], fails[:5]
    path = info["path"][uniform]
    assert ((path & q.PATH_RETRY) != 0).all()
    assert ((path & q.PATH_FALLBACK) == 0).mean() >= 0.75


def test_deterministic_across_calls(dev):
    logits, k, p = workload(4, 32)
    first, _, _ = run_gpu(logits, "bf16", k, p, dev, row_info=False)
    for _ in range(4):
        again, _, _ = run_gpu(logits, "bf16", k, p, dev, row_info=False)
        assert np.array_equal(first, again)


# ---------------------------------------------------------------------------
# Stage diagnostics against CPU restatements
# ---------------------------------------------------------------------------
def test_row_info_matches_cpu_restatements(dev):
    import top_selection_row_gb300 as q

    for n in (2, 3, 4, 5):
        w = WORKLOADS[n]
        logits, k, p = workload(n, 16)
        got, st, info = run_gpu(logits, w.dtype, k, p, dev)
        ref = dict(select_batch(logits, w.dtype, k, p))
        for r in range(logits.shape[0]):
            x = widen(logits[r], w.dtype)
            rec = info[r]
            # |Z_t| is the count of logits >= t (A4), t the threshold used
            if rec["path"] & q.PATH_TRUNC:
                assert rec["survivors"] == int(np.count_nonzero(x >= np.float32(rec["threshold"])))
            # m is the row max
            assert rec["row_max"] == np.float32(x.max())
            # the sample statistics describe the row's values
            assert abs(rec["mu"] - x.mean()) < 0.5 * x.std() + 1e-3
            assert 0.2 * x.std() < rec["sigma"] < 5 * x.std()
            if not ref[r].ambiguous:
                assert rec["kept"] == ref[r].kept
                assert rec["boundary"] == np.float32(ref[r].boundary)
                assert rec["n_boundary"] == ref[r].n_boundary


def test_host_entry_point_matches_device_path(dev):
    import torch

    import top_selection_row_gb300 as q

    logits, k, p = workload(4, 12)
    xd = to_device(logits, "bf16", dev)
    want = q.qrita_select(xd, torch.from_numpy(k).to(dev), torch.from_numpy(p).to(dev))
    torch.cuda.synchronize()
    xh = xd.cpu().pin_memory()
    out = q.qrita_select_host(xh, torch.from_numpy(k), torch.from_numpy(p))
    assert torch.equal(out, want.cpu())


@pytest.mark.parametrize("n,rows", [(2, 64), (2, 13), (4, 3), (1, 4)])
def test_host_entry_sizes_match_device_path(dev, n, rows):
    """The host entry (copies in, selection, copy out) gives the device
    path's masks for batches of several sizes and row counts, call after call."""
    import torch

    import top_selection_row_gb300 as q

    w = WORKLOADS[n]
    logits, k, p = workload(n, rows)
    xd = to_device(logits, w.dtype, dev)
    want = q.qrita_select(xd, torch.from_numpy(k).to(dev), torch.from_numpy(p).to(dev))
    torch.cuda.synchronize()
    xh = xd.cpu().pin_memory()
    for _ in range(2):
        out = q.qrita_select_host(xh, torch.from_numpy(k), torch.from_numpy(p))
        assert torch.equal(out, want.cpu())


def test_runs_on_a_side_stream(dev):
    import torch

    import top_selection_row_gb300 as q

    logits, k, p = workload(2, 8)
    x = to_device(logits, "f32", dev)
    kd = torch.from_numpy(k).to(dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        m = q.qrita_select(x, kd)
    s.synchronize()
    ref = select_batch(logits, "f32", k, None)
    fails, _ = compare_rows(m.cpu().numpy().astype(np.uint8), np.zeros(8, np.int32), ref)
    assert fails == []
