"""GPU parity of the outputs beyond the mask, through the C ABI, against the
output oracle (oracle/qrita_outputs.py): top-k ids in stable order (exact),
candidate lists (ids and counts exact, probabilities within 4e-6 relative),
and draws by inverse CDF (exact unless the oracle flags the uniform as lying
within 1e-6 of a cumulative boundary)."""

import numpy as np
import pytest

from oracle import candidates, sample, select_batch, topk_ids
from parity_helpers import to_device, widen
from workloads import WORKLOADS, f32_to_bf16_bits, generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_selection_row_gb300 as q

    q.lib()
    return torch.device("cuda", 0)


def _ids_case(dev, logits, dtype, k, kmax):
    import torch

    import top_selection_row_gb300 as q

    x = to_device(logits, dtype, dev)
    ids, mask = q.qrita_topk_ids(x, torch.from_numpy(np.asarray(k, np.int32)).to(dev), kmax)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    mask = mask.cpu().numpy().astype(np.uint8)
    ref_mask = select_batch(logits, dtype, k, None)
    for r in range(logits.shape[0]):
        xr = widen(logits[r], dtype)
        kr = int(k[r])
        want = topk_ids(xr, kr) if 1 <= kr <= kmax else []
        got = ids[r][ids[r] >= 0].tolist()
        assert got == want, (r, kr, got[:8], want[:8])
        assert (ids[r][len(want):] == -1).all()
        assert np.array_equal(mask[r], ref_mask[r][1].mask), r


@pytest.mark.parametrize("n,kmax", [(1, 64), (2, 1024), (4, 4096), (5, 2048)])
def test_topk_ids_on_workload_rows(dev, n, kmax):
    w = WORKLOADS[n]
    logits, k, _ = generate(n, rows=min(w.B, 16))
    k = np.where(k >= w.V, kmax, np.minimum(k, kmax)).astype(np.int32)
    _ids_case(dev, logits, w.dtype, k, kmax)


def test_topk_ids_edges(dev):
    rng = np.random.default_rng(11)
    V = 3000
    base = np.round(rng.standard_normal((8, V)) * 2) / 4  # many ties
    x = base.astype(np.float32)
    x[5, 17] = np.nan
    x[6, :] = 1.5  # every logit equal: ids in id order
    x[7, ::2] = -np.inf
    k = np.array([1, 7, 300, 0, -4, 10, 500, 2999], np.int32)
    _ids_case(dev, x, "f32", k, 512)
    _ids_case(dev, f32_to_bf16_bits(x), "bf16", k, 512)
    # k above kmax: no ids; tiny rows with k >= V: every id
    _ids_case(dev, x[:2, :5].copy(), "f32", np.array([9, 5], np.int32), 8)
    _ids_case(dev, x[:3], "f32", np.array([600, 1, 512], np.int32), 512)


def _cand_case(dev, logits, dtype, mask, cap, us):
    import torch

    import top_selection_row_gb300 as q

    x = to_device(logits, dtype, dev)
    m = torch.from_numpy(np.ascontiguousarray(mask, np.uint8)).to(dev)
    ud = torch.from_numpy(np.asarray(us, np.float32)).to(dev)
    ids, probs, count, smp = q.qrita_candidates(x, m, cap, u=ud)
    torch.cuda.synchronize()
    ids, probs, count, smp = ids.cpu().numpy(), probs.cpu().numpy(), count.cpu().numpy(), smp.cpu().numpy()
    flagged = 0
    for r in range(logits.shape[0]):
        xr = widen(logits[r], dtype)
        want_ids, want_p = candidates(xr, mask[r])
        assert count[r] == want_ids.size, r
        nw = min(cap, want_ids.size)
        assert np.array_equal(ids[r][:nw], want_ids[:nw]), r
        got_p = probs[r][:nw].astype(np.float64)
        assert np.all(np.abs(got_p - want_p[:nw]) <= 4e-6 * want_p[:nw] + 1e-30), (r, np.abs(got_p - want_p[:nw]).max())
        tok, amb = sample(xr, mask[r], float(np.float32(us[r])))
        if amb:
            flagged += 1
        else:
            assert smp[r] == tok, (r, smp[r], tok, us[r])
    return flagged


@pytest.mark.parametrize("n", [1, 3, 4, 5])
def test_candidates_and_draws_on_workload_masks(dev, n):
    import torch

    import top_selection_row_gb300 as q

    w = WORKLOADS[n]
    logits, k, p = generate(n, rows=min(w.B, 12))
    x = to_device(logits, w.dtype, dev)
    mask = q.qrita_select(x, torch.from_numpy(k).to(dev), torch.from_numpy(p).to(dev)).cpu().numpy().astype(np.uint8)
    rng = np.random.default_rng(100 + n)
    us = rng.random(logits.shape[0]).astype(np.float32)
    us[0] = 0.0
    us[-1] = np.float32(0.99999994)
    cap = int(mask.sum(axis=1).max())
    # (rows keeping ~1e5 tokens hold a cumulative boundary every ~1e-5, so
    # the 1e-6 band flags a fair share of their draws; the others are exact)
    assert _cand_case(dev, logits, w.dtype, mask, cap, us) <= logits.shape[0] // 2
    # a short cap: the first ids in id order, the full count, the same draws
    _cand_case(dev, logits, w.dtype, mask, 5, us)


def test_candidates_edges(dev):
    rng = np.random.default_rng(12)
    V = 2000
    x = rng.standard_normal((6, V)).astype(np.float32) * 3
    mask = (rng.random((6, V)) < 0.3).astype(np.uint8)
    mask[1] = 0  # nothing kept
    mask[2] = 0
    mask[2, 1234] = 1  # one token
    x[3, :] = -np.inf  # every kept logit -inf: equal probabilities
    x[4, ::3] = 80.0  # huge logits
    us = np.array([0.5, 0.5, 0.9, 0.25, 0.1, 0.0], np.float32)
    _cand_case(dev, x, "f32", mask, V, us)
    _cand_case(dev, f32_to_bf16_bits(x), "bf16", mask, 64, us)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_vector_and_scalar_forms(dev, dtype):
    """Rows whose mask and logits start on 16-byte boundaries (V a multiple of
    16) take the vector kernels; the same rows with V off by a few elements,
    or shifted one element off the boundary, take the scalar ones. Both must
    match the oracle."""
    import torch

    import top_selection_row_gb300 as q

    rng = np.random.default_rng(17)
    for V in (4096, 4099, 5008):
        x = (np.round(rng.standard_normal((6, V)) * 8) / 8).astype(np.float32)  # ties
        x[2, :] = 0.75
        logits = f32_to_bf16_bits(x) if dtype == "bf16" else x
        k = np.array([1, 33, 700, 4096, 0, 2047], np.int32)
        _ids_case(dev, logits, dtype, k, 4096)
        mask = (rng.random((6, V)) < np.array([0.002, 0.05, 0.5, 1.0, 0.0, 0.9])[:, None]).astype(np.uint8)
        us = rng.random(6).astype(np.float32)
        _cand_case(dev, logits, dtype, mask, V, us)
        _cand_case(dev, logits, dtype, mask, 40, us)
        # one element off the 16-byte boundary: the logits and the mask live
        # at offset 1 of larger buffers
        xd = to_device(logits, dtype, dev).reshape(-1)
        xs = torch.empty(xd.numel() + 8, dtype=xd.dtype, device=dev)
        xs[1:1 + xd.numel()] = xd
        xo = xs[1:1 + xd.numel()].view(6, V)
        ms = torch.zeros(6 * V + 16, dtype=torch.uint8, device=dev)
        ms[1:1 + 6 * V] = torch.from_numpy(mask.reshape(-1)).to(dev)
        mo = ms[1:1 + 6 * V].view(6, V)
        ud = torch.from_numpy(us).to(dev)
        ids_o, probs_o, count_o, smp_o = q.qrita_candidates(xo, mo, V, u=ud)
        ids_a, probs_a, count_a, smp_a = q.qrita_candidates(to_device(logits, dtype, dev),
                                                            torch.from_numpy(mask).to(dev), V, u=ud)
        assert torch.equal(count_o, count_a) and torch.equal(ids_o, ids_a) and torch.equal(smp_o, smp_a)
        assert torch.allclose(probs_o, probs_a, rtol=4e-6, atol=0)
        kd = torch.from_numpy(k).to(dev)
        tid_o, _ = q.qrita_topk_ids(xo, kd, 4096)
        tid_a, _ = q.qrita_topk_ids(to_device(logits, dtype, dev), kd, 4096)
        assert torch.equal(tid_o, tid_a)


def test_draws_follow_the_probabilities(dev):
    """Stratified uniforms over one row: each kept id is drawn in proportion
    to its probability (the draw is the inverse distribution function)."""
    import torch

    import top_selection_row_gb300 as q

    rng = np.random.default_rng(13)
    V, N = 500, 4000
    row = (rng.standard_normal(V) * 1.5).astype(np.float32)
    mask1 = (rng.random(V) < 0.2).astype(np.uint8)
    logits = np.repeat(row[None, :], N, axis=0)
    mask = np.repeat(mask1[None, :], N, axis=0)
    us = ((np.arange(N) + 0.5) / N).astype(np.float32)
    x = torch.from_numpy(logits).to(dev)
    _, _, _, smp = q.qrita_candidates(x, torch.from_numpy(mask).to(dev), 1, u=torch.from_numpy(us).to(dev))
    smp = smp.cpu().numpy()
    ids, probs = candidates(row.astype(np.float64), mask1)
    freq = np.array([(smp == i).sum() for i in ids]) / N
    assert np.abs(freq - probs).max() <= 1.5 / N
