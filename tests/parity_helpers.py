"""Shared helpers of the GPU parity tests: run the C-ABI path, compare with
the oracle row by row under the documented pass rule."""

from __future__ import annotations

import numpy as np

from oracle import accepts, select_batch
from oracle.qrita_oracle import STATUS_NONFINITE


def to_device(logits: np.ndarray, dtype: str, dev):
    import torch

    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(dev)
    bits = np.ascontiguousarray(logits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(bits).to(dev).view(torch.bfloat16)


def run_gpu(logits, dtype, k, p, dev, flags=0, row_info=True):
    """qrita_select_ex through the C ABI; returns (mask uint8, status, info)."""
    import torch

    import top_selection_row_gb300 as q

    x = to_device(logits, dtype, dev)
    kd = None if k is None else torch.from_numpy(np.asarray(k, np.int32)).to(dev)
    pd = None if p is None else torch.from_numpy(np.asarray(p, np.float32)).to(dev)
    mask, st, info = q.qrita_select_ex(x, kd, pd, flags=flags, row_status=True, row_info=row_info)
    torch.cuda.synchronize()
    infos = q.decode_row_info(info) if row_info else None
    return mask.cpu().numpy().astype(np.uint8), st.cpu().numpy(), infos


def compare_rows(got_mask, got_status, oracle_rows):
    """Pass rule: top-k and unflagged top-p rows bit-exact; flagged rows may be
    the oracle's prefix or one token shorter / longer. Returns failures and
    the flagged-row count."""
    fails = []
    flagged = 0
    for r, res in oracle_rows:
        g = got_mask[r]
        if res.status == STATUS_NONFINITE:
            if g.any() or got_status[r] != 1:
                fails.append((r, "nonfinite row"))
            continue
        if got_status[r] != 0:
            fails.append((r, f"status {got_status[r]}"))
            continue
        if res.ambiguous:
            flagged += 1
            if not accepts(res, g):
                fails.append((r, "flagged row outside the band", int(g.sum()), res.kept, res.band_kept))
        elif not np.array_equal(g, res.mask):
            diff = np.nonzero(g != res.mask)[0]
            fails.append((r, "mismatch", int(g.sum()), res.kept, diff[:8].tolist()))
    return fails, flagged


def check_against_oracle(logits, dtype, k, p, dev, flags=0, rows=None):
    got, st, info = run_gpu(logits, dtype, k, p, dev, flags=flags)
    ref = select_batch(logits, dtype, k, p, rows=rows)
    fails, flagged = compare_rows(got, st, ref)
    return fails, flagged, got, st, info


def widen(logits, dtype):
    if dtype == "f32":
        return np.asarray(logits, np.float64)
    return (logits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def invariant_failures(x64: np.ndarray, mask: np.ndarray, k, p):
    """Invariants every valid row's mask must satisfy, at any size.

    At least one token kept; with top-p off exactly min(k, V) kept (k on) or
    V kept; min(kept) >= max(dropped); among tokens equal to the boundary the
    kept ids precede the dropped ids; top-p kept is within the top-k count.
    """
    V = x64.shape[0]
    kept = np.nonzero(mask)[0]
    fails = []
    k_on = k is not None and 1 <= k < V
    p_on = p is not None and not np.isnan(p) and p < 1.0
    if p_on and p <= 0:
        p_on = False
        k_on = V > 1
        k = 1
    if kept.size == 0:
        return ["nothing kept"]
    if not p_on:
        want = k if k_on else V
        if kept.size != want:
            fails.append(f"kept {kept.size} != {want}")
    elif k_on and kept.size > k:
        fails.append(f"top-p kept {kept.size} > k {k}")
    dropped_mask = mask == 0
    if dropped_mask.any():
        lo = x64[kept].min()
        hi = x64[dropped_mask].max()
        if lo < hi:
            fails.append(f"min kept {lo} < max dropped {hi}")
        if lo == hi:
            tie = x64 == lo
            kt = np.nonzero(tie & (mask == 1))[0]
            dt = np.nonzero(tie & dropped_mask)[0]
            if kt.size and dt.size and kt.max() > dt.min():
                fails.append("boundary ties not kept by lowest id")
    return fails
