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
    kept ids precede the dropped ids; top-p kept is within the top-k count;
    with top-p on, the kept mass reaches p of the top-k set's mass and
    dropping the last-ranked kept token falls below p (both within the
    1e-6 * p band). The top-k set's mass needs no sort: equal logits weigh
    the same, so it is the mass of the k largest values, whichever
    duplicates they are.
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
    if p_on and not fails:
        m = x64.max()
        with np.errstate(invalid="ignore", over="ignore"):
            def wts(v):
                return np.where(v == m, 1.0, np.exp(v - m))

            top = np.partition(x64, V - k)[V - k:] if k_on else x64
            z_k = wts(top).sum()
            kept_w = wts(x64[kept])
        mass = kept_w.sum()
        band = 1e-6 * p
        if mass / z_k < p - band:
            fails.append(f"kept mass {mass / z_k!r} below p {p!r}")
        if kept.size > 1 and (mass - kept_w.min()) / z_k >= p + band:
            fails.append(f"mass without the last kept token {(mass - kept_w.min()) / z_k!r} still reaches p {p!r}")
    return fails


# ---------------------------------------------------------------------------
# Every row of a large batch against the oracle, on the host cores
# ---------------------------------------------------------------------------
def _attach(name, shape, dtype):
    from multiprocessing import resource_tracker, shared_memory

    shm = shared_memory.SharedMemory(name=name)
    # the creating process owns (and unlinks) the block; a worker only reads
    try:
        resource_tracker.unregister(shm._name, "shared_memory")
    except Exception:
        pass
    return shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf)


def _pooled_worker(job):
    """One worker's rows: the oracle's pass rule and the invariants."""
    lname, lshape, ldtype, mname, mshape, dtype, k, p, st, rows = job
    shm_l, logits = _attach(lname, lshape, ldtype)
    shm_m, masks = _attach(mname, mshape, np.uint8)
    try:
        fails, flagged, bad = [], 0, []
        for r in rows:
            ref = select_batch(logits[r:r + 1], dtype, None if k is None else k[r:r + 1],
                               None if p is None else p[r:r + 1])
            f, fl = compare_rows(masks[r:r + 1], st[r:r + 1], ref)
            fails += [(r,) + tuple(x[1:]) for x in f]
            flagged += fl
            if st[r] == 0 and ref[0][1].status == 0:
                inv = invariant_failures(widen(logits[r], dtype), masks[r],
                                         None if k is None else int(k[r]), None if p is None else float(p[r]))
                if inv:
                    bad.append((r, inv))
        return fails, flagged, bad
    finally:
        del logits, masks
        shm_l.close()
        shm_m.close()


def compare_rows_pooled(logits, dtype, k, p, got, st, workers=None):
    """Every row of a batch against the oracle (pass rule of compare_rows) and
    the invariants, spread over spawned worker processes (one per host core,
    16 at most). The logits and the masks reach the workers through shared
    memory. Returns (failures, flagged rows, invariant failures)."""
    import multiprocessing as mp
    import os
    from multiprocessing import shared_memory

    logits = np.ascontiguousarray(logits)
    got = np.ascontiguousarray(got, dtype=np.uint8)
    B = logits.shape[0]
    if workers is None:
        try:
            workers = len(os.sched_getaffinity(0))
        except AttributeError:
            workers = os.cpu_count() or 1
    workers = max(1, min(16, workers, B))
    shm_l = shared_memory.SharedMemory(create=True, size=max(1, logits.nbytes))
    shm_m = shared_memory.SharedMemory(create=True, size=max(1, got.nbytes))
    try:
        np.ndarray(logits.shape, logits.dtype, buffer=shm_l.buf)[...] = logits
        np.ndarray(got.shape, np.uint8, buffer=shm_m.buf)[...] = got
        kk = None if k is None else np.asarray(k, np.int32)
        pp = None if p is None else np.asarray(p, np.float32)
        ss = np.asarray(st, np.int32)
        jobs = [(shm_l.name, logits.shape, logits.dtype.str, shm_m.name, got.shape, dtype, kk, pp, ss,
                 list(range(i, B, workers))) for i in range(workers)]
        # spawned, never forked: the parent has a CUDA context
        with mp.get_context("spawn").Pool(workers) as pool:
            res = pool.map(_pooled_worker, jobs)
    finally:
        shm_l.close()
        shm_l.unlink()
        shm_m.close()
        shm_m.unlink()
    fails = sorted((f for r in res for f in r[0]), key=lambda t: t[0])
    flagged = sum(r[1] for r in res)
    bad = sorted((b for r in res for b in r[2]), key=lambda t: t[0])
    return fails, flagged, bad
