"""Throughput of exact top-k / top-p selection on GB300: rows/s and HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..5] [--no-sweep]

One step is one call of the whole selection pipeline (sample statistics,
sigma-truncation, quaternary top-k / top-p pivot search, tie resolution,
mask emission) over one batch of the workload. The headline workload is the
largest one: 1024 x 262144 bf16 logits with mixed per-row top-k / top-p
(workload 5); the JSON line also carries every workload's own number under
"per_workload", with the count of rows each path of the kernel took (from
the per-row diagnostics of one untimed call) and the oracle's count of
flagged top-p rows (tests/golden/flagged_counts.json, written from the
oracle alone by tests/golden/make_flagged_counts.py).

Timing: W untimed steps, then exactly K steps bracketed by a barrier and a
device synchronize, timed with CUDA events on the launching stream; inputs
rotate over enough copies that the rotating set exceeds 3x the L2 size, so
no step reads logits from L2. For N > 1 (torchrun) every rank processes its
own batch (weak scaling; rows are independent, there is no collective on
the data path) and the slowest rank's time is reported.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import WORKLOADS, assumptions, generate  # noqa: E402

METRIC = "logit rows/sec and HBM GB/s (% of GB300 peak) for exact top-k/top-p masking"
HEADLINE = 5
KERNEL_SOURCES = [
    os.path.join(ROOT, "top_selection_row_gb300", "csrc", f)
    for f in ("qrita_kernel.cu", "qrita_device.cuh", "qrita_internal.h", "qrita_api.cpp")
]


# ---------------------------------------------------------------------------
# distributed plumbing (tested on CPU with gloo)
# ---------------------------------------------------------------------------
def dist_env():
    """(rank, world, local_rank) from torchrun's environment; (0, 1, 0) alone."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate_rows_per_s(rows_per_rank: int, world: int, seconds_max: float) -> float:
    """Whole-job throughput: every rank's rows over the slowest rank's time."""
    return rows_per_rank * world / seconds_max


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_number: int):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    w = d.get("workloads", {}).get(str(workload_number))
    return None if w is None else w.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            # the raw samples go to QRITA_CLOCKS_DIR when set (kept for
            # inspection), else to the temp directory
            out_dir = os.environ.get("QRITA_CLOCKS_DIR") or tempfile.gettempdir()
            os.makedirs(out_dir, exist_ok=True)
            self.path = os.path.join(out_dir, f"clocks_{os.getpid()}.csv")
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": float(np.median(sms)), "sm_max_mhz": float(max(maxes)),
                "reasons": sorted(reasons), "samples": len(sms)}


def oracle_flagged_counts():
    """Per-workload top-p rows and the oracle's flagged rows, as stored by
    tests/golden/make_flagged_counts.py (None when the file is missing)."""
    path = os.path.join(ROOT, "tests", "golden", "flagged_counts.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        return json.load(f).get("workloads")


PATH_BITS = {
    "top_k": 0x1, "top_p": 0x2, "truncated": 0x4, "hit": 0x8, "fallback": 0x10, "overflow": 0x20,
    "keep_all": 0x40, "retry": 0x80, "hist": 0x100, "sample_threshold": 0x200, "key_histogram": 0x400,
}


def path_counts(info) -> dict:
    """Rows per path bit of qrita_row_info_t.path, plus rows that searched
    their truncation survivors (hit, retry or hist without the fallback)."""
    path = info["path"].astype(np.int64)
    out = {name: int(((path & bit) != 0).sum()) for name, bit in PATH_BITS.items()}
    searched = (path & (0x8 | 0x80 | 0x100 | 0x400)) != 0
    out["searched_survivors"] = int((searched & ((path & 0x10) == 0)).sum())
    out["narrowing_passes_total"] = int(info["passes"].astype(np.int64).sum())
    return out


def workload_config(w, n_rot, l2_bytes):
    return {
        "workload": w.name,
        "global_batch": w.B,
        "vocab": w.V,
        "logits_dtype": w.dtype,
        "seed": 1000 + w.number,
        "assumptions": assumptions(w.number),
        "l2_defeat": f"inputs rotate over {n_rot} copies "
                     f"({n_rot * w.B * w.V * (w.elem_bytes + 1) / 1e6:.0f} MB > 3 x L2 {l2_bytes / 1e6:.0f} MB)",
    }


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def time_workload(number, steps, warmup, dev, world, l2_bytes, stream, rotate=None):
    """Device timing of one workload; returns a dict of numbers. ``rotate``
    overrides the number of rotating input copies (profiling runs use 1)."""
    import torch

    import top_selection_row_gb300 as q

    w = WORKLOADS[number]
    logits, k, p = generate(number)
    bytes_in = w.B * w.V * (w.elem_bytes + 1)
    n_rot = max(1, math.ceil(3 * l2_bytes / bytes_in) + 1) if rotate is None else rotate
    if w.dtype == "f32":
        x0 = torch.from_numpy(logits).to(dev)
    else:
        x0 = torch.from_numpy(logits.view(np.int16)).to(dev).view(torch.bfloat16)
    xs = [x0] + [x0.clone() for _ in range(n_rot - 1)]
    outs = [torch.empty((w.B, w.V), dtype=torch.bool, device=dev) for _ in range(n_rot)]
    kd = torch.from_numpy(k).to(dev)
    pd = torch.from_numpy(p).to(dev)
    k_arg = kd if w.number != 3 else kd  # k = V rows: top-k off per row
    p_arg = pd
    torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            q.qrita_select(xs[i % n_rot], k_arg, p_arg, out=outs[i % n_rot], stream=stream)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # the timed region: K back-to-back calls, one kernel each, nothing between
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            j = (warmup + i) % n_rot
            q.qrita_select(xs[j], k_arg, p_arg, out=outs[j], stream=stream)
        end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    total_ms = start.elapsed_time(end)
    total_s = max_over_ranks(total_ms / 1e3, world, dev)
    # each launch on its own between events (diagnostic: no overlap with its
    # neighbours)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            j = (warmup + i) % n_rot
            ev[i][0].record(stream)
            q.qrita_select(xs[j], k_arg, p_arg, out=outs[j], stream=stream)
            ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    # the same K calls captured once in a CUDA graph and replayed
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(steps):
                j = (warmup + i) % n_rot
                q.qrita_select(xs[j], k_arg, p_arg, out=outs[j], stream=stream)
        g.replay()
        torch.cuda.synchronize(dev)
        gs = torch.cuda.Event(enable_timing=True)
        ge = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            gs.record(stream)
            g.replay()
            ge.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = gs.elapsed_time(ge) / steps
        del g
    except Exception as e:  # capture is optional: report why it is missing
        print(f"bench: CUDA-graph timing skipped ({type(e).__name__}: {e})", file=sys.stderr)
        torch.cuda.synchronize(dev)
    # one untimed call with the per-row diagnostics: rows per path
    with torch.cuda.stream(stream):
        _, _, info = q.qrita_select_ex(xs[0], k_arg, p_arg, out=outs[0], stream=stream, row_info=True)
    torch.cuda.synchronize(dev)
    paths = path_counts(q.decode_row_info(info))
    del xs, outs
    return {
        "paths": paths,
        "w": w,
        "n_rot": n_rot,
        "ms_per_step": total_s * 1e3 / steps,
        "rows_per_s": aggregate_rows_per_s(w.B * steps, world, total_s),
        "kernel_ms_mean": total_s * 1e3 / steps,
        "kernel_ms_isolated_median": float(np.median(per_launch_ms)),
        "graph_ms_per_step": graph_ms,
        "bytes_per_launch": w.B * w.bytes_per_row,
        "launches": steps,
    }


def sort_mask(x, kd, pd):
    """The sort-based comparator the pages measure against (Qrita summary,
    "Problem statement" and "Results"): a stable descending sort of each row,
    the top-k prefix, softmax and cumulative sum over it, the first prefix
    reaching p, scattered back into a keep-mask. Plain PyTorch on the GPU,
    in fp32: a timing and memory comparator, not an exact reference."""
    import torch

    xf = x.float()
    B, V = xf.shape
    vals, idx = torch.sort(xf, dim=1, descending=True, stable=True)
    pos = torch.arange(V, device=xf.device).unsqueeze(0)
    k_on = ((kd >= 1) & (kd < V)).unsqueeze(1)
    keep = torch.where(k_on, pos < kd.unsqueeze(1), torch.ones_like(pos, dtype=torch.bool))
    p_on = (pd < 1.0).unsqueeze(1)
    wts = torch.exp(vals - vals[:, :1]) * keep
    z = wts.sum(dim=1, keepdim=True)
    before = (torch.cumsum(wts, dim=1) - wts) / z  # mass of the tokens ranked before
    keep = keep & torch.where(p_on, (before < pd.unsqueeze(1)) | (pos == 0), torch.ones_like(keep))
    return torch.zeros_like(keep).scatter_(1, idx, keep)


def time_sort_baseline(number, steps, warmup, dev, stream):
    """Time and peak extra device memory of the sort-based comparator on the
    workload, beside the library's (which allocates nothing)."""
    import torch

    w = WORKLOADS[number]
    logits, k, p = generate(number)
    if w.dtype == "f32":
        x = torch.from_numpy(logits).to(dev)
    else:
        x = torch.from_numpy(logits.view(np.int16)).to(dev).view(torch.bfloat16)
    kd = torch.from_numpy(k).to(dev)
    pd = torch.from_numpy(p).to(dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            sort_mask(x, kd, pd)
    torch.cuda.synchronize(dev)
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s.record(stream)
        for _ in range(steps):
            sort_mask(x, kd, pd)
        e.record(stream)
    torch.cuda.synchronize(dev)
    peak = torch.cuda.max_memory_allocated(dev) - base
    ms = s.elapsed_time(e) / steps
    del x, kd, pd
    return {
        "impl": "torch.sort(stable=True) + softmax/cumsum over the sorted row + scatter (fp32, PyTorch on the GPU)",
        "workload": w.name,
        "ms_per_step": ms,
        "rows_per_s": w.B / (ms / 1e3),
        "peak_extra_device_bytes": int(peak),
        "ours_extra_device_bytes": 0,
        "note": "the library allocates nothing per call; the comparator's bytes are its sort and scan temporaries",
    }


def time_outputs(number, steps, warmup, dev, stream, peak, kmax=2048, cap=2048):
    """The outputs after the mask on the workload, inputs resident: the top-k
    ids in rank order (qrita_topk_ids: the selection with top-p off, then the
    ids kernel) beside the selection alone, and the candidate lists with one
    draw per row (qrita_candidates over the workload's mask). Algorithmic
    bytes: ids: the mask read, the kept logits and the id rows written;
    candidates: the mask read, the kept logits, the ids and probabilities
    written (up to cap per row), the count, the uniform and the draw."""
    import torch

    import top_selection_row_gb300 as q

    w = WORKLOADS[number]
    logits, k, p = generate(number)
    if w.dtype == "f32":
        x = torch.from_numpy(logits).to(dev)
    else:
        x = torch.from_numpy(logits.view(np.int16)).to(dev).view(torch.bfloat16)
    kd = torch.from_numpy(k).to(dev)
    pd = torch.from_numpy(p).to(dev)
    mask = q.qrita_select(x, kd, pd, stream=stream)
    torch.cuda.synchronize(dev)
    kept = mask.sum(dim=1).cpu().numpy().astype(np.int64)
    rng = np.random.default_rng(7)
    ud = torch.from_numpy(rng.random(w.B).astype(np.float32)).to(dev)
    ids = torch.empty((w.B, cap), dtype=torch.int32, device=dev)
    probs = torch.empty((w.B, cap), dtype=torch.float32, device=dev)
    count = torch.empty(w.B, dtype=torch.int32, device=dev)
    sample = torch.empty(w.B, dtype=torch.int32, device=dev)
    kmask = torch.empty((w.B, w.V), dtype=torch.bool, device=dev)
    kids = torch.empty((w.B, kmax), dtype=torch.int32, device=dev)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize(dev)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s.record(stream)
            for _ in range(steps):
                fn()
            e.record(stream)
        torch.cuda.synchronize(dev)
        return s.elapsed_time(e) / steps

    cand_ms = timed(lambda: q.qrita_candidates(x, mask, cap, u=ud, stream=stream, out=(ids, probs, count, sample)))
    ids_ms = timed(lambda: q.qrita_topk_ids(x, kd, kmax, out_mask=kmask, out_ids=kids, stream=stream))
    sel_k_ms = timed(lambda: q.qrita_select(x, kd, None, out=kmask, stream=stream))
    kk = np.where((k >= 1) & (k <= kmax), np.minimum(k, w.V), 0).astype(np.int64)
    ids_bytes = int(w.B * w.V + kk.sum() * w.elem_bytes + w.B * kmax * 4)
    cand_bytes = int(w.B * w.V + kept.sum() * w.elem_bytes + np.minimum(kept, cap).sum() * 8 + w.B * 12)
    ids_extra = max(ids_ms - sel_k_ms, 1e-9)
    del x, mask, kmask
    return {
        "workload": w.name,
        "candidates": {
            "call": "qrita_candidates (cap %d, one draw per row)" % cap,
            "ms_per_call": cand_ms,
            "rows_per_s": w.B / (cand_ms / 1e3),
            "algorithmic_bytes": cand_bytes,
            "hbm_gbs": cand_bytes / (cand_ms / 1e3) / 1e9,
            "frac_of_measured_peak": cand_bytes / (cand_ms / 1e3) / 1e9 / peak,
            "kept_per_row_mean": float(kept.mean()),
        },
        "topk_ids": {
            "call": "qrita_topk_ids (kmax %d): the selection with top-p off, then the ids" % kmax,
            "ms_per_call": ids_ms,
            "rows_per_s": w.B / (ids_ms / 1e3),
            "selection_alone_ms": sel_k_ms,
            "ids_kernel_ms_estimate": ids_extra,
            "ids_algorithmic_bytes": ids_bytes,
            "ids_frac_of_measured_peak": ids_bytes / (ids_extra / 1e3) / 1e9 / peak,
            "rows_with_ids": int((kk > 0).sum()),
        },
    }


def time_e2e(number, steps, warmup, dev, stream):
    """End to end through qrita_select_host: pinned host logits / k / p in,
    host mask out, copies inside the timed region."""
    import torch

    import top_selection_row_gb300 as q

    w = WORKLOADS[number]
    logits, k, p = generate(number)
    if w.dtype == "f32":
        xh = torch.from_numpy(logits).pin_memory()
    else:
        xh = torch.from_numpy(logits.view(np.int16)).view(torch.bfloat16).pin_memory()
    kh = torch.from_numpy(k).pin_memory()
    ph = torch.from_numpy(p).pin_memory()
    out = torch.empty((w.B, w.V), dtype=torch.bool).pin_memory()
    staging = torch.empty(q.host_staging_bytes(q.DTYPE_F32 if w.dtype == "f32" else q.DTYPE_BF16, w.B, w.V),
                          dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        q.qrita_select_host(xh, kh, ph, out=out, staging=staging, stream=stream)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        q.qrita_select_host(xh, kh, ph, out=out, staging=staging, stream=stream)
    dt = time.perf_counter() - t0
    return {
        "value": w.B * steps / dt,
        "unit": "rows/s",
        "h2d_bytes_per_step": w.B * w.V * w.elem_bytes + 8 * w.B,
        "d2h_bytes_per_step": w.B * w.V,
    }


def oracle_rows_per_s(number, budget_s=10.0, max_rows=None, data=None):
    """The CPU oracle as it stands, on a bounded sample of the workload's rows
    (rows taken in order, cycling). ``data`` = (logits, k, p) if already made."""
    from oracle import select_batch

    w = WORKLOADS[number]
    logits, k, p = data if data is not None else generate(number)
    done = 0
    t0 = time.perf_counter()
    while True:
        r = done % w.B
        select_batch(logits[r : r + 1], w.dtype, k[r : r + 1], p[r : r + 1])
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_rows is not None and done >= max_rows):
            break
    return done / el, done, el


def _oracle_worker(job):
    """One process of the pooled oracle timing: rows first, first + stride, ..."""
    number, first, stride, budget_s = job
    from oracle import select_batch

    w = WORKLOADS[number]
    logits, k, p = generate(number)
    done = 0
    t0 = time.perf_counter()
    r = first
    while True:
        select_batch(logits[r : r + 1], w.dtype, k[r : r + 1], p[r : r + 1])
        done += 1
        r = (r + stride) % w.B
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done, el


def oracle_rows_per_s_pooled(number, budget_s=10.0):
    """The oracle on every host core: one process per core (spawned), each on
    its own rows for about budget_s; returns (rows/s, rows, cores)."""
    import multiprocessing as mp

    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(number, i, cores, budget_s) for i in range(cores)])
    rows = sum(d for d, _ in res)
    el = max(e for _, e in res)
    return rows / el, rows, cores


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    import top_selection_row_gb300 as q

    q.lib()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 1024 * 1024)
    stream = torch.cuda.Stream(dev)
    peak, peak_kind = measured_peaks()

    per = {}
    numbers = [args.workload] + ([n for n in WORKLOADS if n != args.workload] if not args.no_sweep else [])
    for n in numbers:
        steps = args.steps if n == args.workload else max(10, min(args.steps, 30))
        warm = args.warmup if n == args.workload else 3
        if n == args.workload:
            with ClockSampler(local) as cs:
                res = time_workload(n, steps, warm, dev, world, l2, stream, args.rotate)
            res["clocks"] = cs.summary()
        else:
            res = time_workload(n, steps, warm, dev, world, l2, stream, args.rotate)
        per[n] = res

    head = per[args.workload]
    w = head["w"]
    achieved = head["bytes_per_launch"] / (head["kernel_ms_mean"] / 1e3) / 1e9
    traffic = ncu_traffic(args.workload)
    line = {
        "metric": METRIC,
        "value": head["rows_per_s"],
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded; shapes of the pages' workloads, no dataset)",
        "config": dict(workload_config(w, head["n_rot"], l2), parallelism=f"rows, {world} GPU(s), no collective"),
        "hbm_gbs": achieved,
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json copy bandwidth)",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": head["bytes_per_launch"],
            "kernel_ms_mean": head["kernel_ms_mean"],
            "kernel_ms_note": "mean launch duration over the timed region (K back-to-back launches / K)",
            "kernel_ms_isolated_median": head["kernel_ms_isolated_median"],
            "graph_ms_per_step": head["graph_ms_per_step"],
        },
        "gpu_launches": head["launches"],
        "clocks": head.get("clocks"),
        "per_workload": {},
    }
    flagged = oracle_flagged_counts() or {}
    for n, r in per.items():
        ach = r["bytes_per_launch"] / (r["kernel_ms_mean"] / 1e3) / 1e9
        gms = r["graph_ms_per_step"]
        line["per_workload"][WORKLOADS[n].name] = {
            "paths": r["paths"],
            "oracle_flagged": flagged.get(WORKLOADS[n].name),
            "rows_per_s": r["rows_per_s"],
            "ms_per_step": r["ms_per_step"],
            "kernel_ms_isolated_median": r["kernel_ms_isolated_median"],
            "hbm_gbs": ach,
            "frac_of_measured_peak": ach / peak,
            "frac_of_8tbs_nominal": ach / 8000.0,
            "graph_ms_per_step": gms,
            "graph_rows_per_s": (r["w"].B / (gms / 1e3)) if gms else None,
        }
    if rank == 0:
        if not args.no_sort_baseline:
            sb = time_sort_baseline(args.workload, max(3, min(args.steps, 10)), 2, dev, stream)
            ours_ms = head["kernel_ms_mean"]
            sb["speedup_of_ours"] = sb["ms_per_step"] / ours_ms
            line["sort_baseline"] = sb
        if not args.no_e2e:
            line["e2e"] = time_e2e(args.workload, max(3, min(args.steps, 20)), 2, dev, stream)
        if not args.no_outputs:
            line["outputs"] = time_outputs(args.workload, max(3, min(args.steps, 20)), 3, dev, stream, peak)
        if not args.no_cpu_baseline:
            v1, rows1, el1 = oracle_rows_per_s(args.workload, budget_s=args.cpu_seconds / 2)
            vn, rowsn, cores = oracle_rows_per_s_pooled(args.workload, budget_s=args.cpu_seconds / 2)
            line["cpu_baseline"] = {
                "value": vn,
                "unit": "rows/s",
                "cores": cores,
                "kind": "oracle",
                "sample": (f"{rowsn} rows of {w.name} in about {args.cpu_seconds / 2:.0f} s on {cores} spawned "
                           f"processes (numpy fp64 stable sort per row); one core: {v1:.1f} rows/s "
                           f"({rows1} rows in {el1:.1f} s)"),
                "value_one_core": v1,
            }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# ablations (python bench.py --ablation): the pages' ablation switches
# reproduced with this build's flags, each timed beside the default
# ---------------------------------------------------------------------------
ABLATIONS = [
    ("default", 0),
    ("no truncation (search the full row)", 0x1),
    ("list search: quaternary (3 pivots a round)", 0x4000 | 0x2000),
    ("list search: binary (1 pivot a round)", 0x8000 | 0x2000),
    ("list search: 64 bins a round, no key histogram", 0x2000),
    ("fallback: this build (256-bin pass, then 15 pivots a pass)", 0x2 | 0x2000),
    ("fallback: quaternary (3 pivots a pass)", 0x2 | 0x4000 | 0x2000),
    ("fallback: binary (1 pivot a pass)", 0x2 | 0x8000 | 0x2000),
    ("launch: 1 CTA per row", 0x800 | (0 << 8)),
    ("launch: 2 CTAs per row", 0x800 | (1 << 8)),
    ("launch: 4 CTAs per row", 0x800 | (2 << 8)),
    ("launch: 8 CTAs per row", 0x800 | (3 << 8)),
]

PAGES_ABLATIONS = {
    "truncation": "Gaussian truncation cuts latency by about 74% against searching the full logits",
    "quaternary": "quaternary search is slightly slower than binary on truncation hits and about 2.3 ms faster "
                  "on fallbacks over the whole vocabulary",
    "duplicates": "duplicate handling adds about 3.5% latency (not switchable here: the result would not be exact)",
    "autotune": "tiered block-size autotuning cuts latency by almost 30% against one fixed block size "
                "(here: the launch-shape rule against fixed CTAs per row)",
    "source": "Qrita technical summary (gist.science, paper 2602.01518), \"Results\", ablation studies; "
              "other hardware (H100, RTX4090, MI355X), not a target",
}


def run_ablation(args):
    import torch

    import top_selection_row_gb300 as q

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q.lib()
    stream = torch.cuda.Stream(dev)
    numbers = [int(t) for t in args.ablation_workloads.split(",")]
    out = {}
    for n in numbers:
        w = WORKLOADS[n]
        logits, k, p = generate(n)
        if w.dtype == "f32":
            x = torch.from_numpy(logits).to(dev)
        else:
            x = torch.from_numpy(logits.view(np.int16)).to(dev).view(torch.bfloat16)
        # inputs rotate over enough copies to exceed 3x the L2 size (126 MB)
        n_rot = max(2, math.ceil(3 * 126e6 / (w.B * w.V * (w.elem_bytes + 1))) + 1)
        xs = [x] + [x.clone() for _ in range(n_rot - 1)]
        outs = [torch.empty((w.B, w.V), dtype=torch.bool, device=dev) for _ in xs]
        kd = torch.from_numpy(k).to(dev)
        pd = torch.from_numpy(p).to(dev)
        res = {}
        # the default is timed first and again last; the ratios divide by
        # the mean of the two (the spread shows the run-to-run noise)
        for name, flags in ABLATIONS + [("default (timed again, last)", 0)]:
            with torch.cuda.stream(stream):
                for i in range(args.warmup):
                    q.qrita_select_ex(xs[i % n_rot], kd, pd, out=outs[i % n_rot], stream=stream, flags=flags)
            torch.cuda.synchronize(dev)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                s.record(stream)
                for i in range(args.steps):
                    q.qrita_select_ex(xs[i % n_rot], kd, pd, out=outs[i % n_rot], stream=stream, flags=flags)
                e.record(stream)
            torch.cuda.synchronize(dev)
            res[name] = {"flags": flags, "ms_per_call": s.elapsed_time(e) / args.steps}
        base = 0.5 * (res["default"]["ms_per_call"] + res["default (timed again, last)"]["ms_per_call"])
        for r in res.values():
            r["vs_default"] = r["ms_per_call"] / base
        out[w.name] = res
        del xs, outs
    print(json.dumps({"ablation": out, "pages": PAGES_ABLATIONS}), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    data = generate(args.workload)
    rows_per_step = 2
    for _ in range(args.warmup):
        oracle_rows_per_s(args.workload, budget_s=0.0, max_rows=1, data=data)
    t0 = time.perf_counter()
    total = 0
    for _ in range(args.steps):
        _, rows, _ = oracle_rows_per_s(args.workload, budget_s=1e9, max_rows=rows_per_step, data=data)
        total += rows
    el = time.perf_counter() - t0
    v = total / el
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": v,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; shapes of the pages' workloads, no dataset)",
        "config": {"workload": w.name, "global_batch": w.B, "vocab": w.V, "logits_dtype": w.dtype,
                   "seed": 1000 + w.number, "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows_per_step} rows of {w.name} per step (numpy fp64 stable sort, one thread)"},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--no-sweep", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ablation", action="store_true",
                    help="time the ablation switches (truncation, search width, launch shape) instead")
    ap.add_argument("--ablation-workloads", default="2,3,4,5")
    ap.add_argument("--no-outputs", action="store_true",
                    help="skip timing the outputs after the mask (top-k ids, candidate lists)")
    ap.add_argument("--no-sort-baseline", action="store_true",
                    help="skip the torch.sort-based comparator (time and peak memory)")
    ap.add_argument("--rotate", type=int, default=None,
                    help="input copies to rotate over (default: enough to exceed 3x L2)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.ablation:
        run_ablation(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
