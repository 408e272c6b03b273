"""Write tests/golden/flagged_counts.json: for every workload, how many of its
rows have top-p active and how many of those the oracle flags (cumulative
mass at the top-p boundary within 1e-6 * p of p).

Calls only the oracle (and the seeded input generators). Run from the
repository root:  python tests/golden/make_flagged_counts.py
The bench reports these counts beside its per-workload path counts.
"""

from __future__ import annotations

import json
import multiprocessing as mp
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OUT = os.path.join(ROOT, "tests", "golden", "flagged_counts.json")


def _count(job):
    number, first, stride = job
    from oracle import select_batch
    from workloads import generate

    logits, k, p = generate(number)
    w_dtype = "f32" if logits.dtype.kind == "f" else "bf16"
    rows = list(range(first, logits.shape[0], stride))
    res = select_batch(logits, w_dtype, k, p, rows=rows)
    top_p = sum(1 for r in rows if p[r] < 1.0)
    return top_p, sum(1 for _, x in res if x.ambiguous)


def main():
    from workloads import WORKLOADS

    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    out = {"note": "written by tests/golden/make_flagged_counts.py from the oracle alone", "workloads": {}}
    ctx = mp.get_context("spawn")
    for n, w in WORKLOADS.items():
        procs = max(1, min(cores, w.B, 8))
        with ctx.Pool(procs) as pool:
            res = pool.map(_count, [(n, i, procs) for i in range(procs)])
        out["workloads"][w.name] = {"rows": w.B, "top_p_rows": sum(a for a, _ in res),
                                    "flagged": sum(b for _, b in res)}
        print(w.name, out["workloads"][w.name], flush=True)
    with open(OUT, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
