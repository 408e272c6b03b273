"""Seeded synthetic logit batches shared by the tests, the smoke check and the bench.

This module only draws random inputs. It holds none of the selection
arithmetic, so the oracle and the CUDA path can both take their inputs from
it without sharing any part of the method.

The five workloads stand in for the real model logits of the Qrita pages'
evaluation (Llama / Qwen / GPT-OSS / Gemma vocabularies on H100, RTX4090 and
MI355X; Qrita technical summary, gist.science paper 2602.01518, "Results");
only their shapes and value structure are used. Recipe (numpy PCG64,
seed = 1000 + workload number):

1. B=4,    V=32000,  fp32 N(0,1), 10 outliers/row at 4..10 sigma, k=50, p=1
2. B=64,   V=128256, fp32 N(0,1), 32 outliers/row at 5..12 sigma,
   k ~ U{1..1024}, p=1
3. B=128,  V=151936, fp32 N(0,1)/T, T ~ U[0.5,1.5] per row, 64 outliers/row
   at 4..10 row-sigma, k=V (off), p ~ U[0.5,0.99]
4. B=256,  V=201088, bf16(N(0,2)); floor(0.2*B) rows (chosen by seed) are
   bf16(U[-1,1]) instead; no outliers; k ~ U{1..4096}, p ~ U[0.8,1.0]
5. B=1024, V=262144, bf16(N(0,1)), 128 outliers/row at 4..10 sigma,
   k from {1,20,256,2048,V}, p from {0.9,0.95,1.0}

"Outlier at a sigma" replaces the value at a distinct uniformly chosen
position by mu + a*sigma of that row's background (mu = 0). bf16 values are
rounded to nearest even from fp32 and kept as raw uint16 bits.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    number: int
    name: str
    B: int
    V: int
    dtype: str  # "f32" or "bf16"

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def bytes_per_row(self) -> int:
        """Algorithmic HBM bytes per row: one logits read, one uint8 mask write, k and p."""
        return self.V * self.elem_bytes + self.V + 8


WORKLOADS = {
    1: Workload(1, "b4_v32000_f32_topk50", 4, 32000, "f32"),
    2: Workload(2, "b64_v128256_f32_topk", 64, 128256, "f32"),
    3: Workload(3, "b128_v151936_f32_topp", 128, 151936, "f32"),
    4: Workload(4, "b256_v201088_bf16_topk_topp_ties", 256, 201088, "bf16"),
    5: Workload(5, "b1024_v262144_bf16_mixed", 1024, 262144, "bf16"),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the raw uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).reshape(-1)
    out = np.empty(u.shape, np.uint16)
    step = 1 << 20  # blocks that stay in cache
    for i in range(0, u.size, step):
        b = u[i : i + step]
        # finite inputs only (the generators draw no NaN): no uint32 overflow
        r = (b >> np.uint32(16)) & np.uint32(1)
        r += np.uint32(0x7FFF)
        r += b
        r >>= np.uint32(16)
        out[i : i + step] = r
    return out.reshape(np.shape(a))


def _place_outliers(rng, x: np.ndarray, n_out: int, a_lo: float, a_hi: float, sigma):
    """Replace n_out distinct positions per row by a*sigma, a ~ U[a_lo, a_hi]."""
    B, V = x.shape
    sig = np.broadcast_to(np.asarray(sigma, dtype=np.float64).reshape(-1, 1), (B, 1))
    for r in range(B):
        pos = rng.choice(V, size=n_out, replace=False)
        a = rng.uniform(a_lo, a_hi, size=n_out)
        x[r, pos] = (a * sig[r, 0]).astype(np.float32)


def generate(number: int, rows: int | None = None):
    """Return (logits, k, p) for workload ``number``.

    logits: float32 [B, V] for fp32 workloads, uint16 bf16 bits for bf16 ones.
    k: int32 [B]; p: float32 [B]. ``rows`` truncates the batch (same leading
    rows as the full batch, since every row is drawn in order).
    """
    w = WORKLOADS[number]
    rng = np.random.Generator(np.random.PCG64(1000 + number))
    B, V = w.B, w.V
    if number == 1:
        x = rng.standard_normal((B, V), dtype=np.float32)
        _place_outliers(rng, x, 10, 4.0, 10.0, np.ones(B))
        k = np.full(B, 50, np.int32)
        p = np.ones(B, np.float32)
        logits = x
    elif number == 2:
        x = rng.standard_normal((B, V), dtype=np.float32)
        _place_outliers(rng, x, 32, 5.0, 12.0, np.ones(B))
        k = rng.integers(1, 1024, size=B, endpoint=True).astype(np.int32)
        p = np.ones(B, np.float32)
        logits = x
    elif number == 3:
        T = rng.uniform(0.5, 1.5, size=B)
        x = rng.standard_normal((B, V), dtype=np.float32)
        x = (x / T.reshape(-1, 1)).astype(np.float32)
        _place_outliers(rng, x, 64, 4.0, 10.0, 1.0 / T)
        k = np.full(B, V, np.int32)
        p = rng.uniform(0.5, 0.99, size=B).astype(np.float32)
        logits = x
    elif number == 4:
        x = (rng.standard_normal((B, V), dtype=np.float32) * np.float32(np.sqrt(2.0)))
        n_uni = int(np.floor(0.2 * B))
        uni_rows = rng.choice(B, size=n_uni, replace=False)
        x[uni_rows] = rng.uniform(-1.0, 1.0, size=(n_uni, V)).astype(np.float32)
        k = rng.integers(1, 4096, size=B, endpoint=True).astype(np.int32)
        p = rng.uniform(0.8, 1.0, size=B).astype(np.float32)
        logits = f32_to_bf16_bits(x)
    elif number == 5:
        x = rng.standard_normal((B, V), dtype=np.float32)
        _place_outliers(rng, x, 128, 4.0, 10.0, np.ones(B))
        k = rng.choice(np.array([1, 20, 256, 2048, V], dtype=np.int32), size=B)
        p = rng.choice(np.array([0.9, 0.95, 1.0], dtype=np.float32), size=B)
        logits = f32_to_bf16_bits(x)
    else:
        raise KeyError(number)
    if rows is not None:
        logits, k, p = logits[:rows], k[:rows], p[:rows]
    return np.ascontiguousarray(logits), k.astype(np.int32), p.astype(np.float32)


def assumptions(number: int) -> str:
    """One-line statement of the choices the workload description leaves open."""
    notes = {
        1: "outliers replace 10 distinct positions at U[4,10] sigma",
        2: "outliers replace 32 distinct positions at U[5,12] sigma",
        3: "outlier magnitude assumed U[4,10] row-sigma (64 per row); k=V means top-k off",
        4: "uniform rows are exactly floor(0.2*B), chosen by seed; p drawn U[0.8,1.0]",
        5: "outlier magnitude assumed U[4,10] sigma (128 per row); k=V means top-k off",
    }
    return notes[number]
