"""Seeded synthetic inputs for the SpMM C = A * B (A sparse CSR, B dense).

This module only draws inputs; it holds none of the method's arithmetic (no
format conversion, no product).  Both the oracle-based tests and the GPU path
take their inputs from here, nothing else is shared between them.

All 16-bit values are returned as raw uint16 bit patterns ("bits") together
with a dtype name, "f16" or "bf16".  Values are drawn in float32 and rounded
to nearest-even into the 16-bit type; a value that rounds to exactly zero is
drawn again, so every stored CSR entry is a numeric nonzero.

The named workloads reproduce the synthetic benchmark configurations:
  bcsr_tiny        A 512 x 512 fp16, 64x64 blocks kept with p = 0.5, U[-1,1];
                   B 512 x 128 fp16 U[-1,1]; C fp32.
  wcsr_uniform     A 16384^2 bf16, each entry present with p = 0.01, N(0,1);
                   window 16; B 16384 x 256 bf16 N(0,1); C fp32.
  wcsr_irregular   A 262144^2 bf16, row lengths Zipf(s=1.8) truncated to
                   [1, 20000], columns 70 % in a +-2048 band around the
                   diagonal and 30 % uniform, U[-1,1]; window 16; B N = 128
                   bf16 U[-1,1]; C fp32.
  bcsr_weight      A 18944 x 3584 bf16, 64x64 blocks, exactly 10 % of blocks
                   kept (seeded permutation), N(0, 0.02); B 3584 x 65536 bf16
                   N(0,1); C bf16.
  bcsr_sweep       A 8192^2 bf16, 64x64 blocks, {50,75,90,95} % of blocks
                   zero, U[-1,1]; N in {8,32,64,128,256}; C fp32.
  wcsr_sweep       A 65536^2 bf16, density {0.1,0.5,2} %, uniform columns,
                   window 16, U[-1,1]; N in {8,32,64,128,256}; C fp32.
Seeds: configuration i (0-based, in the order above with the two sweeps
sharing index 4) draws A from default_rng(20260000 + i) and B from
default_rng([20260000 + i, 1]); sweep points add their level and N to the
seed list.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

SEED_BASE = 20260000


# ----------------------------------------------------------------- rounding
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, np.float32).astype(np.float16).view(np.uint16)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Widen 16-bit bits to float32 (exact)."""
    bits = np.asarray(bits, np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == "bf16" else f32_to_f16_bits(x)


def draw_values(rng: np.random.Generator, n: int, dist: str, dtype: str) -> np.ndarray:
    """n nonzero 16-bit values; dist is 'u1' (U[-1,1]), 'n1' (N(0,1)) or 'n002' (N(0,0.02))."""
    out = np.empty(n, np.uint16)
    todo = np.arange(n)
    while len(todo):
        if dist == "u1":
            x = rng.uniform(-1.0, 1.0, size=len(todo)).astype(np.float32)
        elif dist == "n1":
            x = rng.standard_normal(size=len(todo), dtype=np.float32)
        elif dist == "n002":
            x = (rng.standard_normal(size=len(todo), dtype=np.float32) * np.float32(0.02))
        else:
            raise ValueError(dist)
        b = to_bits(x, dtype)
        zero = (b & 0x7FFF) == 0
        out[todo[~zero]] = b[~zero]
        todo = todo[zero]
    return out


def dense_bits(rng: np.random.Generator, shape, dist: str, dtype: str) -> np.ndarray:
    n = int(np.prod(shape))
    return draw_values(rng, n, dist, dtype).reshape(shape)


# ------------------------------------------------------------ sparsity shapes
def _row_ptr_from_rows(rows: np.ndarray, m: int) -> np.ndarray:
    rp = np.zeros(m + 1, np.int64)
    if len(rows):
        np.cumsum(np.bincount(rows, minlength=m), out=rp[1:])
    return rp


def bernoulli_pattern(rng: np.random.Generator, m: int, k: int, p: float):
    """Every entry present independently with probability p (geometric skips
    over the row-major index space).  Returns (row_ptr, col_idx)."""
    total = m * k
    if p <= 0 or total == 0:
        return np.zeros(m + 1, np.int64), np.zeros(0, np.int32)
    if p >= 1:
        pos = np.arange(total, dtype=np.int64)
    else:
        parts = []
        last = -1
        while last < total:
            cnt = int(max(1024, (total - last) * p * 1.05 + 1024))
            gaps = rng.geometric(p, size=cnt).astype(np.int64)
            pos = last + np.cumsum(gaps)
            parts.append(pos)
            last = int(pos[-1])
        pos = np.concatenate(parts)
        pos = pos[pos < total]
    rows = pos // k
    cols = (pos % k).astype(np.int32)
    return _row_ptr_from_rows(rows, m), cols


def block_pattern(rng: np.random.Generator, m: int, k: int, b_row: int, b_col: int,
                  keep: Optional[float] = None, keep_count: Optional[int] = None):
    """Dense b_row x b_col blocks: each kept with probability `keep`
    (Bernoulli per block), or exactly `keep_count` blocks chosen by a seeded
    permutation.  Returns (row_ptr, col_idx)."""
    nbr, nbc = -(-m // b_row), -(-k // b_col)
    if keep_count is not None:
        mask = np.zeros(nbr * nbc, bool)
        mask[rng.permutation(nbr * nbc)[:keep_count]] = True
        mask = mask.reshape(nbr, nbc)
    else:
        mask = rng.random((nbr, nbc)) < keep
    dense = np.kron(mask, np.ones((b_row, b_col), bool))[:m, :k]
    rows, cols = np.nonzero(dense)
    return _row_ptr_from_rows(rows, m), cols.astype(np.int32)


def powerlaw_pattern(rng: np.random.Generator, m: int, k: int, s: float = 1.8, lmin: int = 1,
                     lmax: int = 20000, band: int = 2048, p_band: float = 0.7):
    """Row lengths ~ Zipf(s) truncated to [lmin, lmax] (out-of-range lengths
    redrawn); each column draw lies with probability p_band in
    [i - band, i + band] (uniform, redrawn if outside [0, k)) and otherwise
    uniform in [0, k); duplicate columns in a row are redrawn.  Columns are
    sorted per row.  Returns (row_ptr, col_idx)."""
    lens = rng.zipf(s, size=m).astype(np.int64)
    bad = (lens < lmin) | (lens > lmax) | (lens > k)
    while bad.any():
        lens[bad] = rng.zipf(s, size=int(bad.sum()))
        bad = (lens < lmin) | (lens > lmax) | (lens > k)
    rows = np.repeat(np.arange(m, dtype=np.int64), lens)
    cols = np.empty(len(rows), np.int64)

    def draw(idx):
        pend = idx
        while len(pend):
            r = rows[pend]
            in_band = rng.random(len(pend)) < p_band
            c = np.where(in_band, r + rng.integers(-band, band + 1, size=len(pend)),
                         rng.integers(0, k, size=len(pend)))
            ok = (c >= 0) & (c < k)
            cols[pend[ok]] = c[ok]
            pend = pend[~ok]

    draw(np.arange(len(rows)))
    # Redraw duplicates, looking only at rows that still hold one.
    cand = np.arange(len(rows))
    while True:
        order = np.lexsort((cols[cand], rows[cand]))
        sc = cand[order]
        dup = np.zeros(len(sc), bool)
        dup[1:] = (rows[sc[1:]] == rows[sc[:-1]]) & (cols[sc[1:]] == cols[sc[:-1]])
        if not dup.any():
            break
        draw(sc[dup])
        dup_rows = np.unique(rows[sc[dup]])
        cand = np.nonzero(np.isin(rows, dup_rows))[0]
    order = np.lexsort((cols, rows))
    rp = np.zeros(m + 1, np.int64)
    np.cumsum(lens, out=rp[1:])
    return rp, cols[order].astype(np.int32)


# ------------------------------------------------------------------ workloads
@dataclass
class Workload:
    name: str
    fmt: str            # "bcsr" or "wcsr"
    m: int
    k: int
    n: int
    dtype: str          # "f16" or "bf16" (A and B)
    out_dtype: str      # "f32" or "bf16" (C)
    row_ptr: np.ndarray
    col_idx: np.ndarray
    vals: np.ndarray    # uint16 bits
    b_row: int = 64     # BCSR block height / WCSR window height
    b_col: int = 64     # BCSR block width / WCSR column padding
    b_seed: tuple = ()
    b_dist: str = "u1"
    meta: dict = field(default_factory=dict)
    _B: Optional[np.ndarray] = None

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    def B(self) -> np.ndarray:
        """B as k x n uint16 bits (drawn on first use)."""
        if self._B is None:
            self._B = dense_bits(np.random.default_rng(list(self.b_seed)), (self.k, self.n),
                                 self.b_dist, self.dtype)
        return self._B

    def describe(self) -> str:
        return self.meta.get("desc", self.name)


def _finish(name, fmt, m, k, n, dtype, out_dtype, rp, ci, rng, dist, b_row, b_col, b_seed, b_dist, desc):
    vals = draw_values(rng, len(ci), dist, dtype)
    return Workload(name, fmt, m, k, n, dtype, out_dtype, rp, ci, vals, b_row, b_col,
                    tuple(b_seed), b_dist, {"desc": desc})


def bcsr_tiny(m=512, k=512, n=128, keep=0.5, seed=SEED_BASE + 0) -> Workload:
    rng = np.random.default_rng(seed)
    rp, ci = block_pattern(rng, m, k, 64, 64, keep=keep)
    return _finish("bcsr_tiny", "bcsr", m, k, n, "f16", "f32", rp, ci, rng, "u1", 64, 64,
                   (seed, 1), "u1", f"BCSR {m}x{k} fp16 64x64 blocks p={keep} N={n} C fp32")


def wcsr_uniform(m=16384, k=16384, n=256, density=0.01, seed=SEED_BASE + 1) -> Workload:
    rng = np.random.default_rng(seed)
    rp, ci = bernoulli_pattern(rng, m, k, density)
    return _finish("wcsr_uniform", "wcsr", m, k, n, "bf16", "f32", rp, ci, rng, "n1", 16, 16,
                   (seed, 1), "n1", f"WCSR {m}x{k} bf16 density {density} h16 N={n} C fp32")


def wcsr_irregular(m=262144, k=262144, n=128, seed=SEED_BASE + 2, lmax=20000, band=2048) -> Workload:
    rng = np.random.default_rng(seed)
    rp, ci = powerlaw_pattern(rng, m, k, 1.8, 1, lmax, band, 0.7)
    return _finish("wcsr_irregular", "wcsr", m, k, n, "bf16", "f32", rp, ci, rng, "u1", 16, 16,
                   (seed, 1), "u1", f"WCSR {m}x{k} bf16 Zipf(1.8) rows, banded columns, h16 N={n} C fp32")


def bcsr_weight(m=18944, k=3584, n=65536, keep_frac=0.1, seed=SEED_BASE + 3) -> Workload:
    rng = np.random.default_rng(seed)
    nblk = (-(-m // 64)) * (-(-k // 64))
    rp, ci = block_pattern(rng, m, k, 64, 64, keep_count=int(round(keep_frac * nblk)))
    return _finish("bcsr_weight", "bcsr", m, k, n, "bf16", "bf16", rp, ci, rng, "n002", 64, 64,
                   (seed, 1), "n1",
                   f"BCSR {m}x{k} bf16 64x64 blocks {round(100 * (1 - keep_frac))}% zero N={n} C bf16")


BCSR_SWEEP_SPARSITY = (50, 75, 90, 95)
WCSR_SWEEP_DENSITY = (0.1, 0.5, 2.0)
SWEEP_N = (8, 32, 64, 128, 256)


def bcsr_sweep(sparsity_pct: int, n: int, m: int = 8192, seed=SEED_BASE + 4) -> Workload:
    lvl = BCSR_SWEEP_SPARSITY.index(sparsity_pct) if sparsity_pct in BCSR_SWEEP_SPARSITY else 90 + sparsity_pct
    rng = np.random.default_rng([seed, 0, lvl])
    nblk = (-(-m // 64)) ** 2
    keep = int(round(nblk * (100 - sparsity_pct) / 100.0))
    rp, ci = block_pattern(rng, m, m, 64, 64, keep_count=keep)
    return _finish(f"bcsr_sweep_{sparsity_pct}_N{n}", "bcsr", m, m, n, "bf16", "f32", rp, ci, rng, "u1",
                   64, 64, (seed, 0, lvl, n, 1), "u1",
                   f"BCSR {m}x{m} bf16 64x64 blocks {sparsity_pct}% zero N={n} C fp32")


def wcsr_sweep(density_pct: float, n: int, m: int = 65536, seed=SEED_BASE + 4) -> Workload:
    lvl = WCSR_SWEEP_DENSITY.index(density_pct) if density_pct in WCSR_SWEEP_DENSITY else 90
    rng = np.random.default_rng([seed, 1, lvl])
    rp, ci = bernoulli_pattern(rng, m, m, density_pct / 100.0)
    return _finish(f"wcsr_sweep_{density_pct}_N{n}", "wcsr", m, m, n, "bf16", "f32", rp, ci, rng, "u1",
                   16, 16, (seed, 1, lvl, n, 1), "u1",
                   f"WCSR {m}x{m} bf16 density {density_pct}% h16 N={n} C fp32")


def random_csr(rng: np.random.Generator, m: int, k: int, density: float, dtype: str = "bf16",
               dist: str = "u1"):
    """Small generic Bernoulli CSR for tests: (row_ptr, col_idx, vals bits)."""
    rp, ci = bernoulli_pattern(rng, m, k, density)
    return rp, ci, draw_values(rng, len(ci), dist, dtype)
