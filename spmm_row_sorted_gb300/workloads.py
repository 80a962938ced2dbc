"""Seeded synthetic layers and activations for the truly sparse linear layer.

This module only draws inputs: sparsity patterns, weight values, biases and
activations, from seeded numpy generators.  It holds none of the layer's
arithmetic (no products, sums, pruning or regrowth), so both the CPU oracle
and the CUDA library can be fed from it without sharing any of the method.

The workloads are those of the SNACK paper's setting ("Beyond Masked
Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU", abstract):
unstructured sparsity at 50-99 %, small batches, fp32 or bf16 storage.
Concrete sizes are listed in ``CONFIGS``.

Conventions
-----------
* W is ``out_f x in_f`` and stored as row-sorted COO: ``row[k]`` (output
  feature), ``col[k]`` (input feature), strictly increasing in
  ``(row, col)``; int32.
* Values are float32, or bfloat16 carried as raw ``uint16`` bit patterns
  (numpy has no bf16 type).  bf16 values are the round-to-nearest-even image
  of a float32 draw.
* Activations are row-major ``[batch, features]``.
* Every tensor has its own generator, seeded by ``(seed, tensor_id, ...)``.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# tensor ids for the per-tensor generators
_T_POS, _T_VAL, _T_X, _T_DY, _T_ROWPERM, _T_ZIPFCOL, _T_BIAS, _T_AUX = range(1, 9)


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = np.where(nan, (u >> 16) | 0x40, rounded).astype(np.uint16)
    return out


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits (uint16) to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def nnz_for(out_f: int, in_f: int, density: float) -> int:
    """Number of stored weights for a density: round half up of out*in*density."""
    return int(math.floor(out_f * in_f * density + 0.5))


def _rng(seed: int, *ids: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), *[int(i) for i in ids]])


def uniform_positions(out_f: int, in_f: int, nnz: int, seed: int) -> np.ndarray:
    """nnz distinct linear positions row*in_f+col, uniform without replacement, sorted."""
    n_pos = out_f * in_f
    if nnz > n_pos:
        raise ValueError("nnz exceeds out_f*in_f")
    rng = _rng(seed, _T_POS)
    if nnz == n_pos:
        return np.arange(n_pos, dtype=np.int64)
    if nnz * 2 > n_pos:
        p = rng.permutation(n_pos)[:nnz]
    else:
        p = rng.choice(n_pos, size=nnz, replace=False, shuffle=False)
    p = np.sort(p.astype(np.int64))
    return p


def zipf_row_counts(out_f: int, in_f: int, nnz: int, s: float) -> np.ndarray:
    """Per-rank nnz counts ~ rank**(-s), capped at in_f, summing exactly to nnz.

    The scale lam solves sum_r min(in_f, lam * r**-s) = nnz (bisection); each
    count is floored and the deficit is handed out by largest remainder, ties
    to the lower rank.  Returned in rank order (rank 1 first).
    """
    if nnz > out_f * in_f:
        raise ValueError("nnz exceeds out_f*in_f")
    ranks = np.arange(1, out_f + 1, dtype=np.float64)
    w = ranks ** (-s)

    def total(lam: float) -> float:
        return float(np.minimum(float(in_f), lam * w).sum())

    lo, hi = 0.0, float(in_f) * float(out_f) ** s + 1.0
    for _ in range(300):
        mid = 0.5 * (lo + hi)
        if total(mid) < nnz:
            lo = mid
        else:
            hi = mid
    exact = np.minimum(float(in_f), hi * w)
    counts = np.floor(exact).astype(np.int64)
    deficit = int(nnz - counts.sum())
    # bisection leaves total(hi) in [nnz, nnz+1), so the floored sum never exceeds nnz
    assert deficit >= 0
    if deficit > 0:
        frac = exact - np.floor(exact)
        frac[counts >= in_f] = -1.0
        order = np.lexsort((ranks, -frac))  # largest remainder first, ties to lower rank
        counts[order[:deficit]] += 1
    assert counts.sum() == nnz and counts.max() <= in_f and counts.min() >= 0
    return counts


def zipf_positions(out_f: int, in_f: int, nnz: int, s: float, seed: int) -> np.ndarray:
    """Sorted linear positions with Zipf(s) row lengths and uniform columns per row."""
    counts_by_rank = zipf_row_counts(out_f, in_f, nnz, s)
    perm = _rng(seed, _T_ROWPERM).permutation(out_f)
    counts = np.zeros(out_f, dtype=np.int64)
    counts[perm] = counts_by_rank  # rank i -> row perm[i]
    rng = _rng(seed, _T_ZIPFCOL)
    parts = []
    for r in range(out_f):
        c = int(counts[r])
        if c == 0:
            continue
        if c == in_f:
            cols = np.arange(in_f, dtype=np.int64)
        else:
            cols = np.sort(rng.choice(in_f, size=c, replace=False, shuffle=False).astype(np.int64))
        parts.append(r * in_f + cols)
    if not parts:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(parts)


def fanin_positions(out_f: int, in_f: int, fan_in: int, seed: int) -> np.ndarray:
    """Sorted linear positions with exactly fan_in uniform columns in every row
    (constant fan-in, the layout of structured DST)."""
    if fan_in > in_f:
        raise ValueError("fan_in exceeds in_f")
    rng = _rng(seed, _T_ZIPFCOL)
    keys = rng.random((out_f, in_f)) if out_f * in_f <= (1 << 26) else None
    parts = []
    for r in range(out_f):
        if keys is not None:
            cols = np.sort(np.argpartition(keys[r], fan_in - 1)[:fan_in]) if fan_in > 0 else np.zeros(0, np.int64)
        else:
            cols = np.sort(rng.choice(in_f, size=fan_in, replace=False, shuffle=False))
        parts.append(r * in_f + cols.astype(np.int64))
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def diagonal_positions(out_f: int, in_f: int, n_diag: int, seed: int) -> np.ndarray:
    """Sorted linear positions on n_diag wrapped diagonals: row r holds the
    columns (r + o) mod in_f for n_diag distinct offsets o drawn uniformly from
    [0, in_f) (a diagonal sparsity pattern; every row holds n_diag weights, and
    every column too when out_f == in_f)."""
    if n_diag > in_f:
        raise ValueError("n_diag exceeds in_f")
    offs = _rng(seed, _T_AUX).choice(in_f, size=n_diag, replace=False).astype(np.int64)
    r = np.arange(out_f, dtype=np.int64)[:, None]
    cols = np.sort((r + offs[None, :]) % in_f, axis=1)
    return (r * in_f + cols).reshape(-1)


@dataclasses.dataclass
class Layer:
    """One sparse layer: W (out_f x in_f) as row-sorted COO plus a bias."""

    out_f: int
    in_f: int
    row: np.ndarray  # int32 [nnz]
    col: np.ndarray  # int32 [nnz]
    val: np.ndarray  # float32 [nnz] or uint16 bf16 bits [nnz]
    bias: np.ndarray  # float32 [out_f]
    val_dtype: str  # "f32" | "bf16"

    @property
    def nnz(self) -> int:
        return int(self.row.shape[0])

    def val_f32(self) -> np.ndarray:
        return self.val if self.val_dtype == "f32" else f32_from_bf16_bits(self.val)


@dataclasses.dataclass
class Acts:
    """Activations for one call: X [batch, in_f] and dY [batch, out_f]."""

    x: np.ndarray  # float32 or uint16 bf16 bits
    dy: np.ndarray
    act_dtype: str

    @property
    def batch(self) -> int:
        return int(self.x.shape[0])


def _store(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a32, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_from_f32(a32)
    raise ValueError(dtype)


def make_layer(out_f: int, in_f: int, *, nnz: Optional[int] = None, density: Optional[float] = None,
               val_std: float = 0.02, val_dtype: str = "f32", seed: int = 0,
               zipf_s: Optional[float] = None, bias: str = "zeros", fan_in: Optional[int] = None,
               diagonals: Optional[int] = None) -> Layer:
    """Seeded layer with uniform, Zipf-row, constant fan-in or wrapped-diagonal
    positions and N(0, val_std) values."""
    if fan_in is not None:
        nnz = out_f * fan_in
        p = fanin_positions(out_f, in_f, fan_in, seed)
    elif diagonals is not None:
        nnz = out_f * diagonals
        p = diagonal_positions(out_f, in_f, diagonals, seed)
    else:
        if nnz is None:
            if density is None:
                raise ValueError("give nnz, density or fan_in")
            nnz = nnz_for(out_f, in_f, density)
        if zipf_s is None:
            p = uniform_positions(out_f, in_f, nnz, seed)
        else:
            p = zipf_positions(out_f, in_f, nnz, zipf_s, seed)
    row = (p // in_f).astype(np.int32)
    col = (p % in_f).astype(np.int32)
    v = (_rng(seed, _T_VAL).standard_normal(nnz) * val_std).astype(np.float32)
    if bias == "zeros":
        b = np.zeros(out_f, dtype=np.float32)
    elif bias == "normal":
        b = _rng(seed, _T_BIAS).standard_normal(out_f).astype(np.float32)
    else:
        raise ValueError(bias)
    return Layer(out_f, in_f, row, col, _store(v, val_dtype), b, val_dtype)


def make_acts(batch: int, in_f: int, out_f: int, act_dtype: str = "f32", seed: int = 0,
              stream: int = 0) -> Acts:
    """Seeded X ~ N(0,1) [batch, in_f] and dY ~ N(0,1) [batch, out_f]."""
    x = _rng(seed, _T_X, stream).standard_normal((batch, in_f)).astype(np.float32)
    dy = _rng(seed, _T_DY, stream).standard_normal((batch, out_f)).astype(np.float32)
    return Acts(_store(x, act_dtype), _store(dy, act_dtype), act_dtype)


def random_normal(shape, seed: int, stream: int, std: float = 1.0) -> np.ndarray:
    """Auxiliary seeded float32 N(0, std) array (test probes, finite differences)."""
    return (_rng(seed, _T_AUX, stream).standard_normal(shape) * std).astype(np.float32)


# The five workloads (sizes, densities, dtypes and batches).
CONFIGS = {
    "c1": dict(name="sparse linear 1024x1024, 95% sparse, fp32, batch 8",
               out_f=1024, in_f=1024, density=0.05, val_std=1.0 / math.sqrt(nnz_for(1024, 1024, 0.05) / 1024),
               val_dtype="f32", act_dtype="f32", batches=(8,), ops=("fwd", "dx", "dw")),
    "c2": dict(name="inference layer 4096x4096, 90% sparse, bf16, batch 1/16/64",
               out_f=4096, in_f=4096, density=0.10, val_std=0.02,
               val_dtype="bf16", act_dtype="bf16", batches=(1, 16, 64), ops=("fwd",)),
    "c3": dict(name="sparse MLP 768->3072(GELU)->768, 99% sparse, fp32, 1024 tokens",
               layers=((3072, 768), (768, 3072)), density=0.01, val_dtype="f32", act_dtype="f32",
               batches=(1024,), ops=("fwd", "dx", "dw")),
    "c4": dict(name="layer 16384x16384, 99% sparse, Zipf(1.2) rows, fp32, batch 32, +restructure",
               out_f=16384, in_f=16384, density=0.01, val_std=0.02, zipf_s=1.2,
               val_dtype="f32", act_dtype="f32", batches=(32,), ops=("fwd", "dx", "dw", "restructure"),
               prune_frac=0.10),
    "c5": dict(name="layer 8192x8192, 50% sparse, bf16, batch 128",
               out_f=8192, in_f=8192, density=0.50, val_std=0.02,
               val_dtype="bf16", act_dtype="bf16", batches=(128,), ops=("fwd", "dx", "dw")),
}


def kaiming_std(out_f: int, nnz: int) -> float:
    """sqrt(2 / fan_in) with fan_in = mean stored weights per output row."""
    return math.sqrt(2.0 / (nnz / out_f))


def config_layer(name: str, seed: int = 0, layer_index: int = 0) -> Layer:
    """The seeded layer of a named workload (c3 has two layers)."""
    c = CONFIGS[name]
    if name == "c3":
        out_f, in_f = c["layers"][layer_index]
        nnz = nnz_for(out_f, in_f, c["density"])
        return make_layer(out_f, in_f, nnz=nnz, val_std=kaiming_std(out_f, nnz), val_dtype="f32",
                          seed=seed * 16 + layer_index)
    return make_layer(c["out_f"], c["in_f"], density=c["density"], val_std=c["val_std"],
                      val_dtype=c["val_dtype"], seed=seed, zipf_s=c.get("zipf_s"))
