"""CPU oracle for the truly sparse linear layer (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python
binding never touch it, and it shares no code with them.

The arithmetic lives in ``snack_oracle.c`` (plain C, IEEE double, sums in
storage order); this module compiles it with gcc on first use, loads it with
ctypes and converts numpy inputs (float32, or bfloat16 carried as uint16
bits) to double exactly.

Source of every definition: "Beyond Masked Sparsity: SNACK Enables Truly
Sparse Neural Networks on GPU" (abstract) -- a layer that stores and
computes only the non-zero connections (COO), back-propagates in the sparse
form, and restructures its connections during Dynamic Sparse Training.  See
the C file for the definition each function writes out.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "snack_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_f64p_opt = ctypes.c_void_p


def compile_library(src: str, out: str) -> None:
    """gcc with the oracle's portable flags (no -march): C source -> shared library."""
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-fno-fast-math", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)


def build(force: bool = False) -> str:
    """Compile the oracle library (once, and again when the source changes)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_library(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = bind(ctypes.CDLL(build()))
        return _lib


def bind(lib):
    """Declare the C signatures on a loaded oracle library; returns it."""
    I64, U64, I32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
    lib.oracle_set_threads.argtypes = [I32]
    lib.oracle_get_threads.restype = I32
    lib.oracle_check_coo.argtypes = [I64, I64, I64, _i32p, _i32p]
    lib.oracle_check_coo.restype = I32
    lib.oracle_fwd.argtypes = [I64, I64, I64, _i32p, _i32p, _f64p, I64, _f64p, _f64p_opt, _f64p, _f64p_opt]
    lib.oracle_fwd.restype = I32
    lib.oracle_dx.argtypes = [I64, I64, I64, _i32p, _i32p, _f64p, I64, _f64p, _f64p, _f64p_opt]
    lib.oracle_dx.restype = I32
    lib.oracle_dw.argtypes = [I64, I64, I64, _i32p, _i32p, I64, _f64p, _f64p, _f64p, _f64p_opt, _f64p_opt]
    lib.oracle_dw.restype = I32
    lib.oracle_gelu.argtypes = [ctypes.c_double]
    lib.oracle_gelu.restype = ctypes.c_double
    lib.oracle_gelu_grad.argtypes = [ctypes.c_double]
    lib.oracle_gelu_grad.restype = ctypes.c_double
    lib.oracle_gelu_vec.argtypes = [I64, _f64p, _f64p]
    lib.oracle_gelu_grad_vec.argtypes = [I64, _f64p, _f64p]
    lib.oracle_splitmix64_mix.argtypes = [U64]
    lib.oracle_splitmix64_mix.restype = U64
    lib.oracle_regrow_base.argtypes = [U64, U64]
    lib.oracle_regrow_base.restype = U64
    lib.oracle_regrow_draw.argtypes = [U64, U64, U64, U64]
    lib.oracle_regrow_draw.restype = U64
    lib.oracle_restructure.argtypes = [I64, I64, I64, _i32p, _i32p, _f64p, I64, U64, U64, I64,
                                       _i32p, _i32p, _i64p]
    lib.oracle_restructure.restype = I64
    lib.oracle_row_base.argtypes = [U64, U64, U64]
    lib.oracle_row_base.restype = U64
    lib.oracle_restructure_rows.argtypes = [I64, I64, I64, _i32p, _i32p, _f64p, I64, U64, U64, I64,
                                            _i32p, _i32p, _i64p]
    lib.oracle_restructure_rows.restype = I64
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def as_f64(a: np.ndarray, dtype: str = "f32") -> np.ndarray:
    """Exact widening of stored values to double: float32, or bf16 bits (uint16)."""
    if dtype == "bf16":
        a = (np.ascontiguousarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    elif dtype != "f32" and dtype != "f64":
        raise ValueError(dtype)
    return np.ascontiguousarray(a, dtype=np.float64)


def _idx(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def check_coo(out_f: int, in_f: int, row, col) -> int:
    """0 valid, 1 index out of range, 2 not strictly increasing in (row, col)."""
    row, col = _idx(row), _idx(col)
    return int(_load().oracle_check_coo(out_f, in_f, row.shape[0], row, col))


def fwd(out_f: int, in_f: int, row, col, val: np.ndarray, x: np.ndarray, bias=None):
    """Y = X W^T + bias over the stored weights; returns (Y [B,out_f], T [B,out_f])."""
    row, col = _idx(row), _idx(col)
    val = np.ascontiguousarray(val, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    batch = x.shape[0]
    assert x.shape == (batch, in_f)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    y = np.empty((batch, out_f), dtype=np.float64)
    t = np.empty((batch, out_f), dtype=np.float64)
    rc = _load().oracle_fwd(out_f, in_f, row.shape[0], row, col, val, batch, x, _ptr(b), y, _ptr(t))
    if rc:
        raise ValueError("oracle_fwd: index out of range")
    return y, t


def dx(out_f: int, in_f: int, row, col, val: np.ndarray, dy: np.ndarray):
    """dX = dY W over the stored weights; returns (dX [B,in_f], T [B,in_f])."""
    row, col = _idx(row), _idx(col)
    val = np.ascontiguousarray(val, dtype=np.float64)
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    batch = dy.shape[0]
    assert dy.shape == (batch, out_f)
    out = np.empty((batch, in_f), dtype=np.float64)
    t = np.empty((batch, in_f), dtype=np.float64)
    rc = _load().oracle_dx(out_f, in_f, row.shape[0], row, col, val, batch, dy, out, _ptr(t))
    if rc:
        raise ValueError("oracle_dx: index out of range")
    return out, t


def dw(out_f: int, in_f: int, row, col, x: np.ndarray, dy: np.ndarray, want_db: bool = True):
    """dW[k] = sum_b dY[b,row_k] X[b,col_k] and db[r] = sum_b dY[b,r]; returns (dW, T, db)."""
    row, col = _idx(row), _idx(col)
    x = np.ascontiguousarray(x, dtype=np.float64)
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    batch = x.shape[0]
    assert x.shape == (batch, in_f) and dy.shape == (batch, out_f)
    nnz = row.shape[0]
    g = np.empty(nnz, dtype=np.float64)
    t = np.empty(nnz, dtype=np.float64)
    db = np.empty(out_f, dtype=np.float64) if want_db else None
    rc = _load().oracle_dw(out_f, in_f, nnz, row, col, batch, x, dy, g, _ptr(t), _ptr(db))
    if rc:
        raise ValueError("oracle_dw: index out of range")
    return g, t, db


def gelu(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_gelu_vec(x.size, x.reshape(-1), y.reshape(-1))
    return y


def gelu_grad(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_gelu_grad_vec(x.size, x.reshape(-1), y.reshape(-1))
    return y


def splitmix64_mix(z: int) -> int:
    return int(_load().oracle_splitmix64_mix(int(z) & (2**64 - 1)))


def regrow_base(seed: int, step: int) -> int:
    """State before the first draw of (seed, step)."""
    return int(_load().oracle_regrow_base(seed, step))


def regrow_draw(seed: int, step: int, i: int, n_pos: int) -> int:
    return int(_load().oracle_regrow_draw(seed, step, i, n_pos))


def default_max_draws(n_prune: int) -> int:
    """Draw budget of a restructure call: 64 draws per regrown weight plus 2^20."""
    return 64 * int(n_prune) + (1 << 20)


class RestructureError(ValueError):
    pass


_RESTRUCTURE_ERRORS = {-1: "pattern not valid row-sorted COO", -2: "n_prune out of range",
                       -3: "fewer empty positions than n_prune", -4: "draw budget exhausted",
                       -5: "out of memory"}


def restructure(out_f: int, in_f: int, row, col, val_f64: np.ndarray, n_prune: int, seed: int,
                step: int, max_draws: Optional[int] = None):
    """Prune n_prune smallest |w| and regrow as many at random empty positions.

    Returns (row_out, col_out, src_out, draws): src_out[j] is the old index of a
    surviving weight, -1 for a regrown one (value +0); draws is the number of
    random draws consumed.
    """
    row, col = _idx(row), _idx(col)
    nnz = row.shape[0]
    val_f64 = np.ascontiguousarray(val_f64, dtype=np.float64)
    ro = np.empty(nnz, dtype=np.int32)
    co = np.empty(nnz, dtype=np.int32)
    so = np.empty(nnz, dtype=np.int64)
    md = default_max_draws(n_prune) if max_draws is None else int(max_draws)
    rc = _load().oracle_restructure(out_f, in_f, nnz, row, col, val_f64, int(n_prune),
                                    int(seed) & (2**64 - 1), int(step) & (2**64 - 1), md, ro, co, so)
    if rc < 0:
        raise RestructureError(_RESTRUCTURE_ERRORS.get(int(rc), str(rc)))
    return ro, co, so, int(rc)


def restructure_rows(out_f: int, in_f: int, row, col, val_f64: np.ndarray, n_per_row: int, seed: int,
                     step: int, max_draws_per_row: Optional[int] = None):
    """Per-row (constant fan-in) restructure: every row prunes min(n_per_row, its
    length) smallest |w| and regrows as many columns of the same row that were
    empty, from the row's own draw stream.

    Returns (row_out, col_out, src_out, draws) as restructure() does; every row
    keeps its count and its offsets.
    """
    row, col = _idx(row), _idx(col)
    nnz = row.shape[0]
    val_f64 = np.ascontiguousarray(val_f64, dtype=np.float64)
    ro = np.empty(nnz, dtype=np.int32)
    co = np.empty(nnz, dtype=np.int32)
    so = np.empty(nnz, dtype=np.int64)
    md = default_max_draws(n_per_row) if max_draws_per_row is None else int(max_draws_per_row)
    rc = _load().oracle_restructure_rows(out_f, in_f, nnz, row, col, val_f64, int(n_per_row),
                                         int(seed) & (2**64 - 1), int(step) & (2**64 - 1), md, ro, co, so)
    if rc < 0:
        raise RestructureError(_ROWS_ERRORS.get(int(rc), str(rc)))
    return ro, co, so, int(rc)


_ROWS_ERRORS = {-1: "pattern not valid row-sorted COO", -2: "n_per_row negative",
                -3: "a row has fewer empty columns than it prunes", -4: "a row's draw budget is exhausted",
                -5: "out of memory"}


def row_base(seed: int, step: int, r: int) -> int:
    return int(_load().oracle_row_base(int(seed) & (2**64 - 1), int(step) & (2**64 - 1), int(r)))


def restructure_values(val_stored: np.ndarray, src_out: np.ndarray) -> np.ndarray:
    """Values of a restructured layer in the stored dtype: old bits, or +0 where regrown."""
    out = np.zeros(src_out.shape[0], dtype=val_stored.dtype)
    keep = src_out >= 0
    out[keep] = val_stored[src_out[keep]]
    return out


def mlp_step(layer1, layer2, x64: np.ndarray, dy2_64: np.ndarray):
    """Two sparse layers with GELU between them: forward and backward, all in double.

    layerN = (out_f, in_f, row, col, val_f64, bias_f64).  Returns a dict with
    y1, h, y2, dh, dy1, dx, dw1, db1, dw2, db2 (the T arrays are omitted).
    """
    o1, i1, r1, c1, v1, b1 = layer1
    o2, i2, r2, c2, v2, b2 = layer2
    y1, _ = fwd(o1, i1, r1, c1, v1, x64, b1)
    h = gelu(y1)
    y2, _ = fwd(o2, i2, r2, c2, v2, h, b2)
    dh, _ = dx(o2, i2, r2, c2, v2, dy2_64)
    dy1 = dh * gelu_grad(y1)
    dxx, _ = dx(o1, i1, r1, c1, v1, dy1)
    dw2, _, db2 = dw(o2, i2, r2, c2, h, dy2_64)
    dw1, _, db1 = dw(o1, i1, r1, c1, x64, dy1)
    return dict(y1=y1, h=h, y2=y2, dh=dh, dy1=dy1, dx=dxx, dw1=dw1, db1=db1, dw2=dw2, db2=db2)
