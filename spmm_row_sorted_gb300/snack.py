"""Thin Python binding of libsnack (include/snack.h).

The functions named ``snack_*`` mirror the C entry points one to one and only
marshal arguments: torch tensors become device pointers and byte sizes, the
stream defaults to torch's current stream.  Every computation runs in the CUDA
library; when the library has not been built, loading it raises
``SnackLibraryMissing`` -- there is no fallback of any kind.

``SparseLinear`` is a convenience owner of one layer (pattern, values, bias,
plan and workspace tensors) on top of those calls, and ``sparse_linear`` an
autograd function over it.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

SNACK_OK = 0
STATUS_NAMES = {0: "SNACK_OK", 1: "SNACK_ERR_INVALID_ARG", 2: "SNACK_ERR_UNSORTED", 3: "SNACK_ERR_OUT_OF_RANGE",
                4: "SNACK_ERR_WORKSPACE", 5: "SNACK_ERR_CUDA", 6: "SNACK_ERR_TIMEOUT", 7: "SNACK_ERR_UNSUPPORTED",
                8: "SNACK_ERR_NO_SPACE"}
SNACK_F32, SNACK_BF16 = 0, 1

EXPORTED = ("snack_query_sizes", "snack_create", "snack_spmm_fwd", "snack_spmm_fwd_noalloc", "snack_spmm_dx",
            "snack_spmm_fwd_gelu", "snack_spmm_dx_gelu", "snack_sddmm_dw", "snack_backward",
            "snack_restructure_workspace_size", "snack_restructure", "snack_restructure_rows_workspace_size",
            "snack_restructure_rows", "snack_wait_plan", "snack_destroy", "snack_status_string", "snack_version",
            "snack_trace_start", "snack_trace_read", "snack_trace_stop")


class SnackLibraryMissing(RuntimeError):
    pass


class SnackError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({msg})")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load libsnack.so (must have been built with spmm_row_sorted_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise SnackLibraryMissing(f"{p} is missing: build it with `python -m spmm_row_sorted_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
        st = ctypes.c_int
        lib.snack_query_sizes.argtypes = [i32, i32, i64, i32, st, st, ctypes.POINTER(sz), ctypes.POINTER(sz)]
        lib.snack_query_sizes.restype = st
        lib.snack_create.argtypes = [ctypes.POINTER(vp), i32, i32, i64, i32, st, st, vp, vp, vp, sz, vp, sz,
                                     ctypes.c_int, vp]
        lib.snack_create.restype = st
        lib.snack_spmm_fwd.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        lib.snack_spmm_fwd.restype = st
        lib.snack_spmm_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp]
        lib.snack_spmm_fwd_noalloc.restype = st
        lib.snack_spmm_fwd_gelu.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        lib.snack_spmm_fwd_gelu.restype = st
        lib.snack_spmm_dx_gelu.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        lib.snack_spmm_dx_gelu.restype = st
        lib.snack_spmm_dx.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, sz, vp]
        lib.snack_spmm_dx.restype = st
        lib.snack_sddmm_dw.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        lib.snack_sddmm_dw.restype = st
        lib.snack_backward.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        lib.snack_backward.restype = st
        lib.snack_restructure_workspace_size.argtypes = [vp, i64, ctypes.POINTER(sz)]
        lib.snack_restructure_workspace_size.restype = st
        lib.snack_restructure.argtypes = [vp, vp, vp, vp, i64, u64, u64, vp, vp, vp, vp, vp, sz, vp]
        lib.snack_restructure.restype = st
        lib.snack_restructure_rows_workspace_size.argtypes = [vp, i64, ctypes.POINTER(sz)]
        lib.snack_restructure_rows_workspace_size.restype = st
        lib.snack_restructure_rows.argtypes = [vp, vp, vp, vp, i64, u64, u64, vp, vp, vp, vp, vp, sz, vp]
        lib.snack_restructure_rows.restype = st
        lib.snack_wait_plan.argtypes = [vp, vp]
        lib.snack_wait_plan.restype = st
        lib.snack_destroy.argtypes = [vp]
        lib.snack_destroy.restype = None
        lib.snack_status_string.argtypes = [st]
        lib.snack_status_string.restype = ctypes.c_char_p
        lib.snack_version.argtypes = []
        lib.snack_version.restype = ctypes.c_int
        lib.snack_trace_start.argtypes = [i32]
        lib.snack_trace_start.restype = st
        lib.snack_trace_read.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), i32,
                                         ctypes.POINTER(i32)]
        lib.snack_trace_read.restype = st
        lib.snack_trace_stop.argtypes = []
        lib.snack_trace_stop.restype = st
        _lib = lib
        return lib


def _check(fn: str, status: int) -> None:
    if status != SNACK_OK:
        raise SnackError(fn, status, load().snack_status_string(status).decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return SNACK_F32
    if dt == torch.bfloat16:
        return SNACK_BF16
    raise ValueError(f"unsupported dtype {dt}")


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


# ------------------------------------------------------------- raw entry points


def snack_query_sizes(out_f: int, in_f: int, nnz: int, max_batch: int, val_t: int, act_t: int):
    p, w = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("snack_query_sizes",
           load().snack_query_sizes(out_f, in_f, nnz, max_batch, val_t, act_t, ctypes.byref(p), ctypes.byref(w)))
    return p.value, w.value


def snack_create(out_f: int, in_f: int, nnz: int, max_batch: int, val_t: int, act_t: int, row, col,
                 plan: torch.Tensor, ws: torch.Tensor, validate: bool = False, stream=None) -> int:
    h = ctypes.c_void_p(0)
    _check("snack_create",
           load().snack_create(ctypes.byref(h), out_f, in_f, nnz, max_batch, val_t, act_t, _ptr(row), _ptr(col),
                               _ptr(plan), _nbytes(plan), _ptr(ws), _nbytes(ws), 1 if validate else 0,
                               _stream(stream)))
    return h.value


def snack_spmm_fwd(h: int, row, col, val, x, batch: int, bias, y, ws, stream=None) -> None:
    _check("snack_spmm_fwd",
           load().snack_spmm_fwd(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), _ptr(x), batch, _ptr(bias),
                                 _ptr(y), _ptr(ws), 0 if ws is None else _nbytes(ws), _stream(stream)))


def snack_spmm_fwd_noalloc(h: int, row, col, val, x, batch: int, bias, y, stream=None) -> None:
    """Forward pass using the library's built-in scratch array (no workspace argument)."""
    _check("snack_spmm_fwd_noalloc",
           load().snack_spmm_fwd_noalloc(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), _ptr(x), batch,
                                         _ptr(bias), _ptr(y), _stream(stream)))


def snack_spmm_dx(h: int, row, col, val, dy, batch: int, dx, ws, stream=None) -> None:
    _check("snack_spmm_dx",
           load().snack_spmm_dx(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), _ptr(dy), batch, _ptr(dx),
                                _ptr(ws), 0 if ws is None else _nbytes(ws), _stream(stream)))


def snack_spmm_fwd_gelu(h: int, row, col, val, x, batch: int, bias, y_pre, y, ws, stream=None) -> None:
    _check("snack_spmm_fwd_gelu",
           load().snack_spmm_fwd_gelu(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), _ptr(x), batch, _ptr(bias),
                                      _ptr(y_pre), _ptr(y), _ptr(ws), 0 if ws is None else _nbytes(ws), _stream(stream)))


def snack_spmm_dx_gelu(h: int, row, col, val, dy, batch: int, x_pre, dx, ws, stream=None) -> None:
    _check("snack_spmm_dx_gelu",
           load().snack_spmm_dx_gelu(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), _ptr(dy), batch,
                                     _ptr(x_pre), _ptr(dx), _ptr(ws), 0 if ws is None else _nbytes(ws),
                                     _stream(stream)))


def snack_sddmm_dw(h: int, row, col, x, dy, batch: int, dw, db, ws, stream=None) -> None:
    _check("snack_sddmm_dw",
           load().snack_sddmm_dw(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(x), _ptr(dy), batch, _ptr(dw),
                                 _ptr(db), _ptr(ws), 0 if ws is None else _nbytes(ws), _stream(stream)))


def snack_backward(h: int, row, col, val, x, dy, batch: int, dx, dw, db, ws, stream=None) -> None:
    _check("snack_backward",
           load().snack_backward(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), _ptr(x), _ptr(dy), batch,
                                 _ptr(dx), _ptr(dw), _ptr(db), _ptr(ws), 0 if ws is None else _nbytes(ws),
                                 _stream(stream)))


def snack_restructure_workspace_size(h: int, n_prune: int) -> int:
    b = ctypes.c_size_t(0)
    _check("snack_restructure_workspace_size",
           load().snack_restructure_workspace_size(ctypes.c_void_p(h), n_prune, ctypes.byref(b)))
    return b.value


def snack_restructure(h: int, row, col, val, n_prune: int, seed: int, step: int, row_out, col_out, val_out,
                      src_out, ws, stream=None) -> None:
    _check("snack_restructure",
           load().snack_restructure(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), n_prune,
                                    seed & (2**64 - 1), step & (2**64 - 1), _ptr(row_out), _ptr(col_out),
                                    _ptr(val_out), _ptr(src_out), _ptr(ws), _nbytes(ws), _stream(stream)))


def snack_restructure_rows_workspace_size(h: int, n_per_row: int) -> int:
    b = ctypes.c_size_t(0)
    _check("snack_restructure_rows_workspace_size",
           load().snack_restructure_rows_workspace_size(ctypes.c_void_p(h), n_per_row, ctypes.byref(b)))
    return b.value


def snack_restructure_rows(h: int, row, col, val, n_per_row: int, seed: int, step: int, row_out, col_out, val_out,
                           src_out, ws, stream=None) -> None:
    _check("snack_restructure_rows",
           load().snack_restructure_rows(ctypes.c_void_p(h), _ptr(row), _ptr(col), _ptr(val), n_per_row,
                                         seed & (2**64 - 1), step & (2**64 - 1), _ptr(row_out), _ptr(col_out),
                                         _ptr(val_out), _ptr(src_out), _ptr(ws), _nbytes(ws), _stream(stream)))


def snack_wait_plan(h: int, stream=None) -> None:
    _check("snack_wait_plan", load().snack_wait_plan(ctypes.c_void_p(h), _stream(stream)))


def snack_destroy(h: int) -> None:
    load().snack_destroy(ctypes.c_void_p(h))


def snack_status_string(status: int) -> str:
    return load().snack_status_string(status).decode()


def snack_trace_start(capacity: int) -> None:
    _check("snack_trace_start", load().snack_trace_start(capacity))


def snack_trace_read(max_records: int) -> list:
    """The last records of the calling thread's trace, oldest first: (kernel name, microseconds)."""
    names = (ctypes.c_char_p * max(max_records, 1))()
    us = (ctypes.c_float * max(max_records, 1))()
    n = ctypes.c_int32(0)
    _check("snack_trace_read", load().snack_trace_read(names, us, max_records, ctypes.byref(n)))
    return [(names[i].decode(), float(us[i])) for i in range(n.value)]


def snack_trace_stop() -> None:
    _check("snack_trace_stop", load().snack_trace_stop())


def snack_version() -> int:
    return int(load().snack_version())


# ------------------------------------------------------------- layer owner


class SparseLinear:
    """One truly sparse layer on the GPU: Y = X W^T + b over the stored weights.

    row/col: int32 CUDA tensors (row-sorted COO, strictly increasing in
    (row, col)); val: float32 or bfloat16 CUDA tensor; bias: float32 or None.
    The plan and workspace are torch CUDA tensors owned by this object.
    """

    def __init__(self, out_f: int, in_f: int, row: torch.Tensor, col: torch.Tensor, val: torch.Tensor,
                 bias: Optional[torch.Tensor] = None, max_batch: int = 1024, validate: bool = False,
                 stream=None):
        if not (row.is_cuda and col.is_cuda and val.is_cuda):
            raise ValueError("row, col and val must be CUDA tensors")
        if row.dtype != torch.int32 or col.dtype != torch.int32:
            raise ValueError("row and col must be int32")
        self.out_f, self.in_f = int(out_f), int(in_f)
        self.row, self.col, self.val = row.contiguous(), col.contiguous(), val.contiguous()
        self.bias = None if bias is None else bias.contiguous().float()
        self.nnz = int(self.row.numel())
        self.max_batch = int(max_batch)
        self.dtype = val.dtype
        code = dtype_code(val.dtype)
        plan_b, ws_b = snack_query_sizes(self.out_f, self.in_f, self.nnz, self.max_batch, code, code)
        dev = val.device
        self.plan = torch.empty(plan_b, dtype=torch.uint8, device=dev)
        self.ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
        self.handle = snack_create(self.out_f, self.in_f, self.nnz, self.max_batch, code, code, self.row, self.col,
                                   self.plan, self.ws, validate, stream)

    def close(self) -> None:
        if getattr(self, "handle", None):
            snack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        x = x.contiguous()
        y = out if out is not None else torch.empty((x.shape[0], self.out_f), dtype=self.dtype, device=x.device)
        snack_spmm_fwd(self.handle, self.row, self.col, self.val, x, x.shape[0], self.bias, y, self.ws, stream)
        return y

    def forward_gelu(self, x: torch.Tensor, keep_pre: bool = True, stream=None):
        """GELU(x W^T + b); returns (y, pre) with pre None unless keep_pre."""
        x = x.contiguous()
        y = torch.empty((x.shape[0], self.out_f), dtype=self.dtype, device=x.device)
        pre = torch.empty_like(y) if keep_pre else None
        snack_spmm_fwd_gelu(self.handle, self.row, self.col, self.val, x, x.shape[0], self.bias, pre, y, self.ws,
                            stream)
        return y, pre

    def grad_input_gelu(self, dy: torch.Tensor, x_pre: torch.Tensor, stream=None) -> torch.Tensor:
        """(dy W) * GELU'(x_pre): the gradient at the pre-activation of this layer's input."""
        dy, x_pre = dy.contiguous(), x_pre.contiguous()
        dx = torch.empty((dy.shape[0], self.in_f), dtype=self.dtype, device=dy.device)
        snack_spmm_dx_gelu(self.handle, self.row, self.col, self.val, dy, dy.shape[0], x_pre, dx, self.ws, stream)
        return dx

    def grad_input(self, dy: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        dy = dy.contiguous()
        dx = out if out is not None else torch.empty((dy.shape[0], self.in_f), dtype=self.dtype, device=dy.device)
        snack_spmm_dx(self.handle, self.row, self.col, self.val, dy, dy.shape[0], dx, self.ws, stream)
        return dx

    def grad_weight(self, x: torch.Tensor, dy: torch.Tensor, want_db: bool = True, stream=None):
        x, dy = x.contiguous(), dy.contiguous()
        dw = torch.empty(self.nnz, dtype=torch.float32, device=x.device)
        db = torch.empty(self.out_f, dtype=torch.float32, device=x.device) if want_db else None
        snack_sddmm_dw(self.handle, self.row, self.col, x, dy, x.shape[0], dw, db, self.ws, stream)
        return dw, db

    def backward(self, x: torch.Tensor, dy: torch.Tensor, want_db: bool = True, stream=None):
        """(dX, dW, db) in one call (fused single pass when the batch fits one tile)."""
        x, dy = x.contiguous(), dy.contiguous()
        dx = torch.empty((dy.shape[0], self.in_f), dtype=self.dtype, device=dy.device)
        dw = torch.empty(self.nnz, dtype=torch.float32, device=x.device)
        db = torch.empty(self.out_f, dtype=torch.float32, device=x.device) if want_db else None
        snack_backward(self.handle, self.row, self.col, self.val, x, dy, x.shape[0], dx, dw, db, self.ws, stream)
        return dx, dw, db

    def restructure(self, n_prune: int, seed: int, step: int, stream=None) -> torch.Tensor:
        """Prune/regrow in place of this layer's pattern; returns src index (-1 = regrown)."""
        need = snack_restructure_workspace_size(self.handle, n_prune)
        ws = self.ws if need <= _nbytes(self.ws) else torch.empty(need, dtype=torch.uint8, device=self.val.device)
        row_o = torch.empty_like(self.row)
        col_o = torch.empty_like(self.col)
        val_o = torch.empty_like(self.val)
        src_o = torch.empty_like(self.row)
        snack_restructure(self.handle, self.row, self.col, self.val, n_prune, seed, step, row_o, col_o, val_o,
                          src_o, ws, stream)
        self.row, self.col, self.val = row_o, col_o, val_o
        return src_o

    def restructure_rows(self, n_per_row: int, seed: int, step: int, stream=None) -> torch.Tensor:
        """Per-row (constant fan-in) prune/regrow in place; returns src index (-1 = regrown)."""
        need = snack_restructure_rows_workspace_size(self.handle, n_per_row)
        ws = self.ws if need <= _nbytes(self.ws) else torch.empty(need, dtype=torch.uint8, device=self.val.device)
        row_o = torch.empty_like(self.row)
        col_o = torch.empty_like(self.col)
        val_o = torch.empty_like(self.val)
        src_o = torch.empty_like(self.row)
        snack_restructure_rows(self.handle, self.row, self.col, self.val, n_per_row, seed, step, row_o, col_o, val_o,
                               src_o, ws, stream)
        self.row, self.col, self.val = row_o, col_o, val_o
        return src_o


class _SparseLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, val, layer: SparseLinear):
        if val.data_ptr() != layer.val.data_ptr():
            raise ValueError("val must be the layer's value tensor")
        ctx.layer = layer
        ctx.save_for_backward(x)
        return layer.forward(x)

    @staticmethod
    def backward(ctx, dy):
        (x,) = ctx.saved_tensors
        layer = ctx.layer
        dy = dy.contiguous().to(layer.dtype)
        dx = layer.grad_input(dy) if ctx.needs_input_grad[0] else None
        dw = layer.grad_weight(x, dy, want_db=False)[0] if ctx.needs_input_grad[1] else None
        if dw is not None and layer.dtype != torch.float32:
            dw = dw.to(layer.dtype)
        return dx, dw, None


def sparse_linear(x: torch.Tensor, layer: SparseLinear) -> torch.Tensor:
    """Autograd-aware Y = X W^T + b; gradients flow to x and to layer.val."""
    return _SparseLinearFn.apply(x, layer.val, layer)
