"""The allocation-free forward entry point, snack_spmm_fwd_noalloc.

Some callers cannot allocate device memory where they call the forward pass:
a plugin run from an inference engine's enqueue step, or a real-time loop
whose memory is fixed at start-up.  They cannot pass the workspace that
snack_spmm_fwd takes, so this entry point uses a scratch array built into the
library instead.  The tests call it through the C ABI twice in a row and check
that both results are bit-identical to the workspace entry point's (the same
kernels run on the same inputs) and within the parity bound of the oracle;
that a moderately sparse bf16 layer, which takes the tensor-core path, also
matches the oracle; and that a call needing more than the built-in scratch is
rejected before anything is launched.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from spmm_row_sorted_gb300 import build as snack_build
from spmm_row_sorted_gb300 import snack
from spmm_row_sorted_gb300 import workloads as wl

from gpu_util import ACC_REL, act_tensor, assert_close_T, f64, layer_tensors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    snack_build.build()
    return snack.load()


def call_noalloc(lib, L, row, col, val, x, batch, bias, y):
    stream = torch.cuda.current_stream()
    return lib.snack_spmm_fwd_noalloc(ctypes.c_void_p(L.handle), ctypes.c_void_p(row.data_ptr()),
                                      ctypes.c_void_p(col.data_ptr()), ctypes.c_void_p(val.data_ptr()),
                                      ctypes.c_void_p(x.data_ptr()), batch, ctypes.c_void_p(bias.data_ptr()),
                                      ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("dtype,batch,density", [("f32", 32, None), ("bf16", 16, None), ("bf16", 64, 0.5)])
def test_noalloc_matches_workspace_entry_point(lib, dtype, batch, density):
    out_f, in_f = (700, 900) if density is None else (704, 896)
    if density is None:
        lay = wl.make_layer(out_f, in_f, nnz=40000, zipf_s=1.1, val_std=0.3, val_dtype=dtype, seed=5, bias="normal")
    else:  # half of W stored, bf16, batch >= 32: the moderately sparse (tensor-core) path
        lay = wl.make_layer(out_f, in_f, density=density, val_std=0.1, val_dtype=dtype, seed=5, bias="normal")
    acts = wl.make_acts(batch, in_f, out_f, dtype, seed=5)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=batch)
    x = act_tensor(acts.x, dtype)
    y_ws = L.forward(x)
    outs = []
    for _ in range(2):  # two calls in a row share the built-in scratch
        y = torch.full_like(y_ws, float("nan"))
        st = call_noalloc(lib, L, row, col, val, x, batch, bias, y)
        assert st == 0, snack.snack_status_string(st)
        outs.append(y)
    torch.cuda.synchronize()
    ref, t = oracle.fwd(out_f, in_f, lay.row, lay.col, oracle.as_f64(lay.val, dtype), oracle.as_f64(acts.x, dtype),
                        oracle.as_f64(lay.bias))
    assert_close_T(f64(y_ws), ref, t, ACC_REL, "workspace fwd", stored_bf16=dtype == "bf16")
    for y in outs:  # the same kernels on the same inputs: bit-identical
        assert torch.equal(y, y_ws), "noalloc differs from the workspace entry point"
        assert_close_T(f64(y), ref, t, ACC_REL, "noalloc fwd", stored_bf16=dtype == "bf16")
    L.close()


def test_noalloc_rejects_calls_beyond_the_scratch(lib):
    # in_f * batch * 4 bytes of transposed activations alone exceed 32 MiB
    out_f, in_f, batch = 64, 16384, 1024
    lay = wl.make_layer(out_f, in_f, nnz=5000, val_dtype="f32", seed=1)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=batch)
    x = torch.zeros((batch, in_f), device="cuda")
    y = torch.full((batch, out_f), 7.0, device="cuda")
    with pytest.raises(snack.SnackError) as e:
        snack.snack_spmm_fwd_noalloc(L.handle, row, col, val, x, batch, bias, y)
    assert e.value.status == 4  # SNACK_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)  # nothing was launched
    # a call that fits still works on the same handle
    xs = act_tensor(wl.make_acts(8, in_f, out_f, "f32").x, "f32")
    ys = torch.empty((8, out_f), device="cuda")
    snack.snack_spmm_fwd_noalloc(L.handle, row, col, val, xs, 8, bias, ys)
    torch.cuda.synchronize()
    assert torch.equal(ys, L.forward(xs))
    L.close()
