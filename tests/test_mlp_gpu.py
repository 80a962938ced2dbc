"""GPU parity of the sparse MLP training step (768 -> 3072 -> GELU -> 768, 99 %
sparse, 1024 tokens): forward with the fused GELU epilogue, backward through
GELU' fused into the second layer's input gradient, and both weight
gradients.  Each op is checked against the oracle on the inputs that op
received (the GPU's own activations), so errors do not compound; a final
check compares the whole chain with the all-fp64 oracle chain.

Bounds: a GELU output is GELU(s) of an fp32 sum within 1e-5*T of the exact
pre-activation, and |GELU'| <= 1.13, so |gpu - ref| <= 1.13e-5*T + 1e-6*|ref|
(the second term covers the fp32 evaluation of erf); likewise for the
GELU'-scaled input gradient.
"""

import numpy as np
import pytest
import torch

import oracle
from spmm_row_sorted_gb300 import build as snack_build
from spmm_row_sorted_gb300 import snack
from spmm_row_sorted_gb300 import workloads as wl

from gpu_util import ACC_REL, act_tensor, assert_close_T, bf16_half_ulp, f64, layer_tensors

pytestmark = pytest.mark.gpu
GELU_SLOPE = 1.13


@pytest.fixture(scope="module", autouse=True)
def built():
    snack_build.build()
    snack.load()
    oracle.set_threads(8)


def make(lay, max_batch):
    row, col, val, bias = layer_tensors(lay)
    return snack.SparseLinear(lay.out_f, lay.in_f, row, col, val, bias, max_batch=max_batch, validate=True)


def gelu_bound(t, ref):
    return GELU_SLOPE * 1e-5 * t + 1e-6 * np.abs(ref)


def check_gelu_close(got, ref, t, what):
    err = np.abs(got - ref)
    bound = gelu_bound(t, ref)
    assert np.all(err <= bound), f"{what}: worst err/bound {float(np.max(err / np.maximum(bound, 1e-300))):.3f}"


@pytest.mark.parametrize("batch", [1024, 37, 8, 3])
def test_sparse_mlp_training_step(batch):
    l1 = wl.config_layer("c3", layer_index=0)  # 3072 x 768
    l2 = wl.config_layer("c3", layer_index=1)  # 768 x 3072
    l1.bias = wl.random_normal(l1.out_f, 3, 1, 0.1)
    l2.bias = wl.random_normal(l2.out_f, 3, 2, 0.1)
    x_np = wl.make_acts(batch, 768, 3072, "f32", seed=5).x
    dy2_np = wl.make_acts(batch, 3072, 768, "f32", seed=6).dy
    L1, L2 = make(l1, batch), make(l2, batch)
    x = act_tensor(x_np, "f32")
    dy2 = act_tensor(dy2_np, "f32")

    h, pre1 = L1.forward_gelu(x)
    y2 = L2.forward(h)
    dy1 = L2.grad_input_gelu(dy2, pre1)  # gradient at layer 1's pre-activation
    dx = L1.grad_input(dy1)
    dw2, db2 = L2.grad_weight(h, dy2)
    dw1, db1 = L1.grad_weight(x, dy1)
    torch.cuda.synchronize()

    v1, v2 = oracle.as_f64(l1.val), oracle.as_f64(l2.val)
    b1, b2 = oracle.as_f64(l1.bias), oracle.as_f64(l2.bias)
    x64, dy2_64 = oracle.as_f64(x_np), oracle.as_f64(dy2_np)
    # layer 1 forward: pre-activation and GELU
    p_ref, t1 = oracle.fwd(l1.out_f, l1.in_f, l1.row, l1.col, v1, x64, b1)
    assert_close_T(f64(pre1), p_ref, t1, 1e-5, "pre1")
    check_gelu_close(f64(h), oracle.gelu(p_ref), t1, "gelu(pre1)")
    # layer 2 forward on the GPU's h
    h64 = f64(h)
    y_ref, t2 = oracle.fwd(l2.out_f, l2.in_f, l2.row, l2.col, v2, h64, b2)
    assert_close_T(f64(y2), y_ref, t2, 1e-5, "y2")
    # layer 2 input gradient times GELU'(pre1)
    g_ref, tg = oracle.dx(l2.out_f, l2.in_f, l2.row, l2.col, v2, dy2_64)
    gp = oracle.gelu_grad(f64(pre1))
    # s * GELU'(pre): the fp32 sum s is within 1e-5*tg, and GELU' evaluated in
    # fp32 is within a few ulp of its terms (bounded by 2e-7 * |s| <= 2e-7 * tg)
    err = np.abs(f64(dy1) - g_ref * gp)
    bound = 1e-5 * tg * np.abs(gp) + 2e-7 * tg + 1e-6 * np.abs(g_ref * gp)
    assert np.all(err <= bound), float(np.max(err / bound))
    # layer 1 input gradient on the GPU's dy1
    dy1_64 = f64(dy1)
    dx_ref, tx = oracle.dx(l1.out_f, l1.in_f, l1.row, l1.col, v1, dy1_64)
    assert_close_T(f64(dx), dx_ref, tx, 1e-5, "dx")
    # weight and bias gradients
    d2, td2, db2_ref = oracle.dw(l2.out_f, l2.in_f, l2.row, l2.col, h64, dy2_64)
    assert_close_T(f64(dw2), d2, td2, 1e-5, "dw2")
    assert_close_T(f64(db2), db2_ref, np.abs(dy2_64).sum(0), 1e-5, "db2")
    d1, td1, db1_ref = oracle.dw(l1.out_f, l1.in_f, l1.row, l1.col, x64, dy1_64)
    assert_close_T(f64(dw1), d1, td1, 1e-5, "dw1")
    assert_close_T(f64(db1), db1_ref, np.abs(dy1_64).sum(0), 1e-5, "db1")
    # whole chain against the all-fp64 chain (errors compound; loose relative check)
    full = oracle.mlp_step((l1.out_f, l1.in_f, l1.row, l1.col, v1, b1), (l2.out_f, l2.in_f, l2.row, l2.col, v2, b2),
                           x64, dy2_64)
    for name, got in (("y2", y2), ("dx", dx), ("dw1", dw1), ("dw2", dw2)):
        ref = full[name]
        assert np.max(np.abs(f64(got) - ref)) <= 1e-4 * np.max(np.abs(ref)), name
    L1.close()
    L2.close()


@pytest.mark.parametrize("batch", [16, 4])
def test_gelu_epilogue_bf16_and_no_pre(batch):
    lay = wl.make_layer(300, 200, nnz=6000, val_std=0.2, val_dtype="bf16", seed=8, bias="normal")
    acts = wl.make_acts(batch, 200, 300, "bf16", seed=8)
    L = make(lay, batch)
    x = act_tensor(acts.x, "bf16")
    y, pre = L.forward_gelu(x, keep_pre=False)
    assert pre is None
    y_plain = L.forward(x)
    torch.cuda.synchronize()
    p_ref, t = oracle.fwd(300, 200, lay.row, lay.col, oracle.as_f64(lay.val, "bf16"), oracle.as_f64(acts.x, "bf16"),
                          oracle.as_f64(lay.bias))
    ref = oracle.gelu(p_ref)
    err = np.abs(f64(y) - ref)
    # GELU of an fp32 sum within 1e-5*T, evaluated in fp32, rounded once to bf16
    slack = GELU_SLOPE * ACC_REL * t + 1e-6 * np.abs(ref)
    bound = slack + bf16_half_ulp(np.abs(ref) + slack)
    assert np.all(err <= bound), float(np.max(err / bound))
    # the plain forward is the pre-activation
    assert_close_T(f64(y_plain), p_ref, t, ACC_REL, "plain", stored_bf16=True)
    L.close()
