"""Helpers for the GPU parity tests: move seeded inputs to the device, read
results back as float64, and compare against the oracle with a T-scaled bound."""

import numpy as np
import torch

from spmm_row_sorted_gb300 import workloads as wl

# The stated contract: |gpu - oracle| <= REL * T per output, T = sum of
# |terms| (bias included); 1e-5 for fp32, 2e-3 for bf16 storage.
REL = {"f32": 1e-5, "bf16": 2e-3}
# The bound the tests apply is tighter and follows the kernels' arithmetic:
# every kernel widens bf16 inputs to fp32 exactly (a bf16 value is an fp32
# value with a shorter significand) and accumulates in fp32, so the sums meet
# the fp32 bound 1e-5 * T whatever the storage type.  The products of two
# bf16 values are exact in fp32 too, so the tensor-core path of moderately
# sparse bf16 layers meets the same bound.
ACC_REL = 1e-5
# An output stored in bf16 is that fp32 sum s rounded once to nearest-even:
# |bf16(s) - s| <= half an ulp of bf16 at |s| (8 significant bits), and
# |s| <= |y| + ACC_REL * T, so |bf16(s) - y| <= ACC_REL * T + half_ulp(|y| + ACC_REL * T).
# A result rounded twice (e.g. a bf16 sum with a bias added afterwards) can
# be a whole ulp off and fails this bound.
BF16_STORE = 2.0 ** -8  # half_ulp(v) <= 2^-8 v


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half the spacing of bfloat16 numbers at magnitude v >= 0 (subnormal spacing below 2^-126)."""
    v = np.asarray(v, dtype=np.float64)
    _, ex = np.frexp(v)  # v = m * 2^ex, m in [0.5, 1): the leading bit is 2^(ex - 1)
    lead = np.maximum(ex - 1, -126)
    return np.ldexp(1.0, lead - 8)


def act_tensor(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def layer_tensors(layer: wl.Layer, device="cuda"):
    row = torch.from_numpy(layer.row).to(device)
    col = torch.from_numpy(layer.col).to(device)
    val = act_tensor(layer.val, layer.val_dtype, device)
    bias = torch.from_numpy(layer.bias).to(device)
    return row, col, val, bias


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw stored bits of a float32 / bfloat16 tensor (for bit-exact checks)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


def assert_close_T(got: np.ndarray, ref: np.ndarray, T: np.ndarray, rel: float, what: str,
                   stored_bf16: bool = False):
    """|got - ref| <= rel*T, plus half a bf16 ulp at |ref| + rel*T when got was rounded once to bf16."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = rel * T
    if stored_bf16:
        bound = bound + bf16_half_ulp(np.abs(ref) + rel * T)
    bad = ~(err <= bound)
    both_nan = np.isnan(got) & np.isnan(ref)
    bad &= ~both_nan
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = float(np.nanmax(err / np.maximum(T, 1e-300)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} outside {rel}*T; worst err/T {worst:.3e}; "
                             f"first {idx.tolist()} got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
