"""Helpers for the GPU parity tests: move seeded inputs to the device, read
results back as float64, and compare against the oracle with a T-scaled bound."""

import numpy as np
import torch

from spmm_row_sorted_gb300 import workloads as wl

# |gpu - oracle| <= REL * T per output, T = sum of |terms| (bias included).
REL = {"f32": 1e-5, "bf16": 2e-3}
# An output stored in bf16 is rounded once to nearest-even on top of that:
# |bf16(y) - y| <= 2^-8 |y| (bf16 keeps 8 significant bits).
BF16_STORE = 2.0 ** -8


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
    """|got - ref| <= rel*T (+ 2^-8 |ref| when got was stored in bf16)."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = rel * T
    if stored_bf16:
        bound = bound + BF16_STORE * np.abs(ref)
    bad = ~(err <= bound)
    both_nan = np.isnan(got) & np.isnan(ref)
    bad &= ~both_nan
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = float(np.nanmax(err / np.maximum(T, 1e-300)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} outside {rel}*T; worst err/T {worst:.3e}; "
                             f"first {idx.tolist()} got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
