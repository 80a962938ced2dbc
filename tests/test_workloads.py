"""Seeded input generator: sizes, sortedness, value recipes (CPU only)."""

import numpy as np
import pytest

from spmm_row_sorted_gb300 import workloads as w


def test_nnz_rounding_matches_configs():
    assert w.nnz_for(1024, 1024, 0.05) == 52429
    assert w.nnz_for(4096, 4096, 0.10) == 1677722
    assert w.nnz_for(3072, 768, 0.01) == 23593
    assert w.nnz_for(16384, 16384, 0.01) == 2684355
    assert w.nnz_for(8192, 8192, 0.50) == 33554432


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    a = np.concatenate([np.random.default_rng(0).standard_normal(10000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 3.0e38, -1e-40, 1.00390625, 1.01171875], np.float32)])
    ours = w.bf16_bits_from_f32(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = w.f32_from_bf16_bits(ours)
    assert np.array_equal(back, torch.from_numpy(a).to(torch.bfloat16).float().numpy())


def test_layer_is_row_sorted_and_seeded():
    a = w.config_layer("c1")
    b = w.config_layer("c1")
    assert a.nnz == 52429
    pos = a.row.astype(np.int64) * a.in_f + a.col
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(a.row, b.row) and np.array_equal(a.val, b.val)
    assert abs(a.val.std() - 1 / np.sqrt(52429 / 1024)) < 0.01


def test_zipf_rows():
    counts = w.zipf_row_counts(16384, 16384, 2684355, 1.2)
    assert counts.sum() == 2684355
    assert (counts == 16384).sum() == 36
    assert np.all(np.diff(counts) <= 0)  # non-increasing in rank
    assert 20 <= np.median(counts) <= 30


def test_small_zipf_layer_positions():
    lay = w.make_layer(64, 48, nnz=600, zipf_s=1.2, seed=3)
    pos = lay.row.astype(np.int64) * 48 + lay.col
    assert lay.nnz == 600 and np.all(np.diff(pos) > 0)
    assert lay.row.min() >= 0 and lay.row.max() < 64 and lay.col.max() < 48


@pytest.mark.parametrize("shape", [(64, 64, 5), (48, 200, 7), (300, 40, 40), (1, 9, 3)])
def test_diagonal_layer_positions(shape):
    out_f, in_f, n_diag = shape
    lay = w.make_layer(out_f, in_f, diagonals=n_diag, seed=2)
    pos = lay.row.astype(np.int64) * in_f + lay.col
    assert lay.nnz == out_f * n_diag and np.all(np.diff(pos) > 0)
    # every row holds the same set of offsets (col - row) mod in_f
    offs = ((lay.col.astype(np.int64) - lay.row) % in_f).reshape(out_f, n_diag)
    assert np.all(np.sort(offs, axis=1) == np.sort(offs[0]))
    if out_f == in_f:
        assert np.all(np.bincount(lay.col, minlength=in_f) == n_diag)
