"""Pins of the CPU oracle to facts outside itself (CPU only).

The SNACK abstract ("Beyond Masked Sparsity", abstract) gives the operations
by name only: a layer that stores and computes only its non-zero connections,
sparse back-propagation and connection restructuring.  So the oracle is pinned
to mathematics instead of printed values:

* dense brute force: the sparse forward/backward equal a dense fp64 GEMM with
  the densified W (numpy matmul), on tiny shapes and on every 3x3 pattern;
* 0 % sparsity equals torch's fp64 matmul;
* identity W returns X and dY exactly;
* central finite differences of L = sum(G * Y) give dW and dX;
* linearity and adjointness <dY, W X> = <dX, X> = <dW, val>;
* GELU: Phi(1) from the normal table, torch's exact GELU, an odd-part identity;
* restructure: invariants that fix the pruned set uniquely, regrown positions
  that were empty and distinct, exhaustive 3x3 patterns, SplitMix64 known
  answers, the multiply-high reduction against a shift, and a chi-square test
  of uniformity over empty positions.
"""

import itertools
import math
import os

import numpy as np
import pytest

import oracle
from spmm_row_sorted_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_pattern(rng, out_f, in_f, nnz):
    p = np.sort(rng.choice(out_f * in_f, size=nnz, replace=False))
    return (p // in_f).astype(np.int32), (p % in_f).astype(np.int32)


def densify(out_f, in_f, row, col, val):
    w = np.zeros((out_f, in_f))
    w[row, col] = val
    return w


def check_close(a, ref, t, rel):
    assert a.shape == ref.shape
    err = np.abs(a - ref)
    bound = rel * t + 1e-300
    assert np.all(err <= bound), float(np.max(err / np.maximum(t, 1e-300)))


# ---------------------------------------------------------------- fwd/dx/dw


@pytest.mark.parametrize("out_f", [1, 2, 3, 7, 33])
@pytest.mark.parametrize("in_f", [1, 2, 3, 7, 33])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_dense_brute_force_tiny(out_f, in_f, batch):
    rng = np.random.default_rng(out_f * 1000 + in_f * 10 + batch)
    for nnz in sorted({0, 1, (out_f * in_f) // 3, out_f * in_f}):
        row, col = rand_pattern(rng, out_f, in_f, nnz)
        val = rng.standard_normal(nnz)
        bias = rng.standard_normal(out_f)
        x = rng.standard_normal((batch, in_f))
        dy = rng.standard_normal((batch, out_f))
        w = densify(out_f, in_f, row, col, val)
        y, t = oracle.fwd(out_f, in_f, row, col, val, x, bias)
        check_close(y, x @ w.T + bias, t, 1e-14)
        g, tg = oracle.dx(out_f, in_f, row, col, val, dy)
        check_close(g, dy @ w, tg, 1e-14)
        d, td, db = oracle.dw(out_f, in_f, row, col, x, dy)
        check_close(d, (dy.T @ x)[row, col], td, 1e-14)
        np.testing.assert_allclose(db, dy.sum(axis=0), rtol=1e-14, atol=1e-14)


def test_every_3x3_pattern():
    rng = np.random.default_rng(7)
    pos = np.arange(9)
    x = rng.standard_normal((4, 3))
    dy = rng.standard_normal((4, 3))
    bias = rng.standard_normal(3)
    for mask in range(512):
        p = pos[[(mask >> i) & 1 == 1 for i in range(9)]]
        row, col = (p // 3).astype(np.int32), (p % 3).astype(np.int32)
        val = rng.standard_normal(p.size)
        w = densify(3, 3, row, col, val)
        y, t = oracle.fwd(3, 3, row, col, val, x, bias)
        check_close(y, x @ w.T + bias, t, 1e-14)
        g, tg = oracle.dx(3, 3, row, col, val, dy)
        check_close(g, dy @ w, tg, 1e-14)
        d, td, _ = oracle.dw(3, 3, row, col, x, dy)
        check_close(d, (dy.T @ x)[row, col], td, 1e-14)


def test_zero_sparsity_is_dense_gemm():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    out_f, in_f, batch = 17, 13, 5
    p = np.arange(out_f * in_f)
    row, col = (p // in_f).astype(np.int32), (p % in_f).astype(np.int32)
    val = rng.standard_normal(p.size)
    x = rng.standard_normal((batch, in_f))
    dy = rng.standard_normal((batch, out_f))
    w = torch.tensor(val.reshape(out_f, in_f), dtype=torch.float64)
    xt, dyt = torch.tensor(x), torch.tensor(dy)
    y, t = oracle.fwd(out_f, in_f, row, col, val, x, None)
    check_close(y, torch.nn.functional.linear(xt, w).numpy(), t, 1e-14)
    g, tg = oracle.dx(out_f, in_f, row, col, val, dy)
    check_close(g, (dyt @ w).numpy(), tg, 1e-14)
    d, td, _ = oracle.dw(out_f, in_f, row, col, x, dy)
    check_close(d, (dyt.T @ xt).numpy().reshape(-1), td, 1e-14)


def test_identity_weight():
    rng = np.random.default_rng(11)
    n, batch = 37, 6
    k = np.arange(n, dtype=np.int32)
    x = rng.standard_normal((batch, n))
    dy = rng.standard_normal((batch, n))
    y, _ = oracle.fwd(n, n, k, k, np.ones(n), x, np.zeros(n))
    assert np.array_equal(y, x)
    g, _ = oracle.dx(n, n, k, k, np.ones(n), dy)
    assert np.array_equal(g, dy)
    d, _, _ = oracle.dw(n, n, k, k, x, dy)
    np.testing.assert_allclose(d, np.einsum("bk,bk->k", dy, x), rtol=1e-14)


def test_finite_differences():
    rng = np.random.default_rng(5)
    out_f, in_f, batch, nnz = 9, 11, 4, 30
    row, col = rand_pattern(rng, out_f, in_f, nnz)
    val = rng.standard_normal(nnz)
    bias = rng.standard_normal(out_f)
    x = rng.standard_normal((batch, in_f))
    gy = rng.standard_normal((batch, out_f))  # L = sum(gy * Y)

    def loss(v, xx):
        return float(np.sum(gy * oracle.fwd(out_f, in_f, row, col, v, xx, bias)[0]))

    h = 1e-3
    d, _, db = oracle.dw(out_f, in_f, row, col, x, gy)
    for kk in range(nnz):
        e = np.zeros(nnz)
        e[kk] = h
        fd = (loss(val + e, x) - loss(val - e, x)) / (2 * h)
        assert abs(fd - d[kk]) <= 1e-9 * (1 + abs(d[kk]))
    g, _ = oracle.dx(out_f, in_f, row, col, val, gy)
    for b in range(batch):
        for c in range(in_f):
            e = np.zeros_like(x)
            e[b, c] = h
            fd = (loss(val, x + e) - loss(val, x - e)) / (2 * h)
            assert abs(fd - g[b, c]) <= 1e-9 * (1 + abs(g[b, c]))
    # bias gradient: dL/db_r = sum_b gy[b, r]
    for r in range(out_f):
        bb = np.zeros(out_f)
        bb[r] = h
        lp = float(np.sum(gy * oracle.fwd(out_f, in_f, row, col, val, x, bias + bb)[0]))
        lm = float(np.sum(gy * oracle.fwd(out_f, in_f, row, col, val, x, bias - bb)[0]))
        assert abs((lp - lm) / (2 * h) - db[r]) <= 1e-9 * (1 + abs(db[r]))


def test_linearity_and_adjointness():
    rng = np.random.default_rng(9)
    out_f, in_f, batch, nnz = 40, 25, 7, 200
    row, col = rand_pattern(rng, out_f, in_f, nnz)
    val = rng.standard_normal(nnz)
    bias = rng.standard_normal(out_f)
    x1, x2 = rng.standard_normal((2, batch, in_f))
    dy = rng.standard_normal((batch, out_f))
    a = 1.7
    y12, _ = oracle.fwd(out_f, in_f, row, col, val, a * x1 + x2, bias)
    y1, _ = oracle.fwd(out_f, in_f, row, col, val, x1, bias)
    y2, _ = oracle.fwd(out_f, in_f, row, col, val, x2, bias)
    np.testing.assert_allclose(y12, a * y1 + y2 - a * bias, rtol=1e-12, atol=1e-12)
    y0, _ = oracle.fwd(out_f, in_f, row, col, val, x1, None)
    g, _ = oracle.dx(out_f, in_f, row, col, val, dy)
    d, _, _ = oracle.dw(out_f, in_f, row, col, x1, dy)
    lhs = float(np.sum(dy * y0))
    assert math.isclose(lhs, float(np.sum(g * x1)), rel_tol=1e-12, abs_tol=1e-12)
    assert math.isclose(lhs, float(np.dot(d, val)), rel_tol=1e-12, abs_tol=1e-12)


def test_out_of_range_rejected():
    row = np.array([0, 5], dtype=np.int32)
    col = np.array([0, 0], dtype=np.int32)
    assert oracle.check_coo(3, 3, row, col) == 1
    assert oracle.check_coo(3, 3, np.array([1, 0], np.int32), np.array([0, 0], np.int32)) == 2
    assert oracle.check_coo(3, 3, np.array([1, 1], np.int32), np.array([2, 2], np.int32)) == 2
    with pytest.raises(ValueError):
        oracle.fwd(3, 3, row, col, np.ones(2), np.ones((1, 3)))


# ---------------------------------------------------------------- GELU


def test_gelu_pins():
    torch = pytest.importorskip("torch")
    # GELU(1) = 1 * Phi(1); Phi(1) = 0.8413447460685429 (standard normal table)
    assert abs(float(oracle.gelu(np.array([1.0]))[0]) - 0.8413447460685429) < 1e-15
    xs = np.linspace(-6, 6, 1001)
    ref = torch.nn.functional.gelu(torch.tensor(xs), approximate="none").numpy()
    np.testing.assert_allclose(oracle.gelu(xs), ref, rtol=1e-14, atol=1e-15)
    # x Phi(x) - (-x) Phi(-x) = x (Phi(x) + Phi(-x)) = x
    np.testing.assert_allclose(oracle.gelu(xs) - oracle.gelu(-xs), xs, rtol=1e-13, atol=1e-13)
    h = 1e-5
    fd = (oracle.gelu(xs + h) - oracle.gelu(xs - h)) / (2 * h)
    np.testing.assert_allclose(oracle.gelu_grad(xs), fd, rtol=1e-7, atol=1e-9)
    tx = torch.tensor(xs, requires_grad=True)
    torch.nn.functional.gelu(tx, approximate="none").sum().backward()
    np.testing.assert_allclose(oracle.gelu_grad(xs), tx.grad.numpy(), rtol=1e-13, atol=1e-14)


def test_mlp_step_against_dense_autograd():
    # The sparse MLP step (two sparse layers with GELU between them) against a
    # dense two-layer network in fp64 with the same weights at the stored
    # positions and zeros elsewhere, differentiated by torch autograd for the
    # loss L = sum(dY2 * Y2): every forward value and every gradient the step
    # returns (dW at the stored positions only).
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(17)
    batch, d0, d1, d2 = 5, 9, 14, 7
    layers = []
    for o, i, nnz in ((d1, d0, 60), (d2, d1, 50)):
        p = np.sort(rng.choice(o * i, nnz, replace=False))
        layers.append((o, i, (p // i).astype(np.int32), (p % i).astype(np.int32), rng.standard_normal(nnz),
                       rng.standard_normal(o)))
    x = rng.standard_normal((batch, d0))
    dy2 = rng.standard_normal((batch, d2))
    got = oracle.mlp_step(layers[0], layers[1], x, dy2)

    def dense(lay):
        o, i, r, c, v, b = lay
        w = np.zeros((o, i))
        w[r, c] = v
        return torch.tensor(w, requires_grad=True), torch.tensor(b, requires_grad=True)

    (w1, b1), (w2, b2) = dense(layers[0]), dense(layers[1])
    xt = torch.tensor(x, requires_grad=True)
    y1 = xt @ w1.T + b1
    y1.retain_grad()
    h = torch.nn.functional.gelu(y1, approximate="none")
    h.retain_grad()
    y2 = h @ w2.T + b2
    (torch.tensor(dy2) * y2).sum().backward()
    tol = dict(rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got["y1"], y1.detach().numpy(), **tol)
    np.testing.assert_allclose(got["h"], h.detach().numpy(), **tol)
    np.testing.assert_allclose(got["y2"], y2.detach().numpy(), **tol)
    np.testing.assert_allclose(got["dh"], h.grad.numpy(), **tol)
    np.testing.assert_allclose(got["dy1"], y1.grad.numpy(), **tol)
    np.testing.assert_allclose(got["dx"], xt.grad.numpy(), **tol)
    for name, (o, i, r, c, v, b), w, bb in (("1", layers[0], w1, b1), ("2", layers[1], w2, b2)):
        np.testing.assert_allclose(got["dw" + name], w.grad.numpy()[r, c], **tol)
        np.testing.assert_allclose(got["db" + name], bb.grad.numpy(), **tol)


# ---------------------------------------------------------------- restructure


def test_splitmix64_known_answers():
    with open(os.path.join(GOLDEN, "splitmix64_kat.txt")) as f:
        kat = [int(line, 16) for line in f if line.strip() and not line.startswith("#")]
    gamma = 0x9E3779B97F4A7C15
    for n, want in enumerate(kat, start=1):
        assert oracle.splitmix64_mix((n * gamma) % 2**64) == want


def test_draw_stream_is_splitmix64_from_state_zero():
    # Seed 0 at step 0 gives the base state mix(0 ^ mix(0)) = 0 (the finaliser
    # maps 0 to 0), so draw i must be output i + 1 of SplitMix64 started from
    # state 0 -- the published known answers -- and with n_pos = 2^63 the
    # multiply-high reduction keeps its top 63 bits.  This pins the stream's
    # increment, its one-step offset and its base state.
    with open(os.path.join(GOLDEN, "splitmix64_kat.txt")) as f:
        kat = [int(line, 16) for line in f if line.strip() and not line.startswith("#")]
    assert oracle.regrow_base(0, 0) == 0
    for i, want in enumerate(kat):
        assert oracle.regrow_draw(0, 0, i, 2**63) == want >> 1
        assert oracle.regrow_draw(0, 0, i, 2**64 - 1) == (want * (2**64 - 1)) >> 64


def test_multiply_high_reduction():
    # floor(u * 2^k / 2^64) is u >> (64-k); so draws for n_pos = 2^k are the top
    # bits of draws for n_pos = 2^63, shifted.
    for seed, step in [(0, 0), (1, 7), (2**63 + 5, 12345)]:
        for i in range(200):
            top = oracle.regrow_draw(seed, step, i, 2**63)
            for k in (1, 5, 20, 40):
                assert oracle.regrow_draw(seed, step, i, 2**k) == top >> (63 - k)
            assert oracle.regrow_draw(seed, step, i, 1000) < 1000


def prune_rank_key(v, k):
    return (1 if math.isnan(v) else 0, 0.0 if math.isnan(v) else abs(v), k)


def check_restructure_invariants(out_f, in_f, row, col, val, n_prune, ro, co, so):
    nnz = row.shape[0]
    assert ro.shape[0] == nnz and co.shape[0] == nnz and so.shape[0] == nnz
    pos_old = row.astype(np.int64) * in_f + col
    pos_new = ro.astype(np.int64) * in_f + co
    assert np.all((ro >= 0) & (ro < out_f) & (co >= 0) & (co < in_f))
    assert np.all(np.diff(pos_new) > 0)  # strictly sorted, no duplicates
    surv = so[so >= 0]
    assert np.all(np.diff(surv) > 0)  # survivors keep their order, injective
    assert np.array_equal(pos_new[so >= 0], pos_old[surv])
    assert (so < 0).sum() == n_prune
    pruned = np.setdiff1d(np.arange(nnz), surv)
    assert pruned.size == n_prune
    if n_prune and surv.size:
        worst_pruned = max(prune_rank_key(val[k], k) for k in pruned)
        best_kept = min(prune_rank_key(val[k], k) for k in surv)
        assert worst_pruned < best_kept  # the pruned set is the n_prune smallest (|w|, k)
    grown = pos_new[so < 0]
    assert np.intersect1d(grown, pos_old).size == 0  # regrown only where W was empty


def test_restructure_invariants_random():
    rng = np.random.default_rng(21)
    for trial in range(200):
        out_f = int(rng.integers(1, 20))
        in_f = int(rng.integers(1, 20))
        nnz = int(rng.integers(0, out_f * in_f + 1))
        row, col = rand_pattern(rng, out_f, in_f, nnz)
        val = rng.standard_normal(nnz)
        if nnz and trial % 3 == 0:  # ties and signed zeros
            val = np.round(val)
            val[rng.random(nnz) < 0.3] = -0.0
        if nnz and trial % 7 == 0:
            val[rng.integers(0, nnz)] = np.nan
        n_prune = int(rng.integers(0, min(nnz, out_f * in_f - nnz) + 1))
        ro, co, so, draws = oracle.restructure(out_f, in_f, row, col, val, n_prune, trial, 3)
        assert draws >= n_prune
        check_restructure_invariants(out_f, in_f, row, col, val, n_prune, ro, co, so)


def test_restructure_every_3x3_pattern():
    rng = np.random.default_rng(4)
    for mask in range(512):
        p = np.array([i for i in range(9) if (mask >> i) & 1], dtype=np.int64)
        row, col = (p // 3).astype(np.int32), (p % 3).astype(np.int32)
        val = np.round(rng.standard_normal(p.size) * 2) / 2  # many ties
        for n_prune in range(0, min(p.size, 9 - p.size) + 1):
            ro, co, so, _ = oracle.restructure(3, 3, row, col, val, n_prune, mask, n_prune)
            check_restructure_invariants(3, 3, row, col, val, n_prune, ro, co, so)


def test_restructure_ties_and_nan_order():
    row = np.zeros(6, np.int32)
    col = np.arange(6, dtype=np.int32)
    val = np.array([np.nan, 0.5, -0.5, 0.0, -0.0, 2.0])
    ro, co, so, _ = oracle.restructure(1, 12, row, col, val, 3, 0, 0)
    kept = set(so[so >= 0].tolist())
    # |w| order: 0.0 (k=3), -0.0 (k=4), 0.5 (k=1), -0.5 (k=2), 2.0, NaN
    assert kept == {0, 2, 5}


def test_restructure_errors():
    row = np.array([0, 0], np.int32)
    col = np.array([0, 1], np.int32)
    with pytest.raises(oracle.RestructureError):
        oracle.restructure(1, 2, row, col, np.ones(2), 1, 0, 0)  # no empty position
    with pytest.raises(oracle.RestructureError):
        oracle.restructure(1, 3, row, col, np.ones(2), 3, 0, 0)  # n_prune > nnz
    with pytest.raises(oracle.RestructureError):
        oracle.restructure(1, 3, col, row, np.ones(2), 1, 0, 0)  # not sorted
    with pytest.raises(oracle.RestructureError):
        oracle.restructure(1, 1000, row, col, np.ones(2), 1, 0, 0, max_draws=0)


def test_regrow_uniform_over_empty_positions():
    # 8x8 grid, 16 stored weights, regrow 4: every one of the 48 empty positions
    # must be hit equally often across seeds (chi-square, 47 degrees of freedom).
    rng = np.random.default_rng(99)
    row, col = rand_pattern(rng, 8, 8, 16)
    val = rng.standard_normal(16)
    pos_old = set((row.astype(np.int64) * 8 + col).tolist())
    empty = [p for p in range(64) if p not in pos_old]
    counts = {p: 0 for p in empty}
    n_seeds = 3000
    for seed in range(n_seeds):
        ro, co, so, _ = oracle.restructure(8, 8, row, col, val, 4, seed, 1)
        for p in (ro[so < 0].astype(np.int64) * 8 + co[so < 0]).tolist():
            counts[p] += 1
    obs = np.array([counts[p] for p in empty], dtype=np.float64)
    exp = n_seeds * 4 / len(empty)
    chi2 = float(np.sum((obs - exp) ** 2 / exp))
    # 47 dof: mean 47, sd ~9.7; 110 is beyond p = 1e-6
    assert chi2 < 110, chi2


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(1)
    out_f, in_f, batch, nnz = 50, 60, 9, 700
    row, col = rand_pattern(rng, out_f, in_f, nnz)
    val = rng.standard_normal(nnz)
    x = rng.standard_normal((batch, in_f))
    dy = rng.standard_normal((batch, out_f))
    prev = oracle.get_threads()
    try:
        oracle.set_threads(1)
        a = oracle.fwd(out_f, in_f, row, col, val, x)[0], oracle.dw(out_f, in_f, row, col, x, dy)[0]
        oracle.set_threads(4)
        b = oracle.fwd(out_f, in_f, row, col, val, x)[0], oracle.dw(out_f, in_f, row, col, x, dy)[0]
    finally:
        oracle.set_threads(prev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- per-row (constant fan-in) restructure

def check_rows_invariants(out_f, in_f, row, col, val, n_per_row, ro, co, so):
    nnz = row.shape[0]
    assert np.array_equal(ro, row)  # every row keeps its count and offsets
    rp = np.concatenate([[0], np.cumsum(np.bincount(row, minlength=out_f))]).astype(np.int64)
    for r in range(out_f):
        a, b = rp[r], rp[r + 1]
        n = b - a
        p = min(n_per_row, n)
        cr, sr = co[a:b], so[a:b]
        assert np.all(np.diff(cr) > 0)  # strictly increasing columns in the row
        surv = sr[sr >= 0]
        assert np.all((surv >= a) & (surv < b)) and np.all(np.diff(surv) > 0)
        assert np.array_equal(cr[sr >= 0], col[surv])
        assert (sr < 0).sum() == p
        pruned = np.setdiff1d(np.arange(a, b), surv)
        if p and surv.size:
            assert max(prune_rank_key(val[k], k) for k in pruned) < min(prune_rank_key(val[k], k) for k in surv)
        assert np.intersect1d(cr[sr < 0], col[a:b]).size == 0  # regrown only where the row was empty


def test_rows_one_row_equals_unstructured():
    # row 0's draw stream is the unstructured stream, so a one-row layer must
    # give exactly the unstructured restructure's output
    rng = np.random.default_rng(5)
    for trial in range(100):
        in_f = int(rng.integers(2, 300))
        nnz = int(rng.integers(1, in_f))
        _, col = rand_pattern(rng, 1, in_f, nnz)
        row = np.zeros(nnz, np.int32)
        val = rng.standard_normal(nnz)
        n = int(rng.integers(0, min(nnz, in_f - nnz) + 1))
        a = oracle.restructure(1, in_f, row, col, val, n, trial, 11)
        b = oracle.restructure_rows(1, in_f, row, col, val, n, trial, 11)
        for x, y in zip(a[:3], b[:3]):
            assert np.array_equal(x, y)
        assert a[3] == b[3]


def test_rows_stream_base():
    # base of row r: mix(seed ^ mix(step ^ r*K)); row 0 is the unstructured base
    for seed, step in [(0, 0), (3, 9), (2**64 - 1, 2**40)]:
        assert oracle.row_base(seed, step, 0) == oracle.splitmix64_mix(seed ^ oracle.splitmix64_mix(step))
        k = 0xD1B54A32D192ED03
        for r in (1, 2, 1000):
            want = oracle.splitmix64_mix(seed ^ oracle.splitmix64_mix(step ^ ((r * k) & (2**64 - 1))))
            assert oracle.row_base(seed, step, r) == want


def test_rows_invariants_random():
    rng = np.random.default_rng(33)
    for trial in range(150):
        out_f = int(rng.integers(1, 15))
        in_f = int(rng.integers(2, 25))
        if trial % 2:
            lay = wl.make_layer(out_f, in_f, fan_in=int(rng.integers(0, in_f // 2 + 1)), seed=trial)
            row, col = lay.row, lay.col
        else:
            row, col = rand_pattern(rng, out_f, in_f, int(rng.integers(0, out_f * in_f // 2 + 1)))
        nnz = row.shape[0]
        val = rng.standard_normal(nnz)
        if nnz and trial % 3 == 0:
            val = np.round(val)
            val[rng.random(nnz) < 0.3] = -0.0
        if nnz and trial % 5 == 0:
            val[rng.integers(0, nnz)] = np.nan
        lens = np.bincount(row, minlength=out_f)
        room = int(np.min(in_f - lens)) if out_f else 0
        n = int(rng.integers(0, room + 1))
        ro, co, so, draws = oracle.restructure_rows(out_f, in_f, row, col, val, n, trial, 2)
        check_rows_invariants(out_f, in_f, row, col, val, n, ro, co, so)


def test_rows_every_3x3_pattern():
    rng = np.random.default_rng(8)
    for mask in range(512):
        p = np.array([i for i in range(9) if (mask >> i) & 1], dtype=np.int64)
        row, col = (p // 3).astype(np.int32), (p % 3).astype(np.int32)
        val = np.round(rng.standard_normal(p.size) * 2) / 2
        lens = np.bincount(row, minlength=3)
        for n in range(0, 4):
            if np.any(np.minimum(n, lens) > 3 - lens):
                with pytest.raises(oracle.RestructureError):
                    oracle.restructure_rows(3, 3, row, col, val, n, mask, n)
                continue
            ro, co, so, _ = oracle.restructure_rows(3, 3, row, col, val, n, mask, n)
            check_rows_invariants(3, 3, row, col, val, n, ro, co, so)


def test_rows_are_independent():
    # a row's output depends on that row only (its values, columns and index)
    rng = np.random.default_rng(2)
    lay = wl.make_layer(12, 40, fan_in=10, seed=4)
    val = rng.standard_normal(lay.nnz)
    a = oracle.restructure_rows(12, 40, lay.row, lay.col, val, 3, 6, 1)
    val2 = val.copy()
    val2[lay.row == 5] = rng.standard_normal(10)
    b = oracle.restructure_rows(12, 40, lay.row, lay.col, val2, 3, 6, 1)
    other = lay.row != 5
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x[other], y[other])


def test_rows_regrow_uniform_within_row():
    # one row of 16 columns holding 6: each regrown column is uniform over the 10 empty ones
    row = np.zeros(6, np.int32)
    col = np.array([0, 3, 4, 8, 11, 15], np.int32)
    val = np.arange(1.0, 7.0)
    empty = [c for c in range(16) if c not in set(col.tolist())]
    counts = dict.fromkeys(empty, 0)
    n_seeds = 4000
    for seed in range(n_seeds):
        ro, co, so, _ = oracle.restructure_rows(1, 16, row, col, val, 2, seed, 3)
        for c in co[so < 0].tolist():
            counts[c] += 1
    obs = np.array([counts[c] for c in empty], dtype=np.float64)
    exp = n_seeds * 2 / len(empty)
    chi2 = float(np.sum((obs - exp) ** 2 / exp))
    assert chi2 < 45, chi2  # 9 dof: beyond p = 1e-6


def test_rows_errors():
    row = np.array([0, 0, 1], np.int32)
    col = np.array([0, 1, 0], np.int32)
    with pytest.raises(oracle.RestructureError):
        oracle.restructure_rows(2, 2, row, col, np.ones(3), 1, 0, 0)  # row 0 has no empty column
    with pytest.raises(oracle.RestructureError):
        oracle.restructure_rows(2, 3, row, col, np.ones(3), -1, 0, 0)
    with pytest.raises(oracle.RestructureError):
        oracle.restructure_rows(2, 1000, row, col, np.ones(3), 1, 0, 0, max_draws_per_row=0)
