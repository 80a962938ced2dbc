"""GPU parity: every op of the CUDA library, called through the C ABI, against
the fp64 oracle on the same seeded inputs.

Bar: |gpu - oracle| <= 1e-5 * T per output, where T is the oracle's sum of
|terms|, for fp32 and for bf16 storage alike (every kernel accumulates in fp32
on exactly widened inputs), plus half a bf16 ulp for an output rounded to
bf16 once; this is inside the stated contract (1e-5 * T fp32, 2e-3 * T bf16).
Indices and restructure outputs bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
from spmm_row_sorted_gb300 import build as snack_build
from spmm_row_sorted_gb300 import snack
from spmm_row_sorted_gb300 import workloads as wl

from gpu_util import ACC_REL, act_tensor, assert_close_T, bits, f64, layer_tensors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    snack_build.build()
    snack.load()
    oracle.set_threads(8)


def run_layer_ops(layer: wl.Layer, acts: wl.Acts, ops=("fwd", "dx", "dw"), max_batch=None, with_bias=True):
    row, col, val, bias = layer_tensors(layer)
    B = acts.batch
    L = snack.SparseLinear(layer.out_f, layer.in_f, row, col, val, bias if with_bias else None,
                           max_batch=max_batch or max(B, 1), validate=True)
    x = act_tensor(acts.x, acts.act_dtype)
    dy = act_tensor(acts.dy, acts.act_dtype)
    out = {}
    if "fwd" in ops:
        out["y"] = L.forward(x)
    if "dx" in ops:
        out["dx"] = L.grad_input(dy)
    if "dw" in ops:
        out["dw"], out["db"] = L.grad_weight(x, dy)
    torch.cuda.synchronize()
    L.close()
    return out


def check_layer_ops(layer: wl.Layer, acts: wl.Acts, ops=("fwd", "dx", "dw"), max_batch=None, with_bias=True,
                    got=None):
    got = got or run_layer_ops(layer, acts, ops, max_batch, with_bias)
    bf = acts.act_dtype == "bf16"
    rel = ACC_REL  # fp32 accumulation in every kernel; bf16 outputs add their one rounding
    v64 = oracle.as_f64(layer.val, layer.val_dtype)
    x64 = oracle.as_f64(acts.x, acts.act_dtype)
    dy64 = oracle.as_f64(acts.dy, acts.act_dtype)
    b64 = oracle.as_f64(layer.bias) if with_bias else None
    if "fwd" in ops:
        y, t = oracle.fwd(layer.out_f, layer.in_f, layer.row, layer.col, v64, x64, b64)
        assert_close_T(f64(got["y"]), y, t, rel, "fwd", stored_bf16=bf)
    if "dx" in ops:
        g, t = oracle.dx(layer.out_f, layer.in_f, layer.row, layer.col, v64, dy64)
        assert_close_T(f64(got["dx"]), g, t, rel, "dx", stored_bf16=bf)
    if "dw" in ops:
        d, t, db = oracle.dw(layer.out_f, layer.in_f, layer.row, layer.col, x64, dy64)
        assert_close_T(f64(got["dw"]), d, t, ACC_REL, "dw")  # fp32 output
        tdb = np.abs(dy64).sum(axis=0)
        assert_close_T(f64(got["db"]), db, tdb, ACC_REL, "db")
    return got


# ---------------------------------------------------------------- small shapes, several tiles, ragged tails

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("batch", [1, 2, 3, 5, 8, 13, 32, 33, 64, 100, 130])
def test_small_random(dtype, batch):
    lay = wl.make_layer(97, 131, nnz=2500, val_std=0.5, val_dtype=dtype, seed=batch, bias="normal")
    acts = wl.make_acts(batch, 131, 97, dtype, seed=batch)
    check_layer_ops(lay, acts)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 37, 30), (37, 1, 20), (300, 4000, 60000), (4000, 300, 60000),
                                   (33, 65, 0), (1000, 1000, 1000)])
def test_shapes(dtype, shape):
    out_f, in_f, nnz = shape
    lay = wl.make_layer(out_f, in_f, nnz=nnz, val_std=0.3, val_dtype=dtype, seed=nnz + 7, bias="normal")
    for batch in (1, 7, 32):
        acts = wl.make_acts(batch, in_f, out_f, dtype, seed=batch)
        check_layer_ops(lay, acts)


def test_one_row_holds_everything():
    # a single row with 20000 weights: split across many tiles and warps
    out_f, in_f = 50, 20000
    row = np.full(in_f, 17, dtype=np.int32)
    col = np.arange(in_f, dtype=np.int32)
    val = wl.random_normal(in_f, seed=1, stream=0, std=0.1)
    lay = wl.Layer(out_f, in_f, row, col, val, wl.random_normal(out_f, 1, 1), "f32")
    for batch in (1, 4, 32, 40):
        check_layer_ops(lay, wl.make_acts(batch, in_f, out_f, "f32", seed=batch))


def test_zipf_rows_skew():
    lay = wl.make_layer(2048, 3000, nnz=200000, zipf_s=1.2, val_dtype="f32", seed=3, bias="normal")
    for batch in (1, 8, 32):
        check_layer_ops(lay, wl.make_acts(batch, 3000, 2048, "f32", seed=batch))


def test_empty_rows_and_columns():
    # rows 0..99 and columns 0..49 and 150..199 empty
    rng = np.random.default_rng(0)
    pos = np.sort(rng.choice(100 * 100, 3000, replace=False))
    row = (100 + pos // 100).astype(np.int32)
    col = (50 + pos % 100).astype(np.int32)
    val = wl.random_normal(3000, 2, 0)
    lay = wl.Layer(250, 200, row, col, val, wl.random_normal(250, 2, 1), "f32")
    for batch in (1, 6, 32):
        check_layer_ops(lay, wl.make_acts(batch, 200, 250, "f32", seed=batch))


def test_batch_smaller_than_max_batch_and_zero_batch():
    lay = wl.make_layer(300, 200, nnz=5000, val_dtype="f32", seed=9, bias="normal")
    for batch in (1, 3, 16):
        check_layer_ops(lay, wl.make_acts(batch, 200, 300, "f32", seed=batch), max_batch=64)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(300, 200, row, col, val, bias, max_batch=64)
    y = torch.empty((0, 300), device="cuda")
    L.forward(torch.empty((0, 200), device="cuda"), out=y)
    dw, db = L.grad_weight(torch.empty((0, 200), device="cuda"), torch.empty((0, 300), device="cuda"))
    assert torch.all(dw == 0) and torch.all(db == 0)
    L.close()


# ---------------------------------------------------------------- the five workloads

def test_workload_c1():
    c = wl.CONFIGS["c1"]
    lay = wl.config_layer("c1")
    check_layer_ops(lay, wl.make_acts(8, c["in_f"], c["out_f"], "f32"))


@pytest.mark.parametrize("batch", [1, 16, 64])
def test_workload_c2(batch):
    lay = wl.config_layer("c2")
    acts = wl.make_acts(batch, 4096, 4096, "bf16")
    # one handle serves all three batches, as in single-stream inference
    check_layer_ops(lay, acts, ops=("fwd",), max_batch=64)


@pytest.mark.parametrize("batch", [1, 16])
def test_workload_c2_planted_missing_term_is_caught(batch):
    # Detection power of the bound: drop one stored weight of typical size
    # from the GPU's copy of the 4096^2 bf16 layer only, and the comparison
    # with the oracle (which keeps it) must fail at that weight's row.  A row
    # holds ~410 terms (T ~ 5), so the bound is ~5e-5 plus half a bf16 ulp of
    # y, while a typical term is ~0.01.
    lay = wl.config_layer("c2")
    acts = wl.make_acts(batch, 4096, 4096, "bf16")
    v64 = oracle.as_f64(lay.val, "bf16")
    x64 = oracle.as_f64(acts.x, "bf16")
    y, t = oracle.fwd(4096, 4096, lay.row, lay.col, v64, x64, oracle.as_f64(lay.bias))
    r = int(np.argmin(np.abs(y[0, :64])))  # a row with a small output (smallest rounding slack)
    ks = np.flatnonzero(lay.row == r)
    terms = np.abs(v64[ks] * x64[0, lay.col[ks]])
    k = int(ks[np.argsort(terms)[len(ks) // 2]])  # the row's median-size term
    row, col, val, bias = layer_tensors(lay)
    val[k] = 0.0  # planted on the device copy only
    L = snack.SparseLinear(4096, 4096, row, col, val, bias, max_batch=64)
    got = f64(L.forward(act_tensor(acts.x, "bf16")))
    torch.cuda.synchronize()
    L.close()
    with pytest.raises(AssertionError) as e:
        assert_close_T(got, y, t, ACC_REL, "planted", stored_bf16=True)
    assert f"[0, {r}]" in str(e.value)  # the first flagged output is the planted row at batch row 0
    # every other row still matches
    keep = np.ones(4096, dtype=bool)
    keep[r] = False
    assert_close_T(got[:, keep], y[:, keep], t[:, keep], ACC_REL, "untouched rows", stored_bf16=True)


def test_workload_c3_layers():
    for li in (0, 1):
        lay = wl.config_layer("c3", layer_index=li)
        check_layer_ops(lay, wl.make_acts(1024, lay.in_f, lay.out_f, "f32", seed=li))


def test_workload_c4_ops_and_restructure():
    lay = wl.config_layer("c4")
    acts = wl.make_acts(32, 16384, 16384, "f32")
    check_layer_ops(lay, acts)
    n_prune = int(0.10 * lay.nnz)
    restructure_and_check(lay, n_prune, seed=0, step=1, acts=acts)


def test_workload_c5_sampled():
    # 33.5M stored weights at batch 128: compare sampled batch rows / weights
    lay = wl.config_layer("c5")
    acts = wl.make_acts(128, 8192, 8192, "bf16")
    got = run_layer_ops(lay, acts)
    rel = ACC_REL
    v64 = oracle.as_f64(lay.val, "bf16")
    rows = np.array([0, 37, 127])
    x64 = oracle.as_f64(acts.x, "bf16")[rows]
    dy64 = oracle.as_f64(acts.dy, "bf16")[rows]
    y, t = oracle.fwd(8192, 8192, lay.row, lay.col, v64, x64, oracle.as_f64(lay.bias))
    assert_close_T(f64(got["y"])[rows], y, t, rel, "fwd c5", stored_bf16=True)
    g, t = oracle.dx(8192, 8192, lay.row, lay.col, v64, dy64)
    assert_close_T(f64(got["dx"])[rows], g, t, rel, "dx c5", stored_bf16=True)
    ks = np.random.default_rng(0).choice(lay.nnz, 4096, replace=False)
    d, t, _ = oracle.dw(8192, 8192, lay.row[ks], lay.col[ks], oracle.as_f64(acts.x, "bf16"),
                        oracle.as_f64(acts.dy, "bf16"), want_db=False)
    assert_close_T(f64(got["dw"])[ks], d, t, ACC_REL, "dw c5")


# ---------------------------------------------------------------- restructure

def restructure_and_check(lay: wl.Layer, n_prune: int, seed: int, step: int, acts=None):
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(lay.out_f, lay.in_f, row, col, val, bias, max_batch=acts.batch if acts else 8)
    src = L.restructure(n_prune, seed, step)
    torch.cuda.synchronize()
    ro, co, so, _ = oracle.restructure(lay.out_f, lay.in_f, lay.row, lay.col, oracle.as_f64(lay.val, lay.val_dtype),
                                       n_prune, seed, step)
    assert np.array_equal(L.row.cpu().numpy(), ro), "row_out"
    assert np.array_equal(L.col.cpu().numpy(), co), "col_out"
    assert np.array_equal(src.cpu().numpy(), so.astype(np.int32)), "src_out"
    vo = oracle.restructure_values(lay.val, so)
    want_bits = vo.view(np.uint32) if lay.val_dtype == "f32" else vo.view(np.uint16)
    assert np.array_equal(bits(L.val), want_bits), "val_out bits"
    if acts is not None:  # the rebuilt plan serves the new pattern
        new = wl.Layer(lay.out_f, lay.in_f, ro, co, vo, lay.bias, lay.val_dtype)
        x = act_tensor(acts.x, acts.act_dtype)
        dy = act_tensor(acts.dy, acts.act_dtype)
        got = {"y": L.forward(x), "dx": L.grad_input(dy)}
        got["dw"], got["db"] = L.grad_weight(x, dy)
        torch.cuda.synchronize()
        check_layer_ops(new, acts, got=got)
    L.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", [(8, 8, 20, 5), (1, 50, 10, 10), (40, 30, 600, 0), (40, 30, 600, 600),
                                  (64, 64, 3000, 1000), (500, 700, 30000, 3000), (3, 3, 4, 4),
                                  (300, 700, 20000, 0), (300, 700, 20000, 1), (50, 1, 20, 5), (7, 3, 10, 5),
                                  (70000, 70000, 30000, 3000)])
def test_restructure_small(dtype, case):
    out_f, in_f, nnz, n_prune = case
    lay = wl.make_layer(out_f, in_f, nnz=nnz, val_std=1.0, val_dtype=dtype, seed=nnz)
    for seed, step in ((0, 0), (5, 123)):
        restructure_and_check(lay, n_prune, seed, step, acts=wl.make_acts(4, in_f, out_f, dtype))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", [(500, 700, 30000, 3000, None), (64, 64, 3000, 1000, None), (7, 3, 10, 5, None),
                                  (2000, 3000, 200000, 20000, 1.2), (70000, 20, 3000, 300, None),
                                  (40, 30, 600, 0, None), (70000, 70000, 30000, 3000, None),
                                  (300, 400, 40000, 20000, None), (65536, 32768, 20000, 2000, None),
                                  (65536, 65536, 20000, 2000, None), (300, 5000, 2000, 300, None),
                                  (200, 300, 8000, 2000, None), (200, 300, 8000, 2001, None)])
def test_restructure_chain_plan_equals_fresh(dtype, case):
    # The restructure rebuilds the handle's plan in place: row offsets and the
    # 16-bit columns from its merge, and the column view updated into the
    # plan's second view (row and column bits within 31 -- 65536 x 32768 is at
    # the limit --, at most a quarter of the weights pruned: 2000 of 8000 is,
    # 2001 is not; mostly empty columns in 300 x 5000) or rebuilt (70000^2 and
    # 65536^2; half pruned).  After three
    # restructures in a row the COO still
    # matches the oracle, and every op on the handle is bit-identical to the
    # same op on a new handle made for the final pattern, at a small-batch and
    # at a tile-path batch: same column view, storage indices and tiles.
    out_f, in_f, nnz, n_prune, zipf = case
    lay = wl.make_layer(out_f, in_f, nnz=nnz, zipf_s=zipf, val_std=0.5, val_dtype=dtype, seed=7, bias="normal")
    row, col, val, bias = layer_tensors(lay)
    mb = 32
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=mb)
    r, c, v = lay.row, lay.col, lay.val
    for step in range(3):
        src = L.restructure(n_prune, seed=2, step=step)
        torch.cuda.synchronize()
        r, c, so, _ = oracle.restructure(out_f, in_f, r, c, oracle.as_f64(v, dtype), n_prune, 2, step)
        v = oracle.restructure_values(v, so)
        assert np.array_equal(L.row.cpu().numpy(), r) and np.array_equal(L.col.cpu().numpy(), c), step
        assert np.array_equal(src.cpu().numpy(), so.astype(np.int32)), step
        assert np.array_equal(bits(L.val), v.view(np.uint32) if dtype == "f32" else v.view(np.uint16)), step
    F = snack.SparseLinear(out_f, in_f, L.row.clone(), L.col.clone(), L.val.clone(), bias, max_batch=mb)
    for batch in (4, mb):
        acts = wl.make_acts(batch, in_f, out_f, dtype, seed=batch)
        x, dy = act_tensor(acts.x, dtype), act_tensor(acts.dy, dtype)
        for M in (L, F):
            M.out = (M.forward(x), M.grad_input(dy), *M.grad_weight(x, dy), *M.backward(x, dy))
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(L.out, F.out)):
            assert torch.equal(a, b), (batch, i)
    F.close()
    L.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_restructure_deferred_column_view(dtype):
    # After a restructure the column view is rebuilt on the handle's second
    # stream once the call has returned.  Its scratch lives in the plan: the
    # workspace is overwritten right after the call, the forward runs at once
    # (it does not wait), and the column-view readers run on another stream
    # (they wait for the rebuild through the handle's event); every result
    # matches the oracle on the new pattern, at a small-batch and a tile batch.
    out_f, in_f, nnz = 3000, 5000, 300000
    lay = wl.make_layer(out_f, in_f, nnz=nnz, zipf_s=1.1, val_std=0.3, val_dtype=dtype, seed=8, bias="normal")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=32)
    ro, co, so, _ = oracle.restructure(out_f, in_f, lay.row, lay.col, oracle.as_f64(lay.val, dtype), 30000, 3, 4)
    new = wl.Layer(out_f, in_f, ro, co, oracle.restructure_values(lay.val, so), lay.bias, dtype)
    other = torch.cuda.Stream()
    for batch in (4, 32):
        acts = wl.make_acts(batch, in_f, out_f, dtype, seed=batch)
        x, dy = act_tensor(acts.x, dtype), act_tensor(acts.dy, dtype)
        M = snack.SparseLinear(out_f, in_f, row.clone(), col.clone(), val.clone(), bias, max_batch=32)
        M.restructure(30000, seed=3, step=4)
        M.ws.fill_(0)  # the rebuild must not read the caller's workspace (a zero there would stop it)
        got = {"y": M.forward(x)}
        other.wait_stream(torch.cuda.current_stream())  # inputs and the new COO, not the rebuild
        with torch.cuda.stream(other):
            got["dx"] = M.grad_input(dy, stream=other)
            got["dw"], got["db"] = M.grad_weight(x, dy, stream=other)
            bdx, bdw, bdb = M.backward(x, dy, stream=other)
        other.synchronize()
        torch.cuda.synchronize()
        assert np.array_equal(M.row.cpu().numpy(), ro) and np.array_equal(M.col.cpu().numpy(), co)
        check_layer_ops(new, acts, got=got)
        check_layer_ops(new, acts, ops=("dx", "dw"), got={"dx": bdx, "dw": bdw, "db": bdb})
        snack.snack_wait_plan(M.handle)
        M.close()
    L.close()


def test_restructure_ties_zeros_nan():
    lay = wl.make_layer(60, 70, nnz=2000, val_dtype="f32", seed=4)
    v = np.round(lay.val * 50).astype(np.float32) / 50  # many exact ties
    v[::7] = 0.0
    v[3::11] = -0.0
    v[5] = np.nan
    lay.val = v
    restructure_and_check(lay, 700, seed=9, step=2)


def test_restructure_crowded_empties_general_sort():
    # Every empty position sits in the last row, so the regrown positions all
    # land in one bucket of the position range: the bucket overflows and the
    # regrown list is sorted the general way.  Output still bit-exact.
    out_f, in_f = 64, 512
    full = np.arange(63 * in_f, dtype=np.int64)
    rng = np.random.default_rng(5)
    tail = 63 * in_f + np.sort(rng.choice(in_f, 100, replace=False))
    p = np.concatenate([full, tail])
    val = wl.random_normal(p.size, seed=5, stream=0, std=0.3)
    lay = wl.Layer(out_f, in_f, (p // in_f).astype(np.int32), (p % in_f).astype(np.int32), val,
                   wl.random_normal(out_f, 5, 1), "f32")
    for step in range(3):
        restructure_and_check(lay, 200, seed=11, step=step)


def test_restructure_bucket_overflow_general_sort():
    # 1500 regrown positions, all in the last row of a 64 x 4096 layer: they
    # crowd two of the 23 equal-width buckets (256 slots each), the buckets
    # run over, and the lists come from the general sort (queued after the
    # host reads the verdict); the merge passes queued before it write nothing.
    out_f, in_f = 64, 4096
    rng = np.random.default_rng(6)
    tail = 63 * in_f + np.sort(rng.choice(in_f, 1000, replace=False))
    p = np.concatenate([np.arange(63 * in_f, dtype=np.int64), tail])
    val = wl.random_normal(p.size, seed=6, stream=0, std=0.3)
    lay = wl.Layer(out_f, in_f, (p // in_f).astype(np.int32), (p % in_f).astype(np.int32), val,
                   wl.random_normal(out_f, 6, 1), "f32")
    restructure_and_check(lay, 1500, seed=3, step=1, acts=wl.make_acts(8, in_f, out_f, "f32"))


def first_chunk_draws(n_pos: int, nnz: int, n_prune: int) -> int:
    # the library's first draw chunk: the expected draws plus the lesser of
    # eight standard deviations and a tenth of them, plus 1024
    empty = n_pos - nnz
    lo, hi = empty - n_prune + 0.5, empty + 0.5
    ex = n_pos * np.log(hi / lo)
    sd = np.sqrt(max(n_pos * n_pos * (1.0 / lo - 1.0 / hi) - n_pos * np.log(hi / lo), 0.0))
    return int(np.ceil(min(ex + 8.0 * sd, 1.1 * ex) + 1024.0))


def test_restructure_extra_draw_chunks():
    # Regrowing every empty position of a 100 x 100 layer: for some seeds the
    # first chunk of draws misses a position (the oracle needs more draws than
    # the chunk holds), the merge passes queued behind the lists' flag write
    # nothing, and the host draws more chunks and sorts the general way.  Both
    # outcomes are bit-exact.
    lay = wl.make_layer(100, 100, nnz=9000, val_dtype="f32", seed=13)
    m1 = first_chunk_draws(10000, 9000, 1000)
    short, full = [], []
    for seed in range(40):
        draws = oracle.restructure(100, 100, lay.row, lay.col, oracle.as_f64(lay.val), 1000, seed, 0)[3]
        (short if draws > m1 else full).append(seed)
    assert short and full, (short, full)
    for seed in short[:3] + full[:1]:
        restructure_and_check(lay, 1000, seed=seed, step=0, acts=wl.make_acts(8, 100, 100, "f32"))


def test_restructure_large_prune_general_sort_column_view():
    # 1.1M regrown positions: more buckets than the bucket sort takes, so the
    # first chunk's lists come from the general sort (speculatively, before the
    # host's verdict); the column view is updated from them.  The COO is
    # bit-exact and the input gradient through the updated view equals a fresh
    # handle's bit for bit.
    out_f = in_f = 20000
    lay = wl.make_layer(out_f, in_f, nnz=4_500_000, val_std=0.1, val_dtype="f32", seed=14)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=8)
    src = L.restructure(1_100_000, 5, 9)
    torch.cuda.synchronize()
    ro, co, so, _ = oracle.restructure(out_f, in_f, lay.row, lay.col, oracle.as_f64(lay.val), 1_100_000, 5, 9)
    assert np.array_equal(L.row.cpu().numpy(), ro) and np.array_equal(L.col.cpu().numpy(), co)
    assert np.array_equal(src.cpu().numpy(), so.astype(np.int32))
    F = snack.SparseLinear(out_f, in_f, L.row.clone(), L.col.clone(), L.val.clone(), bias, max_batch=8)
    dy = act_tensor(wl.make_acts(8, in_f, out_f, "f32").dy, "f32")
    assert torch.equal(L.grad_input(dy), F.grad_input(dy))
    F.close()
    L.close()


def test_restructure_chain_of_steps():
    lay = wl.make_layer(200, 300, nnz=6000, val_dtype="f32", seed=12)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(200, 300, row, col, val, bias, max_batch=8)
    r, c, v = lay.row, lay.col, lay.val
    for step in range(4):
        L.restructure(600, 77, step)
        r2, c2, s2, _ = oracle.restructure(200, 300, r, c, oracle.as_f64(v), 600, 77, step)
        v2 = oracle.restructure_values(v, s2)
        torch.cuda.synchronize()
        assert np.array_equal(L.row.cpu().numpy(), r2) and np.array_equal(L.col.cpu().numpy(), c2)
        assert np.array_equal(bits(L.val), v2.view(np.uint32))
        r, c, v = r2, c2, v2
    L.close()


def test_restructure_no_space():
    lay = wl.make_layer(4, 4, nnz=12, val_dtype="f32", seed=1)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(4, 4, row, col, val, bias, max_batch=1)
    with pytest.raises(snack.SnackError) as e:
        L.restructure(5, 0, 0)  # only 4 empty positions
    assert e.value.status == 8
    L.close()


# ---------------------------------------------------------------- contracts

def test_inputs_untouched_and_deterministic():
    lay = wl.make_layer(777, 555, nnz=40000, zipf_s=1.1, val_dtype="f32", seed=2, bias="normal")
    acts = wl.make_acts(32, 555, 777, "f32")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(777, 555, row, col, val, bias, max_batch=32)
    x = act_tensor(acts.x, "f32")
    dy = act_tensor(acts.dy, "f32")
    keep = [t.clone() for t in (row, col, val, bias, x, dy)]
    y1 = torch.full((32, 777), float("nan"), device="cuda")
    dx1 = torch.full((32, 555), float("nan"), device="cuda")
    L.forward(x, out=y1)
    L.grad_input(dy, out=dx1)
    dw1, db1 = L.grad_weight(x, dy)
    y2, dx2 = L.forward(x), L.grad_input(dy)
    dw2, db2 = L.grad_weight(x, dy)
    torch.cuda.synchronize()
    for a, b in zip(keep, (row, col, val, bias, x, dy)):
        assert torch.equal(a, b)
    assert not torch.isnan(y1).any() and not torch.isnan(dx1).any()  # every output written
    assert torch.equal(y1, y2) and torch.equal(dx1, dx2) and torch.equal(dw1, dw2) and torch.equal(db1, db2)
    L.close()


def test_validation_errors():
    row = torch.tensor([0, 2, 1], dtype=torch.int32, device="cuda")
    col = torch.tensor([0, 0, 0], dtype=torch.int32, device="cuda")
    val = torch.ones(3, device="cuda")
    with pytest.raises(snack.SnackError) as e:
        snack.SparseLinear(3, 3, row, col, val, validate=True)
    assert e.value.status == 2
    row = torch.tensor([0, 1, 5], dtype=torch.int32, device="cuda")
    with pytest.raises(snack.SnackError) as e:
        snack.SparseLinear(3, 3, row, col, val, validate=True)
    assert e.value.status == 3


def test_call_errors():
    lay = wl.make_layer(30, 20, nnz=100, val_dtype="f32", seed=1)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(30, 20, row, col, val, bias, max_batch=4)
    x = torch.zeros((8, 20), device="cuda")
    with pytest.raises(snack.SnackError) as e:
        L.forward(x)  # batch > max_batch
    assert e.value.status == 1
    # a short workspace: batch 32 takes the tile kernels, which need scratch
    L32 = snack.SparseLinear(30, 20, row, col, val, bias, max_batch=32)
    x32 = torch.zeros((32, 20), device="cuda")
    y32 = torch.empty((32, 30), device="cuda")
    with pytest.raises(snack.SnackError) as e:
        snack.snack_spmm_fwd(L32.handle, row, col, val, x32, 32, bias, y32, L32.ws[:256])
    assert e.value.status == 4
    L32.close()
    # batch 2 runs the small-batch kernel, which uses no workspace
    y = torch.empty((2, 30), device="cuda")
    snack.snack_spmm_fwd(L.handle, row, col, val, x[:2], 2, bias, y, L.ws[:256])
    buf = torch.zeros(4 * 30, device="cuda")
    with pytest.raises(snack.SnackError) as e:  # y overlaps x
        snack.snack_spmm_fwd(L.handle, row, col, val, buf[:40], 2, bias, buf[10:70], L.ws)
    assert e.value.status == 1
    L.close()


def test_autograd_function():
    lay = wl.make_layer(64, 48, nnz=700, val_dtype="f32", seed=3, bias="normal")
    acts = wl.make_acts(8, 48, 64, "f32")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(64, 48, row, col, val.requires_grad_(True), bias, max_batch=8)
    x = act_tensor(acts.x, "f32").requires_grad_(True)
    g = act_tensor(acts.dy, "f32")
    y = snack.sparse_linear(x, L)
    y.backward(g)
    torch.cuda.synchronize()
    v64, x64, g64 = oracle.as_f64(lay.val), oracle.as_f64(acts.x), oracle.as_f64(acts.dy)
    dx, t = oracle.dx(64, 48, lay.row, lay.col, v64, g64)
    assert_close_T(f64(x.grad), dx, t, 1e-5, "autograd dx")
    dw, t, _ = oracle.dw(64, 48, lay.row, lay.col, x64, g64)
    assert_close_T(f64(L.val.grad), dw, t, 1e-5, "autograd dw")
    L.close()


# ---------------------------------------------------------------- fused backward

def run_backward(layer: wl.Layer, acts: wl.Acts, max_batch=None):
    row, col, val, bias = layer_tensors(layer)
    L = snack.SparseLinear(layer.out_f, layer.in_f, row, col, val, bias, max_batch=max_batch or acts.batch)
    x = act_tensor(acts.x, acts.act_dtype)
    dy = act_tensor(acts.dy, acts.act_dtype)
    dx, dw, db = L.backward(x, dy)
    torch.cuda.synchronize()
    L.close()
    return {"dx": dx, "dw": dw, "db": db}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("batch", [1, 3, 8, 32, 64, 128, 200])
def test_backward_matches_oracle(dtype, batch):
    lay = wl.make_layer(500, 700, nnz=30000, zipf_s=1.1, val_std=0.3, val_dtype=dtype, seed=batch, bias="normal")
    acts = wl.make_acts(batch, 700, 500, dtype, seed=batch)
    check_layer_ops(lay, acts, ops=("dx", "dw"), got=run_backward(lay, acts))


def test_backward_workloads_c1_c4():
    for name, B in (("c1", 8), ("c4", 32)):
        lay = wl.config_layer(name)
        acts = wl.make_acts(B, lay.in_f, lay.out_f, "f32")
        check_layer_ops(lay, acts, ops=("dx", "dw"), got=run_backward(lay, acts))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_rows_repeated_calls(dtype):
    # Rows split between tiles (long Zipf rows span several) leave partials
    # that the fix-up adds in tile order: one handle, several batch sizes
    # (one and several batch tiles), every tile-path op twice in a row, each
    # call bit-identical to the one before and within the bound of the oracle.
    lay = wl.make_layer(600, 900, nnz=60000, zipf_s=1.3, val_std=0.3, val_dtype=dtype, seed=17, bias="normal")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(600, 900, row, col, val, bias, max_batch=300)
    for batch in (9, 300, 33, 300, 9):
        acts = wl.make_acts(batch, 900, 600, dtype, seed=batch)
        x, dy = act_tensor(acts.x, dtype), act_tensor(acts.dy, dtype)
        got = {"y": L.forward(x), "dx": L.grad_input(dy)}
        got["dw"], got["db"] = L.grad_weight(x, dy)
        dx_b, dw_b, _ = L.backward(x, dy)
        again = (L.forward(x), L.grad_input(dy), L.backward(x, dy)[0])
        torch.cuda.synchronize()
        assert torch.equal(got["y"], again[0]) and torch.equal(got["dx"], again[1]), batch
        assert torch.equal(dx_b, again[2]) and torch.equal(dx_b, got["dx"]), batch
        check_layer_ops(lay, acts, got=got)
    L.close()


@pytest.mark.parametrize("batch,out_f,in_f,nnz", [(32, 300, 400, 20000), (5, 300, 400, 20000),
                                                  (8, 3000, 600, 900000)])
def test_backward_equals_separate_calls_bitwise(batch, out_f, in_f, nnz):
    # dX and db come from the same kernels and tiles as the separate calls, so
    # they are bit-identical; dW may differ in summation order (checked above
    # against the oracle).  Batches 5 and 8 run the small-batch path; the last
    # case stages 94 KB of dY per CTA (above the default 48 KB limit).
    lay = wl.make_layer(out_f, in_f, nnz=nnz, val_dtype="f32", seed=4, bias="normal")
    acts = wl.make_acts(batch, in_f, out_f, "f32", seed=4)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=batch)
    x, dy = act_tensor(acts.x, "f32"), act_tensor(acts.dy, "f32")
    dx_f, dw_f, db_f = L.backward(x, dy)
    dx_s = L.grad_input(dy)
    dw_s, db_s = L.grad_weight(x, dy)
    torch.cuda.synchronize()
    assert torch.equal(dx_f, dx_s) and torch.equal(db_f, db_s)
    L.close()


# ---------------------------------------------------------------- shared-memory limits

def _staged_layers():
    # batch 8 fp32, column view: dY of 3000 outputs staged (94 KB per CTA) and of 2000 outputs
    # (62.5 KB), both above the 48 KB default limit, through the same small-batch kernels
    big = wl.make_layer(3000, 600, nnz=900000, val_dtype="f32", seed=4, bias="normal")
    small = wl.make_layer(2000, 600, nnz=600000, val_dtype="f32", seed=5, bias="normal")
    return big, small


def test_shared_memory_limits_only_rise():
    # One thread: a backward on the big layer raises the fused kernel's limit, an input
    # gradient on the smaller layer must not lower it, and the big layer's backward runs
    # again with the same bits; then two host threads drive the two layers at once.
    import threading

    big, small = _staged_layers()
    acts_b = wl.make_acts(8, 600, 3000, "f32", seed=6)
    acts_s = wl.make_acts(8, 600, 2000, "f32", seed=7)

    def make(lay):
        row, col, val, bias = layer_tensors(lay)
        return snack.SparseLinear(lay.out_f, lay.in_f, row, col, val, bias, max_batch=8)

    B, S = make(big), make(small)
    xb, dyb = act_tensor(acts_b.x, "f32"), act_tensor(acts_b.dy, "f32")
    xs, dys = act_tensor(acts_s.x, "f32"), act_tensor(acts_s.dy, "f32")
    first = [t.clone() for t in B.backward(xb, dyb)]
    dx_s = S.grad_input(dys)
    again = B.backward(xb, dyb)
    torch.cuda.synchronize()
    for a, b in zip(first, again):
        assert torch.equal(a, b)
    check_layer_ops(big, acts_b, ops=("dx", "dw"), got={"dx": first[0], "dw": first[1], "db": first[2]})
    check_layer_ops(small, acts_s, ops=("dx",), got={"dx": dx_s})
    ref_s = dx_s.clone()

    errors = []

    def drive(layer, x, dy, want, kind):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(20):
                    got = layer.backward(x, dy, stream=st)[0] if kind == "bwd" else layer.grad_input(dy, stream=st)
                st.synchronize()
                if not torch.equal(got, want):
                    errors.append(kind + " differs")
        except Exception as e:  # a launch refused for a lowered limit surfaces here
            errors.append(repr(e))

    threads = [threading.Thread(target=drive, args=(B, xb, dyb, first[0], "bwd")),
               threading.Thread(target=drive, args=(S, xs, dys, ref_s, "dx"))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    B.close()
    S.close()


# ---------------------------------------------------------------- rows split between CTAs

def test_split_rows_repeat_calls_bitwise():
    # Long Zipf rows span many tiles, whose partials are combined in tile
    # order: repeated calls with 1, 2 and 3 batch tiles on one handle give
    # bit-identical results, and match the oracle.
    lay = wl.make_layer(700, 9000, nnz=400000, zipf_s=1.4, val_std=0.3, val_dtype="f32", seed=21, bias="normal")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(700, 9000, row, col, val, bias, max_batch=300)
    first = {}
    for rep in range(3):
        for batch in (300, 130, 40):
            acts = wl.make_acts(batch, 9000, 700, "f32", seed=batch)
            x, dy = act_tensor(acts.x, "f32"), act_tensor(acts.dy, "f32")
            y = L.forward(x)
            dx = L.grad_input(dy)
            dx_f, dw_f, db_f = L.backward(x, dy)
            torch.cuda.synchronize()
            got = [t.clone() for t in (y, dx, dx_f, dw_f, db_f)]
            if rep == 0:
                first[batch] = got
                check_layer_ops(lay, acts, ops=("fwd", "dx"), got={"y": y, "dx": dx})
            else:
                for a, b in zip(got, first[batch]):
                    assert torch.equal(a, b)
    L.close()


# ---------------------------------------------------------------- small-batch path (batch <= 8)

# The small-batch kernels stage the gathered operand (X, or dY for the column
# view) whole in shared memory when it fits in 96 KB at the padded batch width
# (1, 2, 4 or 8); wider operands, and batches above 8, take the tile kernels.
# Cases on both sides of that limit, for every op.
@pytest.mark.parametrize("dtype,batch,feat", [("f32", 8, 3072), ("f32", 8, 3073), ("f32", 4, 6144), ("f32", 3, 6145),
                                              ("bf16", 8, 6144), ("bf16", 6, 6145), ("bf16", 2, 24576),
                                              ("f32", 1, 40000), ("bf16", 16, 5120), ("bf16", 16, 5121),
                                              ("f32", 12, 2560), ("f32", 9, 2561)])
def test_small_batch_stage_limit(dtype, batch, feat):
    other = 97
    for out_f, in_f in ((other, feat), (feat, other)):
        lay = wl.make_layer(out_f, in_f, nnz=min(60000, out_f * in_f // 3), val_std=0.3, val_dtype=dtype,
                            seed=feat + batch, bias="normal")
        acts = wl.make_acts(batch, in_f, out_f, dtype, seed=batch)
        check_layer_ops(lay, acts)
        check_layer_ops(lay, acts, ops=("dx", "dw"), got=run_backward(lay, acts))


@pytest.mark.parametrize("dtype,batch", [("f32", 8), ("bf16", 6)])
def test_small_batch_weight_gradient_paths(dtype, batch):
    # dW alone: a flat pass while nnz * padded batch <= 2^22, the column-view
    # pass (dW and db only) above that
    for nnz in (30000, 700000):
        lay = wl.make_layer(1500, 3000, nnz=nnz, val_std=0.3, val_dtype=dtype, seed=nnz, bias="normal")
        acts = wl.make_acts(batch, 3000, 1500, dtype, seed=batch)
        check_layer_ops(lay, acts, ops=("dw",))


def test_small_batch_skewed_rows_and_empty_layer():
    # Zipf rows: whole rows per CTA, so the longest row sets one CTA's length
    lay = wl.make_layer(1500, 2000, nnz=150000, zipf_s=1.3, val_std=0.3, val_dtype="f32", seed=12, bias="normal")
    for batch in (1, 2, 7):
        acts = wl.make_acts(batch, 2000, 1500, "f32", seed=batch)
        check_layer_ops(lay, acts)
        check_layer_ops(lay, acts, ops=("dx", "dw"), got=run_backward(lay, acts))
    empty = wl.make_layer(40, 70, nnz=0, val_dtype="f32", seed=1, bias="normal")
    for batch in (1, 8):
        acts = wl.make_acts(batch, 70, 40, "f32", seed=batch)
        check_layer_ops(empty, acts)
        check_layer_ops(empty, acts, ops=("dx", "dw"), got=run_backward(empty, acts))


# ---------------------------------------------------------------- dense path (bf16, >= 25 % stored, batch >= 32)

# (out_f, in_f, density, batch): one and several M tiles, a partial last M
# tile (out_f 8, 200), one partial K chunk (in_f 8), K split across CTAs
# (2048 inputs), batch tiles of 48, 64, 144 and 2 x 256 (batch 300).
@pytest.mark.parametrize("case", [(256, 384, 0.5, 64), (320, 520, 0.3, 33), (128, 128, 1.0, 32), (200, 264, 0.6, 130),
                                  (8, 64, 0.5, 40), (136, 8, 0.5, 300), (1000, 2048, 0.26, 256)])
def test_dense_path_matches_oracle(case):
    out_f, in_f, density, batch = case
    lay = wl.make_layer(out_f, in_f, density=density, val_std=0.2, val_dtype="bf16", seed=out_f, bias="normal")
    acts = wl.make_acts(batch, in_f, out_f, "bf16", seed=in_f)
    check_layer_ops(lay, acts)
    check_layer_ops(lay, acts, ops=("dx", "dw"), got=run_backward(lay, acts))


def test_dense_path_bias_rounded_once():
    # Positive weights and inputs (no cancellation, T ~ |y|) and a bias of the
    # size of the product: the fp32 product and the bias must be added before
    # the single rounding to bf16.  Rounding the product to bf16 first and
    # again after adding the bias is up to a whole ulp off and fails the
    # half-ulp bound on many outputs.
    out_f, in_f, batch = 256, 384, 64
    lay = wl.make_layer(out_f, in_f, density=0.5, val_std=0.2, val_dtype="bf16", seed=31)
    lay.val = wl.bf16_bits_from_f32(np.abs(wl.f32_from_bf16_bits(lay.val)))
    lay.bias = np.linspace(5.0, 40.0, out_f).astype(np.float32)
    acts = wl.make_acts(batch, in_f, out_f, "bf16", seed=31)
    acts.x = wl.bf16_bits_from_f32(np.abs(wl.f32_from_bf16_bits(acts.x)))
    check_layer_ops(lay, acts, ops=("fwd",))


@pytest.mark.parametrize("case", [(136, 200, 0.9, 16), (64, 264, 0.97, 255), (128, 384, 0.5, 256), (72, 136, 0.5, 257),
                                  (128, 8192, 0.3, 32), (8192, 128, 0.3, 32)])
def test_dense_path_tiles_and_splits(case):
    # Nearly full 64-column blocks whose runs start at odd storage indices (the
    # value loads straddle words), batch tiles at the edges (16, 255, 256, 257),
    # one output tile with K split 8 ways (128 x 8192) and the input gradient's
    # long K (8192 x 128): every op against the oracle.
    out_f, in_f, density, batch = case
    lay = wl.make_layer(out_f, in_f, density=density, val_std=0.2, val_dtype="bf16", seed=out_f + batch,
                        bias="normal")
    acts = wl.make_acts(batch, in_f, out_f, "bf16", seed=batch)
    check_layer_ops(lay, acts)
    check_layer_ops(lay, acts, ops=("dx", "dw"), got=run_backward(lay, acts))


def test_dense_path_after_per_row_restructure():
    # the per-row restructure rewrites the columns of every row: the masks and
    # value offsets of the tensor-core path are rebuilt from them
    lay = wl.make_layer(128, 256, fan_in=96, val_std=0.2, val_dtype="bf16", seed=12, bias="normal")
    restructure_rows_and_check(lay, 20, seed=6, step=1, acts=wl.make_acts(40, 256, 128, "bf16", seed=4))


def test_dense_layer_narrow_batch_takes_gather_path():
    # the same dense layer at batch 8 (below the dense path's minimum), built for batch 64
    lay = wl.make_layer(256, 384, density=0.5, val_std=0.2, val_dtype="bf16", seed=3, bias="normal")
    acts = wl.make_acts(8, 384, 256, "bf16", seed=3)
    check_layer_ops(lay, acts, max_batch=64)


def test_dense_path_after_restructure():
    # the dense copy is rebuilt from the new pattern on every call
    lay = wl.make_layer(192, 256, density=0.5, val_std=0.2, val_dtype="bf16", seed=9, bias="normal")
    acts = wl.make_acts(48, 256, 192, "bf16", seed=9)
    restructure_and_check(lay, int(0.1 * lay.nnz), seed=5, step=2, acts=acts)


# ---------------------------------------------------------------- 16-bit index copies of the plan

@pytest.mark.parametrize("shape", [(20, 70000, 3000), (70000, 20, 3000), (10, 140000, 2000), (65536, 65536, 4000)])
def test_index_width_boundaries(shape):
    # feature counts above 65536 keep 32-bit indices; 65536 itself uses the 16-bit copies;
    # 140000 inputs also take the general column sort.  Batch 9 runs the tile kernels,
    # batch 1 the small-batch kernels.
    out_f, in_f, nnz = shape
    for dtype in ("f32", "bf16"):
        lay = wl.make_layer(out_f, in_f, nnz=nnz, val_std=0.5, val_dtype=dtype, seed=nnz, bias="normal")
        for batch in (1, 9):
            acts = wl.make_acts(batch, in_f, out_f, dtype, seed=1)
            check_layer_ops(lay, acts)
    restructure_and_check(lay, nnz // 10, seed=1, step=1, acts=acts)


# ---------------------------------------------------------------- constant fan-in forward

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", [(300, 700, 37, 9), (1000, 500, 1, 33), (64, 4000, 400, 130), (2000, 3000, 30, 300),
                                  (8, 64, 48, 16)])
def test_constant_fan_in_forward(dtype, case):
    # Every row holds K stored weights: the forward takes whole rows per warp
    # (no merge path, no split rows); batches above 8 take that kernel, every
    # op still matches the oracle, and so does the same layer after a per-row
    # restructure (which keeps the fan-in).
    out_f, in_f, K, batch = case
    lay = wl.make_layer(out_f, in_f, fan_in=K, val_std=0.3, val_dtype=dtype, seed=K + batch, bias="normal")
    acts = wl.make_acts(batch, in_f, out_f, dtype, seed=batch)
    check_layer_ops(lay, acts)
    restructure_rows_and_check(lay, max(1, K // 4), seed=3, step=2, acts=acts)


def test_row_count_multiple_of_out_f_without_constant_fan_in():
    # nnz = 3 * out_f but the rows differ in length: the tile kernels run
    lay = wl.make_layer(500, 700, nnz=1500, zipf_s=1.1, val_std=0.3, val_dtype="f32", seed=5, bias="normal")
    assert len(set(np.bincount(lay.row, minlength=500).tolist())) > 1
    for batch in (9, 32):
        check_layer_ops(lay, wl.make_acts(batch, 700, 500, "f32", seed=batch))


# ---------------------------------------------------------------- per-row (constant fan-in) restructure

def restructure_rows_and_check(lay: wl.Layer, n_per_row: int, seed: int, step: int, acts=None):
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(lay.out_f, lay.in_f, row, col, val, bias, max_batch=acts.batch if acts else 8)
    src = L.restructure_rows(n_per_row, seed, step)
    torch.cuda.synchronize()
    ro, co, so, _ = oracle.restructure_rows(lay.out_f, lay.in_f, lay.row, lay.col,
                                            oracle.as_f64(lay.val, lay.val_dtype), n_per_row, seed, step)
    assert np.array_equal(L.row.cpu().numpy(), ro), "row_out"
    assert np.array_equal(L.col.cpu().numpy(), co), "col_out"
    assert np.array_equal(src.cpu().numpy(), so.astype(np.int32)), "src_out"
    vo = oracle.restructure_values(lay.val, so)
    want_bits = vo.view(np.uint32) if lay.val_dtype == "f32" else vo.view(np.uint16)
    assert np.array_equal(bits(L.val), want_bits), "val_out bits"
    if acts is not None:  # the rebuilt column view serves the new pattern
        new = wl.Layer(lay.out_f, lay.in_f, ro, co, vo, lay.bias, lay.val_dtype)
        x = act_tensor(acts.x, acts.act_dtype)
        dy = act_tensor(acts.dy, acts.act_dtype)
        got = {"y": L.forward(x), "dx": L.grad_input(dy)}
        got["dw"], got["db"] = L.grad_weight(x, dy)
        torch.cuda.synchronize()
        check_layer_ops(new, acts, got=got)
    L.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", [("fanin", 300, 500, 40, 4), ("fanin", 64, 1000, 300, 256), ("zipf", 400, 3000, 9000, 12),
                                  ("uniform", 200, 333, 5000, 3), ("fanin", 50, 70, 10, 0)])
def test_restructure_rows_matches_oracle(dtype, case):
    kind, out_f, in_f, size, n = case
    if kind == "fanin":
        lay = wl.make_layer(out_f, in_f, fan_in=size, val_std=0.3, val_dtype=dtype, seed=out_f, bias="normal")
    elif kind == "zipf":
        lay = wl.make_layer(out_f, in_f, nnz=size, zipf_s=1.2, val_std=0.3, val_dtype=dtype, seed=out_f, bias="normal")
    else:
        lay = wl.make_layer(out_f, in_f, nnz=size, val_std=0.3, val_dtype=dtype, seed=out_f, bias="normal")
    acts = wl.make_acts(16, in_f, out_f, dtype, seed=2)
    restructure_rows_and_check(lay, n, seed=7, step=3, acts=acts)


def test_restructure_rows_ties_nan_and_chain():
    lay = wl.make_layer(40, 64, fan_in=16, val_std=1.0, val_dtype="f32", seed=3, bias="normal")
    v = np.round(lay.val).astype(np.float32)
    v[::7] = -0.0
    v[5] = np.nan
    lay.val = v
    restructure_rows_and_check(lay, 5, seed=1, step=0)
    # a chain of steps on one handle, against the oracle chain
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(40, 64, row, col, val, bias, max_batch=8)
    r, c, vv = lay.row, lay.col, oracle.as_f64(lay.val)
    for step in range(4):
        L.restructure_rows(3, 11, step)
        r, c, so, _ = oracle.restructure_rows(40, 64, r, c, vv, 3, 11, step)
        vv = np.where(so >= 0, vv[np.maximum(so, 0)], 0.0)
    torch.cuda.synchronize()
    assert np.array_equal(L.col.cpu().numpy(), c) and np.array_equal(L.row.cpu().numpy(), r)
    L.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_restructure_rows_chain_column_view(dtype):
    # Consecutive per-row restructures on one handle, each small enough for
    # the incremental column-view update (out_f * n_per_row within a quarter
    # of nnz): every update merges the view the one before left, and after
    # each step every op that reads the column view matches the oracle.
    out_f, in_f, K, n = 300, 500, 40, 6
    lay = wl.make_layer(out_f, in_f, fan_in=K, val_std=0.5, val_dtype=dtype, seed=21, bias="normal")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=16)
    r, c, v = lay.row, lay.col, lay.val
    acts = wl.make_acts(16, in_f, out_f, dtype, seed=5)
    x, dy = act_tensor(acts.x, dtype), act_tensor(acts.dy, dtype)
    for step in range(5):
        src = L.restructure_rows(n, 9, step)
        r, c, so, _ = oracle.restructure_rows(out_f, in_f, r, c, oracle.as_f64(v, dtype), n, 9, step)
        v = oracle.restructure_values(v, so)
        got = {"y": L.forward(x), "dx": L.grad_input(dy)}
        got["dw"], got["db"] = L.grad_weight(x, dy)
        torch.cuda.synchronize()
        assert np.array_equal(L.col.cpu().numpy(), c) and np.array_equal(src.cpu().numpy(), so.astype(np.int32)), step
        check_layer_ops(wl.Layer(out_f, in_f, r, c, v, lay.bias, dtype), acts, got=got)
    L.close()


def test_restructure_rows_bucket_overflow_rebuilds():
    # Every row holds columns 0..999 of 1024 and regrows all of its 24 empty
    # columns: the regrown positions all fall in the last of the column-order
    # buckets, which overflows, and the column view is rebuilt instead of
    # updated; the results are the same.
    out_f, in_f, K = 32, 1024, 1000
    rng = np.random.default_rng(4)
    row = np.repeat(np.arange(out_f, dtype=np.int32), K)
    col = np.tile(np.arange(K, dtype=np.int32), out_f)
    val = rng.normal(0.0, 0.5, size=out_f * K).astype(np.float32)
    lay = wl.Layer(out_f, in_f, row, col, val, rng.normal(size=out_f).astype(np.float32), "f32")
    restructure_rows_and_check(lay, 24, seed=2, step=1, acts=wl.make_acts(8, in_f, out_f, "f32", seed=8))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1024, 1024, 51), (768, 3072, 31), (3072, 768, 8), (300, 7000, 3)])
def test_diagonal_patterns(dtype, shape):
    # A diagonal sparsity pattern (wrapped diagonals, the same column offsets
    # in every row) is an ordinary row-sorted COO pattern: every op matches the
    # oracle at a small-batch and a tile-path batch, and both restructures
    # (unstructured and per-row) stay bit-exact on it.
    out_f, in_f, n_diag = shape
    lay = wl.make_layer(out_f, in_f, diagonals=n_diag, val_std=0.5, val_dtype=dtype, seed=n_diag, bias="normal")
    for batch in (4, 32):
        check_layer_ops(lay, wl.make_acts(batch, in_f, out_f, dtype, seed=batch))
    acts = wl.make_acts(8, in_f, out_f, dtype, seed=3)
    restructure_and_check(lay, lay.nnz // 10, seed=4, step=1, acts=acts)
    restructure_rows_and_check(lay, max(1, n_diag // 4), seed=4, step=1, acts=acts)


def test_restructure_rows_workload_c4_fanin():
    # 16384 x 16384 with a constant fan-in of 164 (99 % sparse), 10 % of every row per call
    lay = wl.make_layer(16384, 16384, fan_in=164, val_std=0.02, val_dtype="f32", seed=0)
    acts = wl.make_acts(32, 16384, 16384, "f32", seed=0)
    restructure_rows_and_check(lay, 16, seed=12345, step=1, acts=acts)


def test_restructure_rows_full_row_is_no_space_like_the_oracle():
    # Zipf rows saturate: the longest row holds every column, so it cannot regrow
    lay = wl.make_layer(400, 600, nnz=9000, zipf_s=1.2, val_std=0.3, val_dtype="f32", seed=400)
    with pytest.raises(oracle.RestructureError):
        oracle.restructure_rows(400, 600, lay.row, lay.col, oracle.as_f64(lay.val), 12, 7, 3)
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(400, 600, row, col, val, bias, max_batch=4)
    with pytest.raises(snack.SnackError) as e:
        L.restructure_rows(12, 7, 3)
    assert e.value.status == 8
    # the other rows were restructured on the device before the error was
    # seen; the handle still serves the input pattern
    acts = wl.make_acts(4, 600, 400, "f32", seed=2)
    x, dy = act_tensor(acts.x, "f32"), act_tensor(acts.dy, "f32")
    got = {"y": L.forward(x), "dx": L.grad_input(dy)}
    got["dw"], got["db"] = L.grad_weight(x, dy)
    torch.cuda.synchronize()
    check_layer_ops(lay, acts, got=got)
    # and the next unstructured restructure draws against the input pattern
    # (the occupancy bits the finished rows had changed are restored)
    src = L.restructure(900, seed=7, step=4)
    torch.cuda.synchronize()
    ro, co, so, _ = oracle.restructure(400, 600, lay.row, lay.col, oracle.as_f64(lay.val), 900, 7, 4)
    assert np.array_equal(L.row.cpu().numpy(), ro) and np.array_equal(L.col.cpu().numpy(), co)
    assert np.array_equal(src.cpu().numpy(), so.astype(np.int32))
    L.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_restructure_mixed_chain(dtype):
    # Per-row and unstructured restructures alternate on one handle (the
    # unstructured ones pruning a tenth, updated in place, and a third,
    # rebuilt): each draws against the pattern the one before left, as the
    # oracle chain does, and every op of the last pattern matches the oracle.
    out_f, in_f = 600, 800
    lay = wl.make_layer(out_f, in_f, fan_in=40, val_std=0.5, val_dtype=dtype, seed=5, bias="normal")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(out_f, in_f, row, col, val, bias, max_batch=16)
    r, c, v = lay.row, lay.col, lay.val
    for step, (kind, n) in enumerate((("rows", 4), ("all", 2400), ("rows", 6), ("all", 8000), ("all", 2400))):
        if kind == "rows":
            src = L.restructure_rows(n, 3, step)
            r, c, so, _ = oracle.restructure_rows(out_f, in_f, r, c, oracle.as_f64(v, dtype), n, 3, step)
        else:
            src = L.restructure(n, seed=3, step=step)
            r, c, so, _ = oracle.restructure(out_f, in_f, r, c, oracle.as_f64(v, dtype), n, 3, step)
        torch.cuda.synchronize()
        v = oracle.restructure_values(v, so)
        assert np.array_equal(L.row.cpu().numpy(), r) and np.array_equal(L.col.cpu().numpy(), c), step
        assert np.array_equal(src.cpu().numpy(), so.astype(np.int32)), step
    new = wl.Layer(out_f, in_f, r, c, v, lay.bias, dtype)
    for batch in (4, 16):
        acts = wl.make_acts(batch, in_f, out_f, dtype, seed=batch)
        x, dy = act_tensor(acts.x, dtype), act_tensor(acts.dy, dtype)
        got = {"y": L.forward(x), "dx": L.grad_input(dy)}
        got["dw"], got["db"] = L.grad_weight(x, dy)
        torch.cuda.synchronize()
        check_layer_ops(new, acts, got=got)
    L.close()


def test_restructure_rows_errors():
    lay = wl.make_layer(4, 8, fan_in=8, val_dtype="f32", seed=1)  # every row full
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(4, 8, row, col, val, bias, max_batch=4)
    with pytest.raises(snack.SnackError) as e:
        L.restructure_rows(1, 0, 0)
    assert e.value.status == 8  # NO_SPACE
    with pytest.raises(snack.SnackError) as e:
        L.restructure_rows(257, 0, 0)
    assert e.value.status == 7  # UNSUPPORTED
    L.close()
    wide = wl.make_layer(3, 70000, fan_in=5, val_dtype="f32", seed=1)
    row, col, val, bias = layer_tensors(wide)
    L = snack.SparseLinear(3, 70000, row, col, val, bias, max_batch=4)
    with pytest.raises(snack.SnackError) as e:
        L.restructure_rows(1, 0, 0)
    assert e.value.status == 7
    L.close()


# ---------------------------------------------------------------- kernel trace

def _ident(name: str) -> str:
    import re
    m = re.search(r"(k_[A-Za-z0-9_]*?)(?:I|E|$|<|\()", name)
    return m.group(1) if m else name


def test_kernel_trace_records_every_launch():
    # The trace brackets every launch of the calling thread with two events:
    # a small-batch forward is one kernel, a tile-path forward several
    # (transpose, tiles, ...); a ring of two keeps the last two records; the
    # results are bit-identical with and without the trace.
    lay = wl.make_layer(300, 400, nnz=20000, val_std=0.3, val_dtype="f32", seed=3, bias="normal")
    row, col, val, bias = layer_tensors(lay)
    L = snack.SparseLinear(300, 400, row, col, val, bias, max_batch=32)
    x32 = act_tensor(wl.make_acts(32, 400, 300, "f32", seed=1).x, "f32")
    x4 = act_tensor(wl.make_acts(4, 400, 300, "f32", seed=2).x, "f32")
    ref32, ref4 = L.forward(x32), L.forward(x4)
    torch.cuda.synchronize()
    snack.snack_trace_start(64)
    try:
        y4 = L.forward(x4)
        y32 = L.forward(x32)
        recs = snack.snack_trace_read(64)
        idents = [_ident(n) for n, _ in recs]
        assert idents[0] == "k_spmm_small" and "k_spmm_tiles" in idents[1:] and "k_transpose" in idents[1:], idents
        assert all(us > 0.0 for _, us in recs)
        snack.snack_trace_start(2)  # restarts with an empty ring
        for _ in range(3):
            L.forward(x4)
        recs2 = snack.snack_trace_read(10)
        assert [_ident(n) for n, _ in recs2] == ["k_spmm_small"] * 2
    finally:
        snack.snack_trace_stop()
    torch.cuda.synchronize()
    assert torch.equal(y32, ref32) and torch.equal(y4, ref4)
    L.close()
