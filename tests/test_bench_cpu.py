"""Host-side checks of bench.py's bookkeeping (no GPU): the kernel launches it
claims per step agree with the committed ncu launch list, and the DRAM
traffic it reports is taken only from a profile of the current kernels."""

import os
import re

import bench


def test_launches_per_step_match_the_launch_list():
    path = os.path.join(bench.ROOT, "profiles", "launches_c4_step.md")
    text = open(path).read()
    m = re.search(r"\((\d+) launches\)", text)
    assert m, "launch list summary has no launch count"
    # fwd: transpose, tiles, fix-up; backward: both transposes, tiles, fix-up
    assert 3 + 3 + bench.restructure_launches() == int(m.group(1))
    per_op = dict(re.findall(r"^\| (fwd|bwd|restructure) \| (\d+) \|", text, flags=re.M))
    assert int(per_op["restructure"]) == bench.restructure_launches()


def test_traffic_only_for_matching_kernel_sources(monkeypatch):
    monkeypatch.setattr(bench, "kernel_digest", lambda: "not-these-sources")
    assert bench.profiled_traffic("restructure") is None
    assert bench.profiled_traffic("fwd") is None


def test_algorithmic_bytes_formulas():
    b = bench.alg_bytes(nnz=100, batch=2, out_f=10, in_f=20)
    # fwd: indices + values once, X and Y once, bias
    assert b["fwd"] == 100 * 12 + 2 * 20 * 4 + 2 * 10 * 4 + 4 * 10
    # restructure: read the old COO, write the new COO (the scope table's floor; source map not counted)
    assert b["restructure"] == 2 * 100 * 12


def test_kernel_identifiers_from_runtime_names():
    # mangled names (as the CUDA runtime reports them) and demangled ones (ncu)
    cases = {
        "_ZN5snack12_GLOBAL__N_112k_spmm_tilesIffLi4ELi8ELb1ELb1EEEvNS_10SpmmParamsE": "k_spmm_tiles",
        "_ZN5snack12_GLOBAL__N_112k_merge_keptINS0_6ColPolELi2EEEvT_NS0_6MkArgsE": "k_merge_kept",
        "_ZN5snack12_GLOBAL__N_17k_tilesEPKiiliiiPi": "k_tiles",
        "_ZN5snack12_GLOBAL__N_112k_transpose2IfEEvNS_13TransposePairIT_EEii": "k_transpose2",
        "k_merge_kept<RowPol<float, unsigned int>, 1>": "k_merge_kept",
        "k_bkt_rank": "k_bkt_rank",
    }
    for name, ident in cases.items():
        assert bench.kernel_ident(name) == ident, name


def test_kernel_times_aggregate_the_trace_by_op():
    # a fake trace of two steps: 1 fwd launch, 1 bwd launch, 3 restructure
    # launches (two merges told apart by order); every step's records form
    # one block in launch order
    launches = {"fwd": 1, "bwd": 1, "restructure": 3}
    step_recs = [("k_spmm_tiles", 10.0), ("k_spmm_tiles", 20.0), ("k_merge_kept", 5.0), ("k_draw", 1.0),
                 ("k_merge_kept", 7.0)]

    class FakeSnack:
        def __init__(self):
            self.recs = []

        def snack_trace_start(self, cap):
            self.recs = []

        def snack_wait_plan(self, h, stream):
            pass

        def snack_trace_read(self, n):
            return self.recs[-n:]

        def snack_trace_stop(self):
            pass

    fake = FakeSnack()

    class FakeStream:
        def synchronize(self):
            pass

    def step(cp, i):
        fake.recs.extend(step_recs)

    out = bench.kernel_times(fake, step, [{"h": 0}], FakeStream(), 2, launches)
    assert out[("fwd", "k_spmm_tiles")]["us_per_launch"] == 10.0
    assert out[("bwd", "k_spmm_tiles")]["us_per_step"] == 20.0
    assert out[("restructure", "k_merge_kept:0")]["us_per_step"] == 5.0
    assert out[("restructure", "k_merge_kept:1")]["us_per_step"] == 7.0
    assert out[("restructure", "k_draw")]["launches_per_step"] == 1
