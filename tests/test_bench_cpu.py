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
