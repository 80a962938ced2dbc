"""Benchmark of the truly sparse layer on GB300: one step = forward SpMM,
input-gradient SpMM, weight-gradient SDDMM (+ bias gradient) and one DST
restructure (prune 10 % smallest |w|, regrow at random empty positions) of a
16384 x 16384 layer at 99 % sparsity with Zipf(1.2) row lengths, fp32, batch 32.

Prints one JSON line.  `value` is algorithmic bytes per second over the step
(bytes of indices + values + activations each op must move, summed over the
four ops, divided by the device time of the step), inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (fp64, the machine's host cores) on the same
workload and metric.  Under torchrun (N > 1) every rank runs an independent
replica of the layer on its own GPU (no collective on the data path); rank 0
prints the aggregate.
"""

from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SpMM fwd/dx/dw µs, GB/s and % of GB300 HBM roofline at 90–99% sparsity"
WORKLOAD = ("16384x16384 sparse linear layer, 99% sparse (nnz 2,684,355, row lengths Zipf s=1.2), fp32 values "
            "N(0,0.02), batch 32 fp32 X,dY ~ N(0,1); step = fwd + backward (dX + dW + db in one fused pass) + "
            "DST restructure (prune 10% smallest |w| = 268,435, regrow as many at uniform empty positions)")
OUT_F = IN_F = 16384
BATCH = 32
PRUNE_FRAC = 0.10
N_COPIES = 8  # rotating layer copies: consecutive steps never find their inputs in L2


def alg_bytes(nnz: int, batch: int, out_f: int, in_f: int, s_v: int = 4, s_x: int = 4) -> dict:
    """Bytes each op must move at least (indices + values + activations once).

    fwd/dx/dw are the single ops; bwd is dx and dw together (snack_backward),
    which reads the pattern and the values once: pattern + values + dW out +
    X + dY in + dX out + db out."""
    fwd = nnz * (8 + s_v) + batch * in_f * s_x + batch * out_f * s_x + 4 * out_f
    dx = nnz * (8 + s_v) + batch * out_f * s_x + batch * in_f * s_x
    dw = nnz * (8 + 4) + batch * in_f * s_x + batch * out_f * s_x + 4 * out_f
    bwd = nnz * (8 + s_v + 4) + 2 * batch * in_f * s_x + batch * out_f * s_x + 4 * out_f
    restructure = 2 * nnz * (8 + s_v)  # read the old COO, write the new one (the 4 B/weight source map not counted)
    return {"fwd": fwd, "dx": dx, "dw": dw, "bwd": bwd, "restructure": restructure}


STEP_OPS = ("fwd", "bwd", "restructure")


def measured_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_digest() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "spmm_row_sorted_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(op: str, kernel: str = None):
    """DRAM bytes per call of `op` (or, with `kernel`, of that kernel of the op per call) from the
    committed ncu summary, if the kernels are unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic_c4.md")
    if not os.path.exists(path):
        return None
    want = kernel_digest()
    with open(path) as f:
        for line in f:
            if line.startswith("traffic:"):
                try:
                    d = json.loads(line[len("traffic:"):])
                except ValueError:
                    return None
                if d.get("kernel_digest") != want:
                    return None
                table, key = (d.get("kernel_bytes", {}), f"{op}:{kernel}") if kernel else (d.get("bytes_per_call", {}), op)
                return int(table[key]) if key in table else None
    return None


def kernel_ident(name: str) -> str:
    """The kernel's identifier (k_...) from the name the CUDA runtime gives (mangled or not)."""
    import re
    m = re.search(r"(k_[A-Za-z0-9_]*?)(?:I|E|$|<|\()", name)
    if m:
        return m.group(1)
    m = re.search(r"(k_[A-Za-z0-9_]+)", name)
    return m.group(1) if m else name


class ClockSampler:
    """Samples nvidia-smi during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


NVML_POLL = r"""
import ctypes, sys, time
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    sys.exit(1)
h = ctypes.c_void_p()
if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(sys.argv[1].encode()), ctypes.byref(h)) != 0:
    sys.exit(1)
mx = ctypes.c_uint()
nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
period = float(sys.argv[2])
mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
print("max", mx.value, flush=True)
while True:
    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
        r = rs.value if reasons(h, ctypes.byref(rs)) == 0 else 0
        print(time.monotonic(), mhz.value, r, flush=True)
    time.sleep(period)
"""


class NvmlClockSampler:
    """Polls NVML (libnvidia-ml through ctypes, read-only queries) every
    `period_s` from a separate process: the SM clock, its maximum and the
    active clock-event reasons.  The samples whose time falls inside the timed
    region are kept, so a region of a few milliseconds still gets samples
    (nvidia-smi's loop gives one per 100 ms); polling from another process
    leaves the launching thread alone.  No samples when NVML is missing."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device_index: int, period_s: float = 0.0005):
        self.period = period_s
        self.rows = []
        self.max_mhz = None
        self.proc = None
        self.t0 = self.t1 = None
        try:
            import torch

            pr = torch.cuda.get_device_properties(torch_device_index)
            self.bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
            self.ok = True
        except Exception:
            self.ok = False

    @property
    def handle(self):
        return self.ok or None

    def _read(self):
        for line in self.proc.stdout:
            parts = line.split()
            if parts and parts[0] == "max":
                self.max_mhz = float(parts[1])
                self.ready.set()
            elif len(parts) == 3:
                self.rows.append((float(parts[0]), float(parts[1]), int(parts[2])))

    def __enter__(self):
        if self.ok:
            self.ready = threading.Event()
            self.proc = subprocess.Popen([sys.executable, "-c", NVML_POLL, self.bus, str(self.period)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            self.ready.wait(timeout=10)
            time.sleep(0.005)
        self.t0 = time.monotonic()
        return self

    def __exit__(self, *exc):
        self.t1 = time.monotonic()
        if self.proc is not None:
            time.sleep(0.002)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        inside = [(m, r) for t, m, r in self.rows if self.t0 is not None and self.t0 <= t <= self.t1]
        src = f"nvml from a separate process every {self.period * 1e3:.1f} ms, samples inside the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": src}
        reasons = sorted({n for _, r in inside for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in inside), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(m for m, _ in inside), "reasons": reasons, "samples": len(inside), "source": src}


def clock_sampler(index: int):
    """NVML sampler when NVML loads, else the nvidia-smi one."""
    s = NvmlClockSampler(index)
    return s if s.handle is not None else ClockSampler(index)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest replica's)."""
    if world <= 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every replica moves its own bytes in the slowest replica's time."""
    return world * bytes_per_step_per_rank / (ms_per_step / 1e3) / 1e9


def make_workload(seed: int):
    from spmm_row_sorted_gb300 import workloads as wl

    lay = wl.make_layer(OUT_F, IN_F, density=0.01, val_std=0.02, val_dtype="f32", seed=seed, zipf_s=1.2)
    acts = wl.make_acts(BATCH, IN_F, OUT_F, "f32", seed=seed)
    return lay, acts


def sub_layer(lay, r0: int, nrows: int):
    """Rows [r0, r0+nrows) of the layer as a layer of their own (same columns)."""
    from spmm_row_sorted_gb300 import workloads as wl

    lo, hi = np.searchsorted(lay.row, [r0, r0 + nrows])
    return wl.Layer(nrows, lay.in_f, (lay.row[lo:hi] - r0).astype(np.int32), lay.col[lo:hi].copy(),
                    lay.val[lo:hi].copy(), lay.bias[r0:r0 + nrows].copy(), lay.val_dtype)


class OracleSampler:
    """Times the fp64 oracle on row-block samples of the workload.

    A sample is the sub-layer of `nrows` consecutive output rows (all input
    columns, full batch); one sample step runs forward, input gradient, weight
    gradient and a 10 % restructure of that sub-layer.  Its algorithmic bytes
    follow the same formula as the GPU step (forward, backward, restructure),
    so bytes/second compare directly.
    """

    def __init__(self, lay, acts):
        import oracle

        self.oracle = oracle
        self.threads = os.cpu_count() or 1
        oracle.set_threads(self.threads)
        self.lay, self.acts = lay, acts
        self.x64 = oracle.as_f64(acts.x)
        self.dy64_full = oracle.as_f64(acts.dy)
        self.cursor = 0

    def step(self, nrows: int, step_index: int):
        o = self.oracle
        r0 = self.cursor
        nrows = min(nrows, OUT_F - r0)
        self.cursor = (r0 + nrows) % OUT_F
        sub = sub_layer(self.lay, r0, nrows)
        v64 = o.as_f64(sub.val)
        dy64 = np.ascontiguousarray(self.dy64_full[:, r0:r0 + nrows])
        n_prune = int(PRUNE_FRAC * sub.nnz)
        t0 = time.perf_counter()
        o.fwd(nrows, IN_F, sub.row, sub.col, v64, self.x64, o.as_f64(sub.bias))
        o.dx(nrows, IN_F, sub.row, sub.col, v64, dy64)
        o.dw(nrows, IN_F, sub.row, sub.col, self.x64, dy64)
        o.restructure(nrows, IN_F, sub.row, sub.col, v64, n_prune, 0, step_index)
        dt = time.perf_counter() - t0
        b = alg_bytes(sub.nnz, BATCH, nrows, IN_F)
        return dt, sum(b[op] for op in STEP_OPS), nrows

    def rows_for(self, seconds: float) -> int:
        """Rows per sample so that one sample step takes about `seconds`."""
        dt, _, n = self.step(1024, 0)
        self.cursor = 0
        rows = int(1024 * seconds / max(dt, 1e-6))
        return max(16, min(OUT_F, rows))


def time_oracle(lay, acts, seconds_total: float, steps: int, warmup: int):
    s = OracleSampler(lay, acts)
    rows = s.rows_for(seconds_total / max(1, steps + warmup))
    for i in range(warmup):
        s.step(rows, i)
    tsum, bsum, rsum = 0.0, 0, 0
    for i in range(steps):
        dt, b, r = s.step(rows, warmup + i)
        tsum += dt
        bsum += b
        rsum += r
    sample = (f"{steps} sample steps of {rows} consecutive output rows x 16384 inputs each (fwd+dx+dw+restructure "
              f"of that row block, batch 32), {rsum} rows in all, fp64 oracle on {s.threads} threads")
    return bsum / tsum / 1e9, tsum / steps, sample, s.threads


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    lay, acts = make_workload(0)
    value, sec, sample, threads = time_oracle(lay, acts, seconds_total=args.cpu_seconds_total, steps=args.steps,
                                              warmup=args.warmup)
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from spmm_row_sorted_gb300 import build as snack_build
    from spmm_row_sorted_gb300 import snack

    snack_build.build()
    snack.load()
    lay, acts = make_workload(rank)
    nnz = lay.nnz
    n_prune = int(PRUNE_FRAC * nnz)
    byts = alg_bytes(nnz, BATCH, OUT_F, IN_F)
    step_bytes = sum(byts[op] for op in STEP_OPS)

    # the step's stream above the lowest priority: the column-view update a
    # restructure leaves running (on a stream of the lowest priority) then
    # fills the gaps of the next step's kernels instead of competing with them
    stream = torch.cuda.Stream(device=dev, priority=-1)
    plan_b, ws_b = snack.snack_query_sizes(OUT_F, IN_F, nnz, BATCH, 0, 0)
    copies = []
    with torch.cuda.stream(stream):
        row0 = torch.from_numpy(lay.row).to(dev)
        col0 = torch.from_numpy(lay.col).to(dev)
        val0 = torch.from_numpy(lay.val).to(dev)
        bias = torch.from_numpy(lay.bias).to(dev)
        x0 = torch.from_numpy(acts.x).to(dev)
        dy0 = torch.from_numpy(acts.dy).to(dev)
        for c in range(1 if args.profile else N_COPIES):
            # a step's inputs (X, dY) and results (Y, dX, db, dW) each in one
            # buffer, so the end-to-end loop moves them with one copy per
            # direction (every part starts on a 16-byte boundary)
            inp = torch.empty(BATCH * IN_F + BATCH * OUT_F, device=dev)
            out = torch.empty(BATCH * OUT_F + BATCH * IN_F + OUT_F + nnz, device=dev)
            cp = {"row": [row0.clone(), torch.empty_like(row0)], "col": [col0.clone(), torch.empty_like(col0)],
                  "val": [val0.clone(), torch.empty_like(val0)], "cur": 0, "src": torch.empty_like(row0),
                  "inp": inp, "out": out, "bias": bias.clone(),
                  "x": inp[:BATCH * IN_F].view(BATCH, IN_F), "dy": inp[BATCH * IN_F:].view(BATCH, OUT_F),
                  "y": out[:BATCH * OUT_F].view(BATCH, OUT_F),
                  "dx": out[BATCH * OUT_F:BATCH * OUT_F + BATCH * IN_F].view(BATCH, IN_F),
                  "db": out[BATCH * (OUT_F + IN_F):BATCH * (OUT_F + IN_F) + OUT_F],
                  "dw": out[BATCH * (OUT_F + IN_F) + OUT_F:],
                  "plan": torch.empty(plan_b, dtype=torch.uint8, device=dev)}
            cp["x"].copy_(x0)
            cp["dy"].copy_(dy0)
            copies.append(cp)
        ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
    stream.synchronize()
    for cp in copies:
        cp["h"] = snack.snack_create(OUT_F, IN_F, nnz, BATCH, 0, 0, cp["row"][0], cp["col"][0], cp["plan"], ws,
                                     validate=True, stream=stream)
    rws = max(snack.snack_restructure_workspace_size(copies[0]["h"], n_prune), ws_b)
    ws = torch.empty(rws, dtype=torch.uint8, device=dev)
    stream.synchronize()

    def step(cp, i, ev=None):
        cur = cp["cur"]
        row, col, val = cp["row"][cur], cp["col"][cur], cp["val"][cur]
        if ev is not None:
            ev[0].record(stream)
        snack.snack_spmm_fwd(cp["h"], row, col, val, cp["x"], BATCH, cp["bias"], cp["y"], ws, stream)
        if ev is not None:
            ev[1].record(stream)
        snack.snack_backward(cp["h"], row, col, val, cp["x"], cp["dy"], BATCH, cp["dx"], cp["dw"], cp["db"], ws,
                             stream)
        if ev is not None:
            ev[2].record(stream)
        nxt = 1 - cur
        snack.snack_restructure(cp["h"], row, col, val, n_prune, 12345, i, cp["row"][nxt], cp["col"][nxt],
                                cp["val"][nxt], cp["src"], ws, stream)
        if ev is not None:
            ev[3].record(stream)
        cp["cur"] = nxt

    if args.profile:  # untimed steps on one copy, for profilers (ncu -k ... -c ...)
        for i in range(args.warmup + args.steps):
            step(copies[0], i)
        stream.synchronize()
        for cp in copies:
            snack.snack_destroy(cp["h"])
        print("profile run done", flush=True)
        return 0
    for i in range(args.warmup):
        step(copies[i % N_COPIES], i)
    stream.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STEP_OPS) + 1)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with clock_sampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            step(copies[i % N_COPIES], args.warmup + i, evs[i])
        for cp in copies:  # column-view rebuilds still running on the handles' second streams
            snack.snack_wait_plan(cp["h"], stream)
        t_end.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ops = list(STEP_OPS)
    # Per-op breakdown, outside the timed region: the column-view rebuild a
    # restructure leaves on its handle's second stream overlaps the next
    # step's forward in the timed loop, so there the op events do not isolate
    # the ops.  Here every op starts after all earlier work, and the
    # restructure's time runs until its rebuild has finished as well.
    n_bd = max(1, min(args.steps, 100))
    bd = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_bd)]
    for i in range(n_bd):
        cp = copies[i % N_COPIES]
        for c2 in copies:
            snack.snack_wait_plan(c2["h"], stream)
        e = bd[i]
        step(cp, 2 * 10**6 + i, e[:4])
        snack.snack_wait_plan(cp["h"], stream)
        e[4].record(stream)
    stream.synchronize()
    op_ms = {"fwd": statistics.mean(e[0].elapsed_time(e[1]) for e in bd),
             "bwd": statistics.mean(e[1].elapsed_time(e[2]) for e in bd),
             "restructure": statistics.mean(e[2].elapsed_time(e[4]) for e in bd)}
    restructure_on_stream_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in bd)
    overlapped_ms = {op: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                     for j, op in enumerate(ops)}
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(step_bytes, world, elapsed_ms / args.steps)
    peak, peak_kind = measured_peak_gbs()
    op_report = {}
    for op in ops:
        gbs = byts[op] / (op_ms[op] / 1e3) / 1e9
        flops = {"fwd": 2 * nnz * BATCH, "bwd": 4 * nnz * BATCH}.get(op)
        op_report[op] = {"us": op_ms[op] * 1e3, "alg_bytes": byts[op], "gbs": gbs, "frac": gbs / peak,
                         "gflops": (flops / (op_ms[op] / 1e3) / 1e9) if flops else None,
                         "us_in_timed_loop": overlapped_ms[op] * 1e3}
    op_report["restructure"]["us_until_return"] = restructure_on_stream_ms * 1e3
    launches = {"fwd": 3, "bwd": 3, "restructure": restructure_launches()}
    kern = kernel_times(snack, step, copies, stream, min(args.steps, 50), launches)
    # the dominant kernel: the longest per step among those whose work has a
    # scope-table byte count -- the forward's and the fused backward's tile
    # kernels (their ops' other launches only transpose the activations and
    # add split rows' partial sums) and the restructure's merge (it reads the
    # old COO and writes the new one)
    owns = {("fwd", "k_spmm_tiles"): "fwd", ("bwd", "k_spmm_tiles"): "bwd", ("restructure", "k_merge_kept:0"): "restructure"}
    cands = [(k, v) for k, v in kern.items() if (k[0], k[1]) in owns]
    (dop, dname), dk = max(cands, key=lambda kv: kv[1]["us_per_step"])
    d_op = owns[(dop, dname)]
    d_gbs = byts[d_op] / (dk["us_per_launch"] / 1e6) / 1e9
    longest = max(kern.items(), key=lambda kv: kv[1]["us_per_step"])
    dominant_op = max(ops, key=lambda o: op_ms[o])
    roofline = {"bound": "hbm", "achieved": d_gbs, "peak": peak, "unit": "GB/s", "frac": d_gbs / peak,
                "traffic": profiled_traffic(dop, dname),
                "kernel": f"{dk['name']} ({d_op}; {dk['launches_per_step']} launch per step, "
                          f"{dk['us_per_launch']:.1f} us per launch in the traced pass)",
                "alg_bytes_per_launch": byts[d_op], "us_per_launch": dk["us_per_launch"], "peak_kind": peak_kind,
                "longest_kernel": {"name": longest[1]["name"], "op": longest[0][0],
                                   "us_per_step": longest[1]["us_per_step"]},
                "op": {"name": f"{dominant_op} ({launches[dominant_op]} launches; the op with the largest time share)",
                       "achieved": op_report[dominant_op]["gbs"], "frac": op_report[dominant_op]["frac"],
                       "traffic": profiled_traffic(dominant_op)},
                "kernels_us_per_step": {f"{k[0]}:{k[1]}": round(v["us_per_step"], 2) for k, v in
                                        sorted(kern.items(), key=lambda kv: -kv[1]["us_per_step"])}}

    # end to end through the C ABI from pinned host buffers: every step's inputs
    # go host -> device and its results device -> host inside the timed region,
    # on two copy streams (one per direction) that overlap them with the
    # neighbouring steps' kernels (each layer copy has its own device and pinned
    # host buffers; events order a copy slot's transfers after the step that
    # last used it)
    e2e_steps = max(1, min(args.steps, 200))
    # a step's inputs X and dY, and its results Y, dX, db and dW, each packed
    # in one pinned host buffer: one copy per direction and step
    hin = torch.cat([torch.from_numpy(acts.x).reshape(-1), torch.from_numpy(acts.dy).reshape(-1)]).pin_memory()
    host_out = [torch.empty(copies[0]["out"].numel()).pin_memory() for _ in range(min(N_COPIES, e2e_steps))]
    h2d = hin.numel() * 4
    d2h = host_out[0].numel() * 4
    hs, ds = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    slots = len(host_out)
    # events made once: a slot's inputs landed, its step ran, its results reached the host
    ready_ev = [torch.cuda.Event() for _ in range(slots)]
    computed_ev = [torch.cuda.Event() for _ in range(slots)]
    drained_ev = [torch.cuda.Event() for _ in range(slots)]
    computed = [None] * slots  # event after the last step that used a slot
    drained = [None] * slots   # event after that step's results reached the host
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    hs.wait_event(e0)
    ds.wait_event(e0)

    def load_inputs(j):
        """Queue step j's host -> device input copy on the H2D stream."""
        cj = j % slots
        if computed[cj] is not None:
            hs.wait_event(computed[cj])  # the slot's previous step has read its inputs
        with torch.cuda.stream(hs):
            copies[cj]["inp"].copy_(hin, non_blocking=True)
        ready_ev[cj].record(hs)

    load_inputs(0)
    for i in range(e2e_steps):
        c = i % slots
        cp = copies[c]
        stream.wait_event(ready_ev[c])
        if drained[c] is not None:
            stream.wait_event(drained[c])  # the slot's previous results have left the device
        if i + 1 < e2e_steps:
            # the next step's inputs go in while this step runs, queued before this
            # step's restructure holds the host at its read-back (a training loop's prefetch)
            load_inputs(i + 1)
        step(cp, 10**6 + i)
        computed[c] = computed_ev[c]
        computed[c].record(stream)
        ds.wait_event(computed[c])
        with torch.cuda.stream(ds):
            host_out[c].copy_(cp["out"], non_blocking=True)
        drained[c] = drained_ev[c]
        drained[c].record(ds)
    for d in drained:
        if d is not None:
            stream.wait_event(d)
    for cp in copies:
        snack.snack_wait_plan(cp["h"], stream)
    e1.record(stream)
    stream.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e = {"value": job_throughput(step_bytes, world, e2e_ms), "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "copies": "overlapped on two copy streams"}

    launches_per_step = 3 + 3 + restructure_launches()  # fwd: transpose, tiles, fixup; bwd: both transposes (+ db), tiles, fixup
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": f"inputs larger than L2: {N_COPIES} rotating layer copies",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "ops": op_report, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cval, _, sample, threads = time_oracle(lay, acts, seconds_total=args.cpu_seconds, steps=10, warmup=0)
        line["cpu_baseline"] = {"value": cval, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample}
    for cp in copies:
        snack.snack_destroy(cp["h"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def kernel_times(snack, step, copies, stream, n_steps: int, launches: dict) -> dict:
    """Per-kernel device times from the library's kernel trace over n_steps steps (after the timed
    region): every launch bracketed by two events, so each kernel runs alone and its time includes
    its launch.  Keyed by (op, identifier), the restructure's two merges told apart as :0 and :1 in
    launch order; values: name, launches and us per step, us per launch."""
    per_step = sum(launches.values())
    snack.snack_trace_start(per_step * n_steps + 64)
    for i in range(n_steps):
        for c2 in copies:
            snack.snack_wait_plan(c2["h"], stream)
        step(copies[i % len(copies)], 3 * 10**6 + i)
    for cp in copies:
        snack.snack_wait_plan(cp["h"], stream)
    stream.synchronize()
    recs = snack.snack_trace_read(per_step * n_steps + 64)
    snack.snack_trace_stop()
    recs = recs[-per_step * n_steps:]
    bounds = [("fwd", launches["fwd"]), ("bwd", launches["bwd"]), ("restructure", launches["restructure"])]
    out = {}
    for s0 in range(0, len(recs), per_step):
        block, pos = recs[s0:s0 + per_step], 0
        for op, cnt in bounds:
            seen = {}
            for name, us in block[pos:pos + cnt]:
                ident = kernel_ident(name)
                if ident == "k_merge_kept":  # the row-order merge, then the column view's
                    ident = f"k_merge_kept:{seen.setdefault('mk', 0)}"
                    seen["mk"] += 1
                d = out.setdefault((op, ident), {"name": ident.split(":")[0], "us": 0.0, "launches": 0})
                d["us"] += us
                d["launches"] += 1
            pos += cnt
    for d in out.values():
        d["us_per_step"] = d["us"] / n_steps
        d["launches_per_step"] = d["launches"] // n_steps
        d["us_per_launch"] = d["us"] / d["launches"]
    return out


# ----------------------------------------------------------------------------
# Per-workload sweep (--configs): every op of every workload, cold and warm,
# beside same-run cuBLAS dense and Dense+Mask comparators and the oracle.
# ----------------------------------------------------------------------------

L2_BYTES = 129 * 2**20
NOMINAL_HBM_GBS = 8000.0
# fp32 FMA peak from unit counts and clock: 152 SMs x 128 fp32 lanes x 2 flop x 2.07 GHz
FMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
ACT_BYTES = {"f32": 4, "bf16": 2}


def _dev_tensor(a, dtype: str, dev):
    import torch

    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(dev)


class _Timer:
    """CUDA-event timing of an enqueue function on one stream: median over reps,
    cold (a read of 2x L2 before every rep) or warm (back-to-back reps)."""

    def __init__(self, torch, stream, dev):
        self.torch, self.s = torch, stream
        self.flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def graph(self, fn):
        """fn captured in a CUDA graph (returns its replay), or fn itself if capture fails."""
        torch = self.torch
        with torch.cuda.stream(self.s):
            fn()
            fn()
        self.s.synchronize()
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g, stream=self.s):
                fn()
        except Exception:
            torch.cuda.synchronize()
            return fn, False
        return g.replay, True

    def time(self, run, reps: int, cold: bool) -> float:
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(self.s):
            for _ in range(3):
                run()
            # hold the stream for a few ms so the host queues every rep before the
            # first one runs: the events then time the device, not launch latency
            torch.cuda._sleep(int(2e6 + 1e5 * reps))
            for e0, e1 in evs:
                if cold:
                    torch.sum(self.flush, dim=0, out=self.flush_out)
                e0.record(self.s)
                run()
                e1.record(self.s)
        self.s.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3

    def time_restructure(self, snack, h, run, reps: int, cold: bool, prep=None) -> tuple:
        """A restructure call timed alone: each rep starts after the previous call's column-view
        update (snack_wait_plan), `prep` (untimed) and, cold, a read of 2x L2; the device sleeps
        briefly so the host queues the call's first launches before they run.  Medians of the time
        until the call returns and until its column-view update is done, in us."""
        torch = self.torch
        ret, done = [], []
        with torch.cuda.stream(self.s):
            for _ in range(3):
                if prep is not None:
                    prep()
                run()
            for _ in range(reps):
                snack.snack_wait_plan(h, self.s)
                if prep is not None:
                    prep()
                if cold:
                    torch.sum(self.flush, dim=0, out=self.flush_out)
                torch.cuda._sleep(int(1e5))
                e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                e0.record(self.s)
                run()
                e1.record(self.s)
                snack.snack_wait_plan(h, self.s)
                e2.record(self.s)
                ret.append((e0, e1))
                done.append((e0, e2))
            snack.snack_wait_plan(h, self.s)
        self.s.synchronize()
        return (statistics.median(a.elapsed_time(b) for a, b in ret) * 1e3,
                statistics.median(a.elapsed_time(b) for a, b in done) * 1e3)


def _oracle_us(oracle, lay, x64, dy64, op: str, budget_terms: float = 3e7) -> tuple:
    """Oracle time of `op` on the layer: the whole layer when nnz*batch is small,
    else the first rows holding about budget_terms terms, scaled by nnz."""
    batch = x64.shape[0]
    frac = min(1.0, budget_terms / max(1.0, lay.nnz * batch))
    if frac >= 1.0:
        sub, dys = lay, dy64
    else:
        per_row = np.cumsum(np.bincount(lay.row, minlength=lay.out_f))
        nrows = max(1, min(lay.out_f, int(np.searchsorted(per_row, lay.nnz * frac)) + 1))
        sub = sub_layer(lay, 0, nrows)
        dys = np.ascontiguousarray(dy64[:, :nrows])
    v64 = oracle.as_f64(sub.val, sub.val_dtype)
    t0 = time.perf_counter()
    if op == "fwd":
        oracle.fwd(sub.out_f, sub.in_f, sub.row, sub.col, v64, x64, oracle.as_f64(sub.bias))
    elif op == "dx":
        oracle.dx(sub.out_f, sub.in_f, sub.row, sub.col, v64, dys)
    elif op == "dw":
        oracle.dw(sub.out_f, sub.in_f, sub.row, sub.col, x64, dys)
    elif op == "restructure":
        oracle.restructure(sub.out_f, sub.in_f, sub.row, sub.col, v64, int(PRUNE_FRAC * sub.nnz), 0, 0)
    dt = time.perf_counter() - t0
    scale = lay.nnz / max(1, sub.nnz)
    return dt * scale * 1e6, (sub.nnz == lay.nnz)


def _layer_rows(name, lay, batch, ours, dense, mask, oracle_t, peak, cores):
    """Result records of one layer at one batch."""
    c = _config(name)
    s_v, s_x = ACT_BYTES[lay.val_dtype], ACT_BYTES[c["act_dtype"]]
    byts = alg_bytes(lay.nnz, batch, lay.out_f, lay.in_f, s_v=s_v, s_x=s_x)
    out = []
    for op, t in ours.items():
        cold, warm, graphed = t
        base = "restructure" if op.startswith("restructure") else op  # every restructure row: its bytes
        flops = {"fwd": 2, "dx": 2, "dw": 2, "bwd": 4}.get(op, 0) * lay.nnz * batch
        gbs = byts[base] / (cold * 1e-6) / 1e9
        rec = {"config": name, "layer": f"{lay.out_f}x{lay.in_f}", "nnz": lay.nnz, "batch": batch, "op": op,
               "dtype": lay.val_dtype, "us_cold": cold, "us_warm": warm, "graph": graphed,
               "alg_bytes": byts[base], "gbs": gbs, "frac_measured": gbs / peak, "frac_nominal": gbs / NOMINAL_HBM_GBS,
               "gflops": flops / (cold * 1e-6) / 1e9 if flops else None,
               "frac_fma": (flops / (cold * 1e-6) / 1e12 / FMA_PEAK_TFLOPS) if flops else None,
               "dense_us": dense.get(op), "dense_mask_us": mask.get(op),
               "oracle_us": oracle_t.get(op, (None, None))[0], "oracle_full": oracle_t.get(op, (None, None))[1],
               "oracle_cores": cores}
        out.append(rec)
    return out


# The 16384^2 layer with a constant fan-in of 164 (99 % sparse), as the
# structured DST variant keeps it: not one of the five workloads, timed in the
# c4 sweep beside them.
FANIN_CONFIG = dict(name="16384x16384 constant fan-in 164 (99%), fp32, batch 32", out_f=16384, in_f=16384,
                    val_dtype="f32", act_dtype="f32", batches=(32,), ops=("fwd", "dx", "dw"))


def _config(name):
    from spmm_row_sorted_gb300 import workloads as wl

    return FANIN_CONFIG if name == "c4-fanin" else wl.CONFIGS[name]


def _bench_layer(torch, F, snack, timer, name, lay, batch, ops, reps, dev, oracle, cores):
    """Times our ops and the two dense comparators on one layer and batch."""
    from spmm_row_sorted_gb300 import workloads as wl

    c = _config(name)
    act = c["act_dtype"]
    tdt = torch.float32 if act == "f32" else torch.bfloat16
    acts = wl.make_acts(batch, lay.in_f, lay.out_f, act, seed=0)
    row = torch.from_numpy(lay.row).to(dev)
    col = torch.from_numpy(lay.col).to(dev)
    val = _dev_tensor(lay.val, lay.val_dtype, dev)
    bias = torch.from_numpy(lay.bias).to(dev)
    x = _dev_tensor(acts.x, act, dev)
    dy = _dev_tensor(acts.dy, act, dev)
    L = snack.SparseLinear(lay.out_f, lay.in_f, row, col, val, bias, max_batch=batch, validate=True)
    y = torch.empty((batch, lay.out_f), dtype=tdt, device=dev)
    dx = torch.empty((batch, lay.in_f), dtype=tdt, device=dev)
    dw = torch.empty(lay.nnz, dtype=torch.float32, device=dev)
    db = torch.empty(lay.out_f, dtype=torch.float32, device=dev)
    h, ws = L.handle, L.ws
    fns = {"fwd": lambda: snack.snack_spmm_fwd(h, row, col, val, x, batch, bias, y, ws),
           "dx": lambda: snack.snack_spmm_dx(h, row, col, val, dy, batch, dx, ws),
           "dw": lambda: snack.snack_sddmm_dw(h, row, col, x, dy, batch, dw, db, ws),
           "bwd": lambda: snack.snack_backward(h, row, col, val, x, dy, batch, dx, dw, db, ws)}
    ours = {}
    for op in ops:
        run, graphed = timer.graph(fns[op])
        ours[op] = (timer.time(run, reps, True), timer.time(run, reps, False), graphed)
    if "restructure" in c["ops"]:
        n_prune = int(PRUNE_FRAC * lay.nnz)
        rws = torch.empty(snack.snack_restructure_workspace_size(h, n_prune), dtype=torch.uint8, device=dev)
        bufs = [(row, col, val), (torch.empty_like(row), torch.empty_like(col), torch.empty_like(val))]
        src = torch.empty_like(row)
        state = {"cur": 0, "i": 0}

        def restructure():
            a, b = bufs[state["cur"]], bufs[1 - state["cur"]]
            snack.snack_restructure(h, a[0], a[1], a[2], n_prune, 12345, state["i"], b[0], b[1], b[2], src, rws)
            state["cur"] ^= 1
            state["i"] += 1

        rr = max(20, reps // 4)
        cold, warm = timer.time_restructure(snack, h, restructure, rr, True), timer.time_restructure(snack, h, restructure, rr, False)
        ours["restructure"] = (cold[0], warm[0], False)  # until the call returns
        ours["restructure_all"] = (cold[1], warm[1], False)  # until its column-view update is done
        # Back to back, each call prunes the previous call's regrown zeros (ties at |w| = 0).  With
        # fresh values before every call (the layer's value distribution, as after an optimizer
        # step; untimed) the select sees a continuous distribution instead.
        fresh = torch.from_numpy(lay.val).to(dev)

        def refill():
            bufs[state["cur"]][2].copy_(fresh)

        cold, warm = (timer.time_restructure(snack, h, restructure, rr, True, refill),
                      timer.time_restructure(snack, h, restructure, rr, False, refill))
        ours["restructure_fresh"] = (cold[0], warm[0], False)
        ours["restructure_fresh_all"] = (cold[1], warm[1], False)
        if state["cur"] == 1:  # back on the first buffers
            restructure()
    # comparators: dense W (cuBLAS via F.linear / matmul) and Dense+Mask (W*M materialised every call)
    dense, mask = {}, {}
    Wd = torch.zeros((lay.out_f, lay.in_f), dtype=tdt, device=dev)
    Wd[row.long(), col.long()] = val.to(tdt)
    M = torch.zeros_like(Wd)
    M[row.long(), col.long()] = 1
    bias_t = bias.to(tdt)
    dfns = {"fwd": (lambda: F.linear(x, Wd, bias_t), lambda: F.linear(x, Wd * M, bias_t)),
            "dx": (lambda: dy @ Wd, lambda: dy @ (Wd * M)),
            "dw": (lambda: dy.t() @ x, lambda: (dy.t() @ x) * M),
            "bwd": (lambda: (dy @ Wd, dy.t() @ x), lambda: (dy @ (Wd * M), (dy.t() @ x) * M))}
    for op in ops:
        for store, idx in ((dense, 0), (mask, 1)):
            run, _ = timer.graph(dfns[op][idx])
            store[op] = timer.time(run, reps, True)
    del Wd, M
    oracle_t = {}
    if oracle is not None:
        x64, dy64 = oracle.as_f64(acts.x, act), oracle.as_f64(acts.dy, act)
        for op in list(ops) + (["restructure"] if "restructure" in c["ops"] else []):
            if op != "bwd":
                oracle_t[op] = _oracle_us(oracle, lay, x64, dy64, op)
    L.close()
    return ours, dense, mask, oracle_t


def _c3_step(torch, F, snack, timer, reps, dev):
    """Full sparse-MLP training step (768 -> 3072 GELU -> 768, 1024 tokens): time and
    peak device memory for ours, dense and Dense+Mask."""
    from spmm_row_sorted_gb300 import workloads as wl

    l1, l2 = wl.config_layer("c3", layer_index=0), wl.config_layer("c3", layer_index=1)
    batch = 1024
    x_np = wl.make_acts(batch, 768, 3072, "f32", seed=5).x
    dy_np = wl.make_acts(batch, 3072, 768, "f32", seed=6).dy
    keep = {}

    def measure(setup, graph=False):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        step = setup()
        torch.cuda.synchronize()
        persistent = torch.cuda.memory_allocated(dev) - base
        torch.cuda.reset_peak_memory_stats(dev)
        with torch.cuda.stream(timer.s):
            step()
        timer.s.synchronize()
        peak = torch.cuda.max_memory_allocated(dev) - base
        r = {"us_warm": timer.time(step, reps, False), "persistent_bytes": persistent, "peak_bytes": peak}
        if graph:
            run, ok = timer.graph(step)
            r["us_graph"] = timer.time(run, reps, False) if ok else None
        return r

    def ours_setup():
        t = {}
        for i, lay in enumerate((l1, l2)):
            row = torch.from_numpy(lay.row).to(dev)
            col = torch.from_numpy(lay.col).to(dev)
            val = torch.from_numpy(lay.val).to(dev)
            t[i] = snack.SparseLinear(lay.out_f, lay.in_f, row, col, val, torch.from_numpy(lay.bias).to(dev),
                                      max_batch=batch)
        t["x"] = torch.from_numpy(x_np).to(dev)
        t["dy2"] = torch.from_numpy(dy_np).to(dev)

        def step():
            L1, L2 = t[0], t[1]
            hh, pre = L1.forward_gelu(t["x"])
            L2.forward(hh)
            dy1 = L2.grad_input_gelu(t["dy2"], pre)
            L2.grad_weight(hh, t["dy2"])
            L1.backward(t["x"], dy1)

        keep["ours"] = t
        return step

    def dense_setup(masked):
        def setup():
            ws = []
            for lay in (l1, l2):
                W = torch.zeros((lay.out_f, lay.in_f), device=dev)
                W[torch.from_numpy(lay.row).to(dev).long(), torch.from_numpy(lay.col).to(dev).long()] = \
                    torch.from_numpy(lay.val).to(dev)
                M = (W != 0).float() if masked else None
                ws.append((W.requires_grad_(True), M, torch.zeros(lay.out_f, device=dev, requires_grad=True)))
            x = torch.from_numpy(x_np).to(dev).requires_grad_(True)
            dy2 = torch.from_numpy(dy_np).to(dev)

            def step():
                (W1, M1, b1), (W2, M2, b2) = ws
                hh = F.gelu(F.linear(x, W1 * M1 if masked else W1, b1))
                y2 = F.linear(hh, W2 * M2 if masked else W2, b2)
                y2.backward(dy2)
                for p in (x, W1, W2, b1, b2):
                    p.grad = None

            keep["dense"] = (ws, x, dy2)
            return step

        return setup

    res = {"ours": measure(ours_setup, graph=True)}
    keep["ours"][0].close()
    keep["ours"][1].close()
    keep.clear()
    res["dense"] = measure(dense_setup(False))
    keep.clear()
    res["dense_mask"] = measure(dense_setup(True))
    keep.clear()
    return res


def _fanin_restructure(torch, snack, timer, dev, reps):
    """The structured DST variant on a 16384 x 16384 layer with a constant fan-in of
    164 (99 % sparse): per-row restructure (16 of every row's 164) beside the
    unstructured restructure of the same layer (10 % of all weights)."""
    from spmm_row_sorted_gb300 import workloads as wl

    lay = wl.make_layer(16384, 16384, fan_in=164, val_std=0.02, val_dtype="f32", seed=0)
    row = torch.from_numpy(lay.row).to(dev)
    col = torch.from_numpy(lay.col).to(dev)
    val = torch.from_numpy(lay.val).to(dev)
    L = snack.SparseLinear(16384, 16384, row, col, val, None, max_batch=32)
    h = L.handle
    n_rows = 16
    n_prune = int(PRUNE_FRAC * lay.nnz)
    ws = torch.empty(max(snack.snack_restructure_rows_workspace_size(h, n_rows),
                         snack.snack_restructure_workspace_size(h, n_prune)), dtype=torch.uint8, device=dev)
    bufs = [(row, col, val), (torch.empty_like(row), torch.empty_like(col), torch.empty_like(val))]
    src = torch.empty_like(row)
    state = {"cur": 0, "i": 0}

    def per_row():
        a, b = bufs[state["cur"]], bufs[1 - state["cur"]]
        snack.snack_restructure_rows(h, a[0], a[1], a[2], n_rows, 12345, state["i"], b[0], b[1], b[2], src, ws)
        state["cur"] ^= 1
        state["i"] += 1

    def unstructured():
        a, b = bufs[state["cur"]], bufs[1 - state["cur"]]
        snack.snack_restructure(h, a[0], a[1], a[2], n_prune, 12345, state["i"], b[0], b[1], b[2], src, ws)
        state["cur"] ^= 1
        state["i"] += 1

    out = []
    byts = alg_bytes(lay.nnz, 32, 16384, 16384)["restructure"]
    for name, fn in (("restructure_rows", per_row), ("restructure", unstructured)):
        cold, warm = timer.time_restructure(snack, h, fn, reps, True), timer.time_restructure(snack, h, fn, reps, False)
        for op, k in ((name, 0), (name + "_all", 1)):
            us = cold[k]
            out.append({"config": "c4-fanin", "layer": "16384x16384", "nnz": lay.nnz, "batch": 0, "op": op,
                    "dtype": "f32", "us_cold": us, "us_warm": warm[k], "graph": False,
                    "alg_bytes": byts, "gbs": byts / (us * 1e-6) / 1e9, "frac_measured": None, "frac_nominal": None,
                    "gflops": None, "frac_fma": None, "dense_us": None, "dense_mask_us": None, "oracle_us": None,
                    "oracle_full": None, "oracle_cores": None})
    L.close()
    return out


def run_configs(args):
    import torch
    import torch.nn.functional as F

    from spmm_row_sorted_gb300 import build as snack_build
    from spmm_row_sorted_gb300 import snack
    from spmm_row_sorted_gb300 import workloads as wl

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.backends.cuda.matmul.allow_tf32 = False
    torch.backends.cudnn.allow_tf32 = False
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.no_fan_in_path:  # a copy of the library whose constant-fan-in layers take the general kernels
        snack.load(snack_build.build(extra_flags=["-DSNACK_NO_FAN_IN_PATH"],
                                     out_dir=os.path.join(ROOT, "spmm_row_sorted_gb300", "_build", "no_fan_in")))
    else:
        snack_build.build()
        snack.load()
    peak, peak_kind = measured_peak_gbs()
    oracle, cores = None, None
    if not args.no_cpu_baseline:
        import oracle as _oracle

        oracle = _oracle
        cores = os.cpu_count() or 1
        oracle.set_threads(cores)
    timer = _Timer(torch, torch.cuda.Stream(device=dev), dev)
    names = args.configs.split(",") if args.configs != "all" else list(wl.CONFIGS)
    records = []
    with ClockSampler(0) as clk:
        for name in names:
            c = _config(name)
            if name == "c4-fanin":
                layers = [wl.make_layer(16384, 16384, fan_in=164, val_std=0.02, val_dtype="f32", seed=0)]
            else:
                layers = [wl.config_layer(name, layer_index=i) for i in range(len(c.get("layers", [None])))]
            ops = ["fwd"] if c["ops"] == ("fwd",) else ["fwd", "dx", "dw", "bwd"]
            for lay in layers:
                for batch in c["batches"]:
                    ours, dense, mask, ot = _bench_layer(torch, F, snack, timer, name, lay, batch, ops, args.reps,
                                                         dev, oracle, cores)
                    for rec in _layer_rows(name, lay, batch, ours, dense, mask, ot, peak, cores):
                        records.append(rec)
                        print(json.dumps(rec), flush=True)
            if name == "c4":
                for rec in _fanin_restructure(torch, snack, timer, dev, max(20, args.reps // 4)):
                    rec["frac_measured"] = rec["gbs"] / peak
                    rec["frac_nominal"] = rec["gbs"] / NOMINAL_HBM_GBS
                    records.append(rec)
                    print(json.dumps(rec), flush=True)
            if name == "c3":
                rec = {"config": "c3", "op": "mlp_step", **_c3_step(torch, F, snack, timer, max(20, args.reps // 4),
                                                                     dev)}
                records.append(rec)
                print(json.dumps(rec), flush=True)
    clocks = clk.summary()
    print(json.dumps({"clocks": clocks, "peak_gbs": peak, "peak_kind": peak_kind}), flush=True)
    if args.configs_out:
        with open(args.configs_out, "w") as f:
            f.write(_configs_markdown(records, clocks, peak, peak_kind, cores))
    return 0


def _configs_markdown(records, clocks, peak, peak_kind, cores) -> str:
    def f(v, nd=1):
        return "—" if v is None else f"{v:,.{nd}f}"

    lines = ["| config | layer | batch | op | µs cold | µs warm | alg. MB | GB/s | % HBM (measured) | % of 8 TB/s | "
             "GFLOP/s | cuBLAS dense µs | Dense+Mask µs | oracle µs |",
             "|---|---|---|---|---|---|---|---|---|---|---|---|---|---|"]
    step = None
    for r in records:
        if r.get("op") == "mlp_step":
            step = r
            continue
        orc = f(r["oracle_us"], 0) + ("" if r["oracle_full"] in (None, True) else " (sampled)")
        lines.append(f"| {r['config']} | {r['layer']} | {r['batch']} | {r['op']} | {f(r['us_cold'])} | "
                     f"{f(r['us_warm'])} | {f(r['alg_bytes'] / 1e6, 2)} | {f(r['gbs'], 0)} | "
                     f"{f(100 * r['frac_measured'])} | {f(100 * r['frac_nominal'])} | {f(r['gflops'], 0)} | "
                     f"{f(r['dense_us'])} | {f(r['dense_mask_us'])} | {orc} |")
    out = "\n".join(lines) + "\n"
    if step:
        out += ("\n| c3 MLP training step (both layers, fwd + dX + dW) | µs (warm, eager) | µs (CUDA graph) | "
                "persistent MB | peak MB |\n|---|---|---|---|---|\n")
        for k in ("ours", "dense", "dense_mask"):
            v = step[k]
            out += (f"| {k} | {f(v['us_warm'])} | {f(v.get('us_graph'))} | {f(v['persistent_bytes'] / 1e6, 2)} | "
                    f"{f(v['peak_bytes'] / 1e6, 2)} |\n")
    out += (f"\nPeak HBM {peak:,.0f} GB/s ({peak_kind}); fp32 FMA peak {FMA_PEAK_TFLOPS:.1f} TFLOP/s (units x clock); "
            f"oracle on {cores} host threads; clocks {json.dumps(clocks)}\n")
    return out


def restructure_launches() -> int:
    """Kernel launches of one restructure of the workload (one draw chunk; the column view updated)."""
    # init, draws, acceptance (its scan and the placement in both orders' buckets), rank (both lists)
    regrow = 1 + 1 + 1 + 1
    select = 1 + 1 + 1 + 2 + 1  # init, first digit, bucket listing, two digits over the list, tile keep counts
    merge = 1 + 1 + 1  # tile bounds, merge (also the row offsets), forward tiles
    colview = 1 + 1 + 1  # tile bounds, column-view merge, column tiles (second stream, after the call)
    return regrow + select + merge + colview


# ----------------------------------------------------------------------------
# Gather ceiling (--gather-ceiling): how fast can the SM bring one 128-byte
# batch vector per stored weight to the FMA units, by each route, on the
# 16384^2 Zipf layer at batch 32 fp32?  Probes in probe/gather_probe.cu.
# ----------------------------------------------------------------------------

PROBE_KINDS = {0: "LDG.128 gather through L1", 1: "TMA tile::gather4 into a shared-memory ring",
               2: "1-D bulk copy per weight into a shared-memory ring", 3: "random 4-byte loads val[perm[k]]",
               4: "random 4-byte stores dst[perm[k]]", 5: "sequential read of col + val"}


def run_gather_ceiling(args):
    import ctypes

    import torch

    from spmm_row_sorted_gb300 import build as snack_build

    lib = ctypes.CDLL(snack_build.build_probe())
    lib.probe_gather.restype = ctypes.c_int
    lib.probe_gather.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_int, ctypes.c_void_p]
    lib.probe_out_elems.restype = ctypes.c_int64
    lib.probe_out_elems.argtypes = [ctypes.c_int, ctypes.c_int]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lay, acts = make_workload(0)
    nnz = lay.nnz
    perm = np.lexsort((lay.row, lay.col)).astype(np.int32)  # storage index of each entry in column order
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    xt = torch.from_numpy(np.ascontiguousarray(acts.x.T)).to(dev).contiguous()  # [16384][32] feature-major
    col = torch.from_numpy(lay.col).to(dev)
    val = torch.from_numpy(lay.val).to(dev)
    pm = torch.from_numpy(perm).to(dev)
    dst = torch.empty(nnz, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(int(lib.probe_out_elems(1, 64 * sms)), device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, device=dev)
    flush_out = torch.empty((), device=dev)
    records = []
    sweeps = {0: (2, 4, 8, 16), 1: (1, 2, 4, 6), 2: (1, 2, 4, 6), 3: (4, 8, 16), 4: (4, 8, 16), 5: (4, 8, 16)}
    for kind, mults in sweeps.items():
        best = None
        for m in mults:
            grid = m * sms

            def launch():
                rc = lib.probe_gather(kind, xt.data_ptr(), IN_F, col.data_ptr(), val.data_ptr(), pm.data_ptr(), nnz,
                                      out.data_ptr(), dst.data_ptr(), err.data_ptr(), grid, stream.cuda_stream)
                if rc != 0:
                    raise RuntimeError(f"probe {kind} failed: {rc}")

            ts = []
            with torch.cuda.stream(stream):
                for _ in range(3):
                    launch()
                for _ in range(args.reps):
                    torch.sum(flush, dim=0, out=flush_out)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    launch()
                    e1.record(stream)
                    ts.append((e0, e1))
            stream.synchronize()
            us = statistics.median(a.elapsed_time(b) for a, b in ts) * 1e3
            if best is None or us < best[1]:
                best = (grid, us)
        if int(err.item()) != 0:
            raise RuntimeError(f"probe {kind} reported a wait that ran out: {int(err.item())}")
        grid, us = best
        rec = {"kind": kind, "route": PROBE_KINDS[kind], "grid": grid, "us": us, "weights_per_us": nnz / us}
        if kind <= 2:
            rec["gathered_GBs"] = nnz * 128 / (us * 1e-6) / 1e9
        elif kind <= 4:
            rec["sectors_per_us"] = nnz / us
        else:
            rec["GBs"] = nnz * 8 / (us * 1e-6) / 1e9
        records.append(rec)
        print(json.dumps(rec), flush=True)
    byts = alg_bytes(nnz, BATCH, OUT_F, IN_F)
    print(json.dumps({"what": "gather ceiling, 16384^2 Zipf layer, batch 32 fp32, cold L2 (2x L2 read between reps)",
                      "nnz": nnz, "fwd_alg_bytes": byts["fwd"], "records": records}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle time of the cpu_baseline sample")
    ap.add_argument("--cpu-seconds-total", type=float, default=120.0,
                    help="--impl reference: oracle time budget over all steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default=None,
                    help="per-workload sweep instead of the step bench: 'all' or a list like c1,c4")
    ap.add_argument("--configs-out", default=None, help="--configs: also write a markdown table here")
    ap.add_argument("--reps", type=int, default=200, help="--configs: timed reps per op")
    ap.add_argument("--no-fan-in-path", action="store_true",
                    help="--configs: time a library copy built without the constant-fan-in forward (for comparison)")
    ap.add_argument("--gather-ceiling", action="store_true",
                    help="time the gather-route probes on the 16384^2 layer at batch 32 and exit")
    ap.add_argument("--profile", action="store_true",
                    help="run warmup+steps untimed on one layer copy and exit (for ncu captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.gather_ceiling:
        return run_gather_ceiling(args)
    if args.configs:
        return run_configs(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
