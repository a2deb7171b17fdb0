#!/usr/bin/env python3
"""Benchmark: the six sparse x dense products on the 60,000 x 2,000 count matrix.

Workload ("main"): 60,000 x 2,000, about 6.02M nonzeros (row nnz NegBin(mean
100, r=2), Zipf(1.1) columns, values 1+Geometric(0.5)), dense width 16, fp32,
seeded synthetic data generated on the device.  One step = the six products
VCSR@B, VCSC@B, B@VCSR, B@VCSC, CSR@B and B@CSR, each once, with the matrix
handles already built (assembly is timed separately and reported).  Every
product is deterministic: the misaligned ones run as gathers over the exact
transpose each handle keeps; the two-phase and atomic variants are timed and
reported beside them.

Metric: effective HBM GB/s = algorithmic bytes / device time, where the
algorithmic bytes of a product are every array of the stored layout, the dense
operand read once and the output written once.  L2 is flushed before every
timed product: a 512 MiB buffer is written and then read back, so that L2 holds
only clean lines of that buffer (none of the product's data, and no dirty
lines whose write-back the product would otherwise pay for).  CUDA events
bracket each product on the launching stream; a product's time is the median
over the timed steps.

``--impl reference`` times the float64 CPU oracle on the same workload and
metric (the deliberately slow reference; host cores).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SpMM ms/product & effective HBM GB/s (% of 8 TB/s), 60k×2k 6M nnz w=16"
WORKLOAD = "main"
WIDTH = 16
PRODUCTS = [  # name, layout, major, direction
    ("VCSR@B", "vcs", "row", "A@B"),
    ("VCSC@B", "vcs", "col", "A@B"),
    ("B@VCSR", "vcs", "row", "B@A"),
    ("B@VCSC", "vcs", "col", "B@A"),
    ("CSR@B", "csr", "row", "A@B"),
    ("B@CSR", "csr", "row", "B@A"),
]
NOMINAL_HBM_GBS = 8000.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def count(self, t0: float) -> int:
        return sum(1 for t, _ in self.lines if t >= t0)

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float = 0.0, t1: float = float("inf")):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if not t0 <= t <= t1:
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def aggregate(ms_local: float, step_bytes: int, ws: int, device):
    """Whole-job figures of N replicas: the slowest rank's ms per step, and the
    bytes all ranks processed per second (GB/s) at that pace."""
    t_max = ms_local
    if ws > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t_max = float(t.item())
    return t_max, step_bytes * ws / (t_max * 1e-3) / 1e9


def source_digest() -> str:
    """Digest of the CUDA sources, to tell whether recorded ncu counters are current."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_dense_products_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_profile(key: str):
    """A value recorded from ncu in profiles/dram_traffic.txt (a product's DRAM bytes
    per launch, or "l1pct:<product>", its kernel's L1/shared throughput in % of peak),
    or None when the record is missing or the CUDA sources changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        rec = {}
        with open(path) as f:
            for ln in f:
                ln = ln.split("#", 1)[0].split()
                if len(ln) == 2:
                    rec[ln[0]] = ln[1]
        if rec.get("source_digest") != source_digest():
            return None
        return float(rec[key])
    except (OSError, KeyError, ValueError):
        return None


def recorded_traffic(product: str):
    """DRAM bytes (read + write) of one launch of `product`'s kernel, from the ncu
    record in profiles/dram_traffic.txt, or None when the kernels changed since."""
    v = recorded_profile(product)
    return None if v is None else int(v)


def algorithmic_bytes(A, n_x_rows: int, n_y_rows: int, w: int, es: int = 4) -> int:
    layout_bytes, _ = A.nbytes()
    return int(layout_bytes + n_x_rows * w * es + n_y_rows * w * es)


# ------------------------------------------------------------------ CPU oracle timing


def host_cores() -> int:
    """Cores this process may run on (the affinity mask), for the threaded oracle."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux hosts
        return os.cpu_count() or 1


def oracle_layouts(coo):
    """The oracle's own stored layouts of the workload, per (layout, major): ptr,
    idx, float64 values (per entry for CSR, per run for VCS), value_ptr or None,
    n_minor.  Built once, not timed."""
    import numpy as np
    import oracle

    r, c, v = coo.rows.numpy(), coo.cols.numpy(), coo.vals.numpy()
    out = {}
    for major in ("row", "col"):
        maj, mnr = (r, c) if major == "row" else (c, r)
        nm, nn = (coo.n_rows, coo.n_cols) if major == "row" else (coo.n_cols, coo.n_rows)
        mp, vals, vp, ind = oracle.vcs_build(nm, nn, maj, mnr, v)
        out[("vcs", major)] = (mp, ind, vals.astype(np.float64), vp, nn)
        if major == "row":
            p, i, vv = oracle.csr_build(nm, nn, maj, mnr, v)
            out[("csr", major)] = (p, i, vv.astype(np.float64), None, nn)
    return out


def run_oracle_sample(lays, Bab, Bba_rows, budget_s: float, threads: int):
    """Times the oracle's six products (threaded layout loops, slice frame) on
    `threads` host threads, repeated until `budget_s` seconds have passed.
    Bab is B of the A@B products (n_cols x w); Bba_rows is B^T of the B@A
    products (n_rows x w)."""
    import oracle

    t0 = time.perf_counter()
    reps = 0
    while True:
        for _, layout, major, direction in PRODUCTS:
            ptr, idx, vals, vp, n_minor = lays[(layout, major)]
            aligned = (direction == "A@B") == (major == "row")
            X = Bab if direction == "A@B" else Bba_rows
            oracle.spmm_slices(ptr, idx, vals, X, aligned, n_minor, vp, threads)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return reps, time.perf_counter() - t0


def cpu_baseline_leg(coo, Bab, Bba_rows, step_bytes: int, seconds: float):
    """The float64 oracle on the host cores: all cores of the affinity mask (the
    reported value) and one core beside it, each for about `seconds`."""
    lays = oracle_layouts(coo)
    cores = host_cores()
    r1, s1 = run_oracle_sample(lays, Bab, Bba_rows, seconds / 3, 1)
    rn, sn = run_oracle_sample(lays, Bab, Bba_rows, seconds, cores)
    return {"value": round(step_bytes * rn / sn / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"the six float64 oracle products over the oracle's own layouts of the full "
                      f"workload on {cores} threads (whole slices per thread for aligned "
                      f"products, private outputs merged in thread order for misaligned ones), "
                      f"{rn} pass(es) in {sn:.1f} s",
            "single_core": {"value": round(step_bytes * r1 / s1 / 1e9, 4), "unit": "GB/s",
                            "cores": 1, "sample": f"{r1} pass(es) in {s1:.1f} s"}}


def layout_bytes_host(coo):
    """Algorithmic bytes of the six products computed on the host (for the reference arm)."""
    import numpy as np

    r, c = coo.rows.numpy().astype(np.int64), coo.cols.numpy().astype(np.int64)
    v = coo.vals.numpy()
    nnz = r.size
    runs_r = np.unique(np.stack([r, v.view(np.uint32).astype(np.int64)]), axis=1).shape[1]
    runs_c = np.unique(np.stack([c, v.view(np.uint32).astype(np.int64)]), axis=1).shape[1]
    vcsr = 4 * (coo.n_rows + 1) + 4 * nnz + 8 * runs_r + 4
    vcsc = 4 * (coo.n_cols + 1) + 4 * nnz + 8 * runs_c + 4
    csr = 4 * (coo.n_rows + 1) + 8 * nnz
    w, es = WIDTH, 4
    ab = (coo.n_cols + coo.n_rows) * w * es
    ba = (coo.n_rows + coo.n_cols) * w * es
    return [vcsr + ab, vcsc + ab, vcsr + ba, vcsc + ba, csr + ab, csr + ba]


def reference_arm(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import numpy as np
    from sparse_dense_products_gb300 import workloads as W
    import oracle

    import torch

    oracle.build()
    # the same matrix and operands as the GPU arm (the generators' draws differ
    # between devices, so generate where that arm does when a GPU is present)
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    coo = W.make(WORKLOAD, seed=0, device=gen).to("cpu")
    Bab = W.dense(coo.n_cols, WIDTH, seed=1, device=gen).double().cpu().numpy()
    Bba_rows = W.dense(coo.n_rows, WIDTH, seed=2, device=gen).double().cpu().numpy()
    per = layout_bytes_host(coo)
    total_bytes = sum(per)
    lays = oracle_layouts(coo)
    cores = host_cores()
    # warm-up steps, then timed steps; one step = the six oracle products on all cores
    for _ in range(args.warmup):
        run_oracle_sample(lays, Bab, Bba_rows, 0.0, cores)
    reps, secs = 0, 0.0
    for _ in range(args.steps):
        r_, s_ = run_oracle_sample(lays, Bab, Bba_rows, 0.0, cores)
        reps += r_
        secs += s_
    gbs = total_bytes * reps / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / reps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "main: 60000x2000 count matrix, %d nnz, width 16, six products "
                               "(VCSR@B VCSC@B B@VCSR B@VCSC CSR@B B@CSR), float64 oracle" % coo.nnz,
                   "l2": "n/a (host)", "generated_on": gen},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "full workload, six float64 oracle products per step over the "
                                   "oracle's own layouts, on every core of the affinity mask"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU helpers


def bit_repeatability(torch, fn, reps: int, column_fn=None, columns=()):
    """Runs fn() `reps` times; counts the output values whose bits differ from the
    first result in at least one repeat, and (with column_fn) the values of each
    listed column computed alone whose bits differ from the same column of the
    batch.  fn returns a 2-D tensor whose second axis is the width."""
    first = fn().clone()
    bits = first.view(torch.int64 if first.dtype == torch.float64 else torch.int32)
    differ = torch.zeros_like(first, dtype=torch.bool)
    reps_differing = 0
    for _ in range(reps - 1):
        o = fn()
        d = o.view(bits.dtype) != bits
        differ |= d
        reps_differing += int(bool(d.any()))
    res = {"reps": reps, "values": int(first.numel()),
           "values_differing_in_a_repeat": int(differ.sum()),
           "repeats_differing": reps_differing}
    if column_fn is not None:
        alone = {}
        for c in columns:
            a = column_fn(c).reshape(-1)
            alone[str(c)] = int((a.view(bits.dtype) != bits[:, c].contiguous()).sum())
        res["column_alone_values_differing"] = alone
    torch.cuda.synchronize()
    return res


def time_product_set(vs, torch, coo, handles, specs, width: int, dtype, reps: int, timed,
                     layout_bytes, seed: int = 1):
    """Times each (name, layout, major, direction, variant) of `specs` at `width`
    on the workload `coo` (device tensors).  Returns {name/variant: {ms, GBs,
    frac_of_measured, frac_of_8TBs, bytes}}; a product's bytes are the stored
    layout it streams (the other-major layout for a misaligned product run over
    the transpose), B read once and out written once."""
    from sparse_dense_products_gb300 import workloads as W

    es = 8 if dtype == torch.float64 else 4
    peak, _ = _peaks()
    dev = coo.rows.device
    Bab = W.dense(coo.n_cols, width, seed=seed, device=dev, dtype=dtype)
    Bt = W.dense(coo.n_rows, width, seed=seed + 1, device=dev, dtype=dtype)
    out = {}
    for name, layout, major, direction, variant in specs:
        A = handles[(layout, major)]
        B = Bab if direction == "A@B" else Bt.t()
        o = vs.empty_out(A, width, direction, dtype=dtype)
        # the named product's own layout (the algorithmic bytes), whatever route runs it
        nb = int(layout_bytes[(layout, major)] + (coo.n_rows + coo.n_cols) * width * es)
        vs.spmm(A, B, direction, variant, out=o)
        ts = timed(lambda: vs.spmm(A, B, direction, variant, out=o), reps)
        ms = statistics.median(ts)
        out[f"{name}/{variant}"] = {"ms": round(ms, 5), "GBs": round(nb / ms / 1e6, 1),
                                    "frac_of_measured": round(nb / ms / 1e6 / peak, 4),
                                    "frac_of_8TBs": round(nb / ms / 1e6 / NOMINAL_HBM_GBS, 4),
                                    "bytes": nb}
    del Bab, Bt
    return out


def cusparse_times(torch, coo_dev, handles, width: int, dtype, reps: int, timed, ours: dict,
                   seed: int = 1, names=None):
    """torch's CSR matmul (cuSPARSE SpMM) on the index-sorted CSR (CSR@B) and on
    the CSR of the exact transpose (B@CSR), beside our deterministic times."""
    import warnings

    from sparse_dense_products_gb300 import workloads as W
    import sparse_dense_products_gb300 as vs

    warnings.filterwarnings("ignore", message="Sparse CSR tensor support is in beta")
    res = {}
    try:
        dev = coo_dev.rows.device
        A = handles[("csr", "row")]
        a = A.arrays()
        A_csr = torch.sparse_csr_tensor(a["ptr"], a["indices"], a["values"].to(dtype),
                                        (coo_dev.n_rows, coo_dev.n_cols))
        with vs.build_csr(coo_dev.cols, coo_dev.rows, coo_dev.vals, (coo_dev.n_cols, coo_dev.n_rows),
                          "row") as hT:
            t = hT.arrays()
        AT_csr = torch.sparse_csr_tensor(t["ptr"], t["indices"], t["values"].to(dtype),
                                         (coo_dev.n_cols, coo_dev.n_rows))
        Bab = W.dense(coo_dev.n_cols, width, seed=seed, device=dev, dtype=dtype)
        Bt = W.dense(coo_dev.n_rows, width, seed=seed + 1, device=dev, dtype=dtype)
        for name, Am, X in (("CSR@B", A_csr, Bab), ("B@CSR", AT_csr, Bt)):
            torch.mm(Am, X)
            ms = statistics.median(timed(lambda: torch.mm(Am, X), reps))
            entry = {"ms": round(ms, 5)}
            key = f"{(names or {}).get(name, name)}/deterministic"
            if key in ours:
                entry["ours"] = key
                entry["ours_over_cusparse_time"] = round(ours[key]["ms"] / ms, 3)
            res[name] = entry
        del A_csr, AT_csr, Bab, Bt
    except Exception as exc:  # reported, never fatal: a comparison, not the path
        res = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}
    return res


def build_handles(vs, coo, layouts, attach: bool = True):
    """Handles of the workload for each (layout, major), transposes attached."""
    hs = {}
    for layout, major in layouts:
        fn = vs.build_vcs if layout == "vcs" else vs.build_csr
        hs[(layout, major)] = fn(coo.rows, coo.cols, coo.vals, (coo.n_rows, coo.n_cols), major)
        if attach:
            hs[(layout, major)].attach_transpose()
    return hs


def layout_bytes_of(handles, coo):
    """Stored-layout bytes of each (layout, major) a product may stream; CSC from CSR."""
    lb = {k: h.nbytes()[0] for k, h in handles.items()}
    if ("csr", "row") in lb and ("csr", "col") not in lb:
        lb[("csr", "col")] = lb[("csr", "row")] - 4 * coo.n_rows + 4 * coo.n_cols
    return lb


def extra_workloads(vs, torch, dev, timed, reps: int, log):
    """The regridding-shaped, large and skewed workloads: ms, GB/s and fraction
    of the measured HBM copy per product, deterministic, atomic and two-phase variants,
    and cuSPARSE beside them."""
    from sparse_dense_products_gb300 import workloads as W

    res = {}
    peak, peak_kind = _peaks()
    # regridding-shaped: backprojection rows of 2-4 entries and their exact
    # transpose (the forward direction), float32 and float64, widths 1, 4, 32
    t0 = time.perf_counter()
    for dtype, tag in ((torch.float32, "f32"), (torch.float64, "f64")):
        coo = W.make("regrid", seed=0, device=dev, dtype=dtype)
        hs = build_handles(vs, coo, [("csr", "row")])
        lb = layout_bytes_of(hs, coo)
        for w in (1, 4, 32):
            specs = [("CSR@B", "csr", "row", "A@B", "deterministic"),
                     ("B@CSR", "csr", "row", "B@A", "deterministic"),
                     ("B@CSR", "csr", "row", "B@A", "atomic"),
                     ("B@CSR", "csr", "row", "B@A", "two_phase")]
            times = time_product_set(vs, torch, coo, hs, specs, w, dtype, reps, timed, lb)
            times["cusparse"] = cusparse_times(torch, coo, hs, w, dtype, reps, timed, times)
            res.setdefault("regrid", {})[f"{tag}/w{w}"] = times
        res["regrid"][f"{tag}/nnz"] = coo.nnz
        res["regrid"][f"{tag}/group_size"] = hs[("csr", "row")].info()["group_size"]
        for h in hs.values():
            h.destroy()
        del coo
    log(f"regrid done in {time.perf_counter() - t0:.1f} s")
    # large: 1,000,000 x 20,000, ~200M nonzeros, the four VCS directions, w 8 and 32
    t0 = time.perf_counter()
    coo = W.make("large", seed=0, device=dev)
    hs = build_handles(vs, coo, [("vcs", "row"), ("vcs", "col")])
    hs[("csr", "row")] = vs.build_csr(coo.rows, coo.cols, coo.vals, (coo.n_rows, coo.n_cols), "row")
    lb = layout_bytes_of(hs, coo)
    large = {"nnz": coo.nnz, "runs_vcsr": hs[("vcs", "row")].info()["n_runs"],
             "runs_vcsc": hs[("vcs", "col")].info()["n_runs"]}
    for w in (8, 32):
        specs = [("VCSR@B", "vcs", "row", "A@B", "deterministic"),
                 ("VCSC@B", "vcs", "col", "A@B", "deterministic"),
                 ("VCSC@B", "vcs", "col", "A@B", "atomic"),
                 ("VCSC@B", "vcs", "col", "A@B", "two_phase"),
                 ("B@VCSR", "vcs", "row", "B@A", "deterministic"),
                 ("B@VCSR", "vcs", "row", "B@A", "atomic"),
                 ("B@VCSR", "vcs", "row", "B@A", "two_phase"),
                 ("B@VCSC", "vcs", "col", "B@A", "deterministic")]
        times = time_product_set(vs, torch, coo, hs, specs, w, torch.float32, reps, timed, lb)
        # cuSPARSE on the index-sorted CSR of the same matrix, beside VCSR@B and B@VCSC
        times["cusparse"] = cusparse_times(torch, coo, hs, w, torch.float32, reps, timed, times,
                                           names={"CSR@B": "VCSR@B", "B@CSR": "B@VCSC"})
        large[f"w{w}"] = times
    det = {k: v for k, v in large["w32"].items() if k.endswith("/deterministic")}
    dom = max(det, key=lambda k: det[k]["ms"])
    name = dom.split("/")[0]
    traffic = recorded_profile("large:" + name)
    large["roofline"] = {"bound": "hbm", "kernel": dom + " w=32", "achieved": det[dom]["GBs"],
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": det[dom]["frac_of_measured"],
                         "traffic": None if traffic is None else int(traffic),
                         "traffic_note": "DRAM bytes per launch scaled from an ncu capture of "
                                         "a smaller matrix of the same recipe (profiles/)"}
    for h in hs.values():
        h.destroy()
    del coo
    res["large"] = large
    log(f"large done in {time.perf_counter() - t0:.1f} s")
    # skewed power-law CSR: 500,000 x 500,000, ~50M nonzeros, width 64
    t0 = time.perf_counter()
    coo = W.make("skewed", seed=0, device=dev)
    hs = build_handles(vs, coo, [("csr", "row")])
    lb = layout_bytes_of(hs, coo)
    specs = [("CSR@B", "csr", "row", "A@B", "deterministic"),
             ("B@CSR", "csr", "row", "B@A", "deterministic"),
             ("B@CSR", "csr", "row", "B@A", "atomic"),
             ("B@CSR", "csr", "row", "B@A", "two_phase")]
    sk = time_product_set(vs, torch, coo, hs, specs, 64, torch.float32, reps, timed, lb)
    sk["cusparse"] = cusparse_times(torch, coo, hs, 64, torch.float32, reps, timed, sk)
    sk["nnz"] = coo.nnz
    for h in hs.values():
        h.destroy()
    del coo
    res["skewed"] = sk
    log(f"skewed done in {time.perf_counter() - t0:.1f} s")
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ GPU arm


def gpu_arm(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl")

    from sparse_dense_products_gb300 import build as vs_build
    vs_build.build()
    import sparse_dense_products_gb300 as vs
    from sparse_dense_products_gb300 import workloads as W

    dev = torch.device("cuda", local)
    coo = W.make(WORKLOAD, seed=0, device=dev)
    n_rows, n_cols = coo.n_rows, coo.n_cols

    # ---- assembly (timed, reported; not part of the step).  Each layout is
    # built twice: the first build of a process also loads the assembly
    # kernels and grows the allocator's pools, so the second one is reported
    # (the first beside it).
    assembly = {}
    assembly_first = {}
    handles = {}
    for key, fn in ((("vcs", "row"), vs.build_vcs), (("vcs", "col"), vs.build_vcs),
                    (("csr", "row"), vs.build_csr)):
        name = f"{'V' if key[0] == 'vcs' else ''}CS{'R' if key[1] == 'row' else 'C'}"
        for rep in range(2):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            h = fn(coo.rows, coo.cols, coo.vals, (n_rows, n_cols), key[1])
            torch.cuda.synchronize()
            ms = round((time.perf_counter() - t0) * 1e3, 3)
            if rep == 0:
                assembly_first[name] = ms
                h.destroy()
            else:
                assembly[name] = ms
                handles[key] = h
    for h in handles.values():
        h.attach_transpose()

    Bab = W.dense(n_cols, WIDTH, seed=1, device=dev)          # A@B operand
    Bt = W.dense(n_rows, WIDTH, seed=2, device=dev)           # B@A operand, stored transposed
    outs = {}
    for name, layout, major, direction in PRODUCTS:
        outs[name] = vs.empty_out(handles[(layout, major)], WIDTH, direction)

    def run(name, layout, major, direction, variant="deterministic"):
        A = handles[(layout, major)]
        B = Bab if direction == "A@B" else Bt.t()
        return vs.spmm(A, B, direction, variant, out=outs[name])

    # algorithmic bytes: the layout arrays actually streamed (a misaligned product
    # with an attached transpose streams the other-major layout), B once, out once
    csr_bytes = handles[("csr", "row")].nbytes()[0]
    csc_bytes = csr_bytes - 4 * n_rows + 4 * n_cols
    layout_read = {("vcs", "row"): handles[("vcs", "row")].nbytes()[0],
                   ("vcs", "col"): handles[("vcs", "col")].nbytes()[0],
                   ("csr", "row"): csr_bytes, ("csr", "col"): csc_bytes}

    def product_bytes(layout, major, direction, variant="deterministic", streamed=False):
        """Algorithmic bytes of the named product: its own stored layout, B read
        once, out written once.  streamed=True counts instead the layout the
        kernel walks (the other-major transpose for a misaligned product run
        over it)."""
        aligned = (direction == "A@B") == (major == "row")
        if streamed and not aligned and variant in ("deterministic", "transposed"):
            major = "col" if major == "row" else "row"
        nx = n_cols if direction == "A@B" else n_rows
        ny = n_rows if direction == "A@B" else n_cols
        return int(layout_read[(layout, major)] + (nx + ny) * WIDTH * 4)

    nbytes = {name: product_bytes(layout, major, direction)
              for name, layout, major, direction in PRODUCTS}
    nbytes_streamed = {name: product_bytes(layout, major, direction, streamed=True)
                       for name, layout, major, direction in PRODUCTS}

    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_sum = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        """Write a buffer four times the size of L2, then read it back: the
        read evicts the dirty lines the write left, so L2 ends holding clean
        lines of this buffer only."""
        flush.fill_(1.0)
        flush_sum.copy_(flush.sum())
    stream = torch.cuda.current_stream(dev)

    def timed(fn, reps):
        """Device ms of fn() per rep, L2 flushed before each rep (events after the flush)."""
        evs = []
        for _ in range(reps):
            flush_l2()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    # ---- warm-up
    for _ in range(args.warmup):
        for p in PRODUCTS:
            run(*p)
    torch.cuda.synchronize()

    # ---- timed steps (barrier + synchronize on both sides)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = vs.kernel_launches()
    per = {name: [] for name, *_ in PRODUCTS}
    with Clocks(local) as clk:
        time.sleep(0.5)  # the sampler is running before the timed steps start
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            for p in PRODUCTS:
                per[p[0]].extend(timed(lambda p=p: run(*p), 1))
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        launches = vs.kernel_launches() - launches0
        # a short timed region sees few samples: keep the same load running,
        # untimed, until the sampler has seen at least 3 (at most 5 s more)
        t_end = time.perf_counter()
        while clk.count(wall0) < 3 and time.perf_counter() - t_end < 5.0:
            for p in PRODUCTS:
                timed(lambda p=p: run(*p), 1)
        clk_window = (wall0, time.perf_counter())
    if ws > 1:
        dist.barrier()
    ms_prod = {k: statistics.median(v) for k, v in per.items()}
    ms_mean = {k: statistics.mean(v) for k, v in per.items()}
    ms_step = sum(ms_prod.values())
    step_bytes = sum(nbytes.values())
    t_max, value = aggregate(ms_step, step_bytes, ws, dev)

    # ---- variants of the misaligned products (reported, not in the step)
    variants = {}
    for name, layout, major, direction in PRODUCTS:
        aligned = (direction == "A@B") == (major == "row")
        if aligned:
            continue
        for variant in ("two_phase", "atomic", "transposed"):
            run(name, layout, major, direction, variant)  # first call: scratch and launch setup
            ts = timed(lambda: run(name, layout, major, direction, variant), max(5, args.steps))
            ms = statistics.median(ts)
            vb = product_bytes(layout, major, direction, variant)
            variants[f"{name}/{variant}"] = {"ms": round(ms, 5), "GBs": round(vb / ms / 1e6, 1)}

    # ---- in-run cuSPARSE reference: torch's CSR matmul on the index-sorted CSR
    # (CSR@B), and on the CSR of the exact transpose for B@CSR (Y^T = A^T B^T)
    ours = {f"{k}/deterministic": {"ms": v} for k, v in ms_prod.items()}
    cusparse = cusparse_times(torch, coo, handles, WIDTH, torch.float32, max(5, args.steps),
                              timed, ours)

    # ---- bit repeatability: 100 repeats of the same product, and each of three
    # columns computed alone against the batch (cuSPARSE, then ours)
    determinism = {}
    try:
        import warnings
        warnings.filterwarnings("ignore", message="Sparse CSR tensor support is in beta")
        a = handles[("csr", "row")].arrays()
        A_csr = torch.sparse_csr_tensor(a["ptr"], a["indices"], a["values"], (n_rows, n_cols))
        cols = (0, WIDTH // 2, WIDTH - 1)
        determinism["cusparse CSR@B"] = bit_repeatability(
            torch, lambda: torch.mm(A_csr, Bab), 100,
            lambda c: torch.mm(A_csr, Bab[:, c:c + 1].contiguous()), cols)
        for name, layout, major, direction in PRODUCTS:
            A = handles[(layout, major)]
            if direction == "A@B":
                f = lambda A=A: vs.spmm(A, Bab, "A@B")
                fc = lambda c, A=A: vs.spmm(A, Bab[:, c:c + 1].contiguous(), "A@B")
            else:
                f = lambda A=A: vs.spmm(A, Bt.t(), "B@A").t()
                fc = lambda c, A=A: vs.spmm(A, Bt.t()[c:c + 1, :].t().contiguous().t(),
                                            "B@A").t()
            determinism[name] = bit_repeatability(torch, f, 100, fc, cols)
        del A_csr
    except Exception as exc:  # reported, never fatal
        determinism = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}

    # ---- the same products with L2 warm (no flush between reps): labelled
    # context, not the metric; near-equal times say the kernels are bound on
    # chip, not by HBM
    l2_warm = {}
    for p in PRODUCTS:
        for _ in range(3):
            run(*p)
        torch.cuda.synchronize()
        evs = []
        for _ in range(max(5, args.steps)):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run(*p)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        l2_warm[p[0]] = round(statistics.median(a.elapsed_time(b) for a, b in evs), 5)

    # ---- the gather floor of each product (vs_gather_floor: the same index
    # stream and operand rows, nothing else), the second roof made concrete
    floor_ms = {}
    for name, layout, major, direction in PRODUCTS:
        B = Bab if direction == "A@B" else Bt.t()
        A = handles[(layout, major)]
        ts = timed(lambda: vs.gather_floor(A, B, direction), max(5, args.steps))
        floor_ms[name] = round(statistics.median(ts), 5)

    # ---- host cost of one asynchronous vs_spmm call (enqueue only)
    torch.cuda.synchronize()
    n_calls = 200
    t0 = time.perf_counter()
    for q in range(n_calls):
        run(*PRODUCTS[q % len(PRODUCTS)])
    host_us = (time.perf_counter() - t0) / n_calls * 1e6
    torch.cuda.synchronize()

    # ---- e2e through vs_spmm_host with pinned host buffers
    Bab_h = Bab.cpu().pin_memory()
    Bt_h = Bt.cpu().pin_memory()
    outs_h = {name: vs.empty_out(handles[(l, m)], WIDTH, d, device="cpu", pin_memory=True)
              for name, l, m, d in PRODUCTS}
    h2d = d2h = 0
    for name, layout, major, direction in PRODUCTS:
        h2d += (n_cols if direction == "A@B" else n_rows) * WIDTH * 4
        d2h += (n_rows if direction == "A@B" else n_cols) * WIDTH * 4
    e2e_times = []
    for it in range(args.warmup + args.steps):
        tot = 0.0
        for name, layout, major, direction in PRODUCTS:
            flush_l2()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            vs.spmm_host(handles[(layout, major)], Bab_h if direction == "A@B" else Bt_h.t(),
                         direction, "deterministic", out=outs_h[name])
            tot += time.perf_counter() - t0
        if it >= args.warmup:
            e2e_times.append(tot)
    e2e_s = statistics.mean(e2e_times)
    e2e_value = step_bytes * ws / e2e_s / 1e9

    # ---- aggregate of the six products with no transpose attached: the aligned
    # gathers plus the two-phase scheme for the misaligned products
    nt_ms, nt_bytes = 0.0, 0
    for name, layout, major, direction in PRODUCTS:
        aligned = (direction == "A@B") == (major == "row")
        if aligned:
            nt_ms += ms_prod[name]
            nt_bytes += nbytes[name]
        else:
            nt_ms += variants[f"{name}/two_phase"]["ms"]
            nt_bytes += product_bytes(layout, major, direction, "two_phase")
    no_transpose = {"ms_per_step": round(nt_ms, 5), "GBs": round(nt_bytes / nt_ms / 1e6, 1),
                    "note": "aligned gathers + two-phase misaligned products (no transpose kept)"}

    # ---- the regridding-shaped, large and skewed workloads (reported beside
    # the headline; not part of its step)
    extra = None
    if not args.skip_extra and rank == 0:
        extra = extra_workloads(vs, torch, dev, timed, max(5, min(args.steps, 10)),
                                lambda m: print(m, file=sys.stderr, flush=True))

    # ---- roofline of the dominant kernel
    peak, peak_kind = _peaks()
    dom = max(ms_prod, key=ms_prod.get)
    achieved = nbytes[dom] / (ms_prod[dom] * 1e-3) / 1e9
    products = {k: {"ms": round(ms_prod[k], 5), "ms_mean": round(ms_mean[k], 5),
                    "GBs": round(nbytes[k] / ms_prod[k] / 1e6, 1),
                    "frac_of_8TBs": round(nbytes[k] / ms_prod[k] / 1e6 / NOMINAL_HBM_GBS, 4),
                    "frac_of_measured": round(nbytes[k] / ms_prod[k] / 1e6 / peak, 4),
                    "bytes": nbytes[k], "bytes_streamed": nbytes_streamed[k]} for k in ms_prod}
    traffic = recorded_traffic(dom)
    # the second roof: every stored entry brings a row of w values of X through
    # L1 or shared memory, at most 128 bytes per clock per SM (nominal width)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    clk_now = clk.summary(*clk_window)
    mhz = clk_now.get("sm_mhz") or clk_now.get("sm_max_mhz") or 2070.0
    onchip_bytes = coo.nnz * WIDTH * 4
    onchip_peak = 128.0 * n_sm * mhz * 1e6 / 1e9  # GB/s
    onchip_ach = onchip_bytes / (ms_prod[dom] * 1e-3) / 1e9
    onchip = {"bound": "l1/shared gather", "kernel": dom, "achieved": round(onchip_ach, 1),
              "peak": round(onchip_peak, 1), "peak_kind": "nominal: 128 B/clk/SM x SMs x sampled SM clock",
              "unit": "GB/s", "frac": round(onchip_ach / onchip_peak, 4),
              "bytes_per_launch": onchip_bytes,
              "gather_floor_ms": floor_ms[dom],
              "product_over_floor": round(ms_prod[dom] / floor_ms[dom], 3),
              # what ncu measured on the L1/shared data path of the same kernel (the
              # nominal peak above counts 128 useful bytes per clock; random 64-byte
              # rows cannot fill it), null once the kernels changed since the capture
              "ncu_l1_shared_throughput_pct": recorded_profile("l1pct:" + dom),
              # shared-memory wavefronts and warp instructions per stored entry of
              # the same kernel (ncu), under the same digest rule
              "ncu_shared_wavefronts_per_entry": recorded_profile("wavefronts_per_entry:" + dom),
              "ncu_instructions_per_entry": recorded_profile("instructions_per_entry:" + dom)}

    # ---- CPU baseline: the float64 oracle on host cores (rank 0, N=1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.skip_cpu:
        cpu = cpu_baseline_leg(coo.to("cpu"), Bab.double().cpu().numpy(),
                               Bt.double().cpu().numpy(), step_bytes, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "main: 60000x2000 count matrix, %d nnz, width 16, six products "
                               "(VCSR@B VCSC@B B@VCSR B@VCSC CSR@B B@CSR), deterministic; "
                               "misaligned ones over the attached exact transpose" % coo.nnz,
                   "l2": "flushed before every product (512 MiB written, then read back)",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "ms_per_product": round(t_max / len(PRODUCTS), 5),
        "frac_of_8TBs": round(value / ws / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "per": "one launch of the product's gather kernel (median of the timed reps)"},
        "roofline_onchip": onchip,
        "host_us_per_call": round(host_us, 2),
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4)},
        "clocks": dict(clk.summary(*clk_window),
                       window="the timed steps, extended by untimed steps to 3 samples"),
        "gpu_launches": launches,
        "products": products,
        "misaligned_variants": variants,
        "products_l2_warm_ms": l2_warm,
        "gather_floor_ms": floor_ms,
        "cusparse": cusparse,
        "bit_repeatability": determinism,
        "no_transpose": no_transpose,
        "extra_workloads": extra,
        "assembly_ms": assembly,
        "assembly_first_build_ms": assembly_first,
        "wall_s_timed_region": round(wall, 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    for h in handles.values():
        h.destroy()
    if ws > 1:
        dist.destroy_process_group()
    return 0


def profile_case(args):
    """One product of one workload, run --warmup + --steps times: the command
    the ncu captures under profiles/ run (no JSON metric line; a short summary
    on stdout).  --profile-rows draws a smaller matrix of the workload's recipe,
    so that a capture of a large configuration stays a few GB."""
    import torch

    from sparse_dense_products_gb300 import build as vs_build
    vs_build.build()
    import sparse_dense_products_gb300 as vs
    from sparse_dense_products_gb300 import workloads as W

    spec = {name: (layout, major, direction) for name, layout, major, direction in PRODUCTS}
    layout, major, direction = spec[args.profile_product]
    dev = torch.device("cuda", 0)
    coo = W.make(args.profile_workload, seed=0, device=dev, rows=args.profile_rows)
    fn = vs.build_vcs if layout == "vcs" else vs.build_csr
    A = fn(coo.rows, coo.cols, coo.vals, (coo.n_rows, coo.n_cols), major)
    variant = args.profile_variant
    if variant in ("deterministic", "transposed"):
        A.attach_transpose()
    w = args.profile_width
    B = W.dense(coo.n_cols, w, seed=1, device=dev) if direction == "A@B" else \
        W.dense(coo.n_rows, w, seed=2, device=dev).t()
    out = vs.empty_out(A, w, direction)
    del coo
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        vs.spmm(A, B, direction, variant, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        vs.spmm(A, B, direction, variant, out=out)
    e1.record()
    torch.cuda.synchronize()
    info = A.info()
    lb, _ = A.nbytes()
    n_x = info["n_cols"] if direction == "A@B" else info["n_rows"]
    n_y = info["n_rows"] if direction == "A@B" else info["n_cols"]
    print(json.dumps({"profile": args.profile_product, "variant": variant,
                      "workload": args.profile_workload,
                      "rows": info["n_rows"], "nnz": info["nnz"], "width": w,
                      "algorithmic_bytes": int(lb + (n_x + n_y) * w * 4),
                      "ms_per_product_warm": round(e0.elapsed_time(e1) / max(args.steps, 1), 5)}))
    A.destroy()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum seconds of oracle work for cpu_baseline")
    ap.add_argument("--skip-cpu", action="store_true", help="omit the cpu_baseline leg")
    ap.add_argument("--skip-extra", action="store_true",
                    help="omit the regridding-shaped, large and skewed workloads")
    ap.add_argument("--profile-product", choices=[p[0] for p in PRODUCTS],
                    help="run only this product (for ncu captures), no metric line")
    ap.add_argument("--profile-workload", default=WORKLOAD)
    ap.add_argument("--profile-rows", type=int, default=None)
    ap.add_argument("--profile-width", type=int, default=WIDTH)
    ap.add_argument("--profile-variant", default="deterministic",
                    choices=["deterministic", "two_phase", "atomic", "transposed"],
                    help="with --profile-product: the variant to run (a misaligned product's "
                         "deterministic variant runs over the attached transpose)")
    args = ap.parse_args()
    if args.profile_product:
        return profile_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
