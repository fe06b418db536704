"""Benchmark of the SpMM hot path: C = A * B with A in BCSR and in WCSR.

One step = one pass of the whole hot path over one batch of synthetic input:
  part 1  WCSR uniform   A 16384 x 16384 bf16, density 1 %, window 16,
                         B 16384 x 256 bf16, C fp32   (WCSR kernel + split reduce)
  part 2  BCSR weight    A 18944 x 3584 bf16, 64x64 blocks, 90 % zero,
                         B 3584 x 65536 bf16, C bf16   (BCSR kernel)
Metric: effective TFLOP/s = sum of 2*nnz*N over the parts / device time
("AsyncSparse", Section IV: throughput counts the original nonzeros only).
Roofline of a kernel: t_roof = max(2*stored*N / P_tensor, bytes_min / BW_hbm),
bytes_min = stored values + format indices + B once + C once.

Timing: W warm-up steps, then K timed steps; L2 is flushed (a 256 MiB write)
before every launch, outside the CUDA-event brackets; each launch is bracketed
by events on the stream it runs on.  Multi-GPU (torchrun): each rank runs its
own copy of the step on its own GPU (independent problems, weak scaling, no
collective on the data path); the reported time is the max over ranks.

--impl reference times the CPU oracle (fp64, OpenMP) on the host cores on a
bounded sample of the same workload per step.
--sweep prints one line per benchmark configuration (instead of the step line);
--sweep bcsr_weight:8192 runs one configuration at another dense width N.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import spmm_workloads as W  # noqa: E402

METRIC = "SpMM effective TFLOP/s (2·nnz·N/t) and % of roofline, BCSR and WCSR"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20

# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture,
# valid only for the kernel source it was taken on (sha256 of the file).
MEASURED_TRAFFIC = {
    # bcsr_weight: 114.9 MB read + 261.7 MB written at N = 8192; B and C scale
    # with N, A (13.6 MB) does not: 13.6 MB + 8 x 363.1 MB at N = 65536
    "bcsr_kernel.cu": {"src_sha": "158009bf8c3f0064", "bytes_per_launch": 2.918e9},
    # wcsr_uniform at its benchmark size: 100.1 MB read + 9.2 MB written (part
    # of C still in L2 when the kernel ends)
    "wcsr_kernel.cu": {"src_sha": "c78a22c320346a38", "bytes_per_launch": 1.093e8},
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def src_sha(name):
    """sha256 of a kernel source with // comments and blank lines removed, so
    that a recorded traffic figure survives comment edits but not code edits."""
    p = os.path.join(ROOT, "sparse_dense_matrix_bcsr_gb300", "csrc", name)
    code = []
    for line in open(p, encoding="utf-8"):
        line = line.split("//", 1)[0].rstrip()
        if line:
            code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


# ---------------------------------------------------------------- workloads
STEP_PARTS = (("wcsr_uniform", W.wcsr_uniform), ("bcsr_weight", W.bcsr_weight))


def part_model(w, info):
    """Algorithmic FLOPs and bytes of one launch on workload w."""
    out_sz = 4 if w.out_dtype == "f32" else 2
    eff_flops = 2.0 * w.nnz * w.n
    stored_flops = 2.0 * info["stored"] * w.n
    bytes_min = 2.0 * info["stored"] + info["idx_bytes"] + 2.0 * w.k * w.n + out_sz * w.m * w.n
    return eff_flops, stored_flops, bytes_min


def gather_model(w, info):
    """WCSR's secondary roof: bytes of B rows gathered from L2 by one launch,
    one row of N 16-bit values per packed (padded) column.  No HBM roofline
    counts them; measure_l2_read_gbs gives the rate they are set against."""
    return 2.0 * info["n_units"] * w.n if w.fmt == "wcsr" else 0.0


_L2_RATES = {}


def measure_l2_read_gbs(S, stream, dev, nbytes):
    """L2-to-SM read rate of this GPU for a footprint of nbytes (the size of
    the B that a WCSR launch gathers from): spmm_probe_l2_read streams a buffer
    of that size (resident in L2 after two untimed passes) 20 times with
    16-byte loads that bypass L1 from every SM; best of three, CUDA events on
    the stream (at least 4 GiB read per timed launch).  Each footprint gets
    its own figure, since the rate depends on it."""
    import torch
    nbytes = max(1 << 20, (int(nbytes) + 15) // 16 * 16)
    if nbytes in _L2_RATES:
        return _L2_RATES[nbytes]
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device=f"cuda:{dev}")
    sink = torch.zeros(4, dtype=torch.int32, device=f"cuda:{dev}")
    sptr = stream.cuda_stream
    passes = max(20, (4 << 30) // nbytes)  # at least 4 GiB per timed launch: launch cost negligible
    best = 0.0
    for _ in range(3):
        S.spmm_probe_l2_read(buf.data_ptr(), nbytes, 2, sink.data_ptr(), sptr)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        S.spmm_probe_l2_read(buf.data_ptr(), nbytes, passes, sink.data_ptr(), sptr)
        e1.record(stream)
        stream.synchronize()
        best = max(best, nbytes * passes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    _L2_RATES[nbytes] = round(best, 1)
    return _L2_RATES[nbytes]


L2_PEAK_SOURCE = ("measured here: spmm_probe_l2_read, 16-byte L1-bypassing loads of an L2-resident "
                  "buffer the size of B from every SM, >= 4 GiB per timed launch, best of 3")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        load = [x for x in sm if mx and x > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- multi-rank host logic
def host_link_rates(stream, dev, nbytes=1 << 30):
    """The host link's own copy rates, the ceiling of the end-to-end figure:
    1 GiB copies each way between pinned host memory and the device on the
    benchmark's stream, after one untimed copy, timed with CUDA events; the
    best of three per direction."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=f"cuda:{dev}")
    out = {}
    for name, dst, src in (("h2d_gbs", d, h), ("d2h_gbs", h, d)):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
        best = 0.0
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                dst.copy_(src, non_blocking=True)
                e1.record(stream)
            stream.synchronize()
            best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        out[name] = round(best, 1)
    return out


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values of x (all-reduce MAX over the default
    process group; a GPU tensor under NCCL, a host tensor under gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as tdist
    dev = f"cuda:{torch.cuda.current_device()}" if tdist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step_per_rank: float, steps: int, world: int, max_ms: float) -> float:
    """Throughput of the whole job: every rank's work over the slowest rank's time."""
    return flops_per_step_per_rank * steps * world / (max_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world):
    import torch
    import sparse_dense_matrix_bcsr_gb300 as S
    from sparse_dense_matrix_bcsr_gb300 import build as lib_build

    lib_build.build()
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    sptr = stream.cuda_stream
    peaks = load_peaks()

    parts = []
    for name, fn in STEP_PARTS:
        w = fn()
        create = S.spmm_bcsr_create if w.fmt == "bcsr" else S.spmm_wcsr_create
        h = create(w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.b_row, w.b_col)
        info = S.spmm_format_info(h)
        B = w.B()
        dB = torch.from_numpy(B.view(np.int16)).to(f"cuda:{dev}").view(
            torch.bfloat16 if w.dtype == "bf16" else torch.float16)
        dC = torch.empty((w.m, w.n), dtype=torch.float32 if w.out_dtype == "f32" else torch.bfloat16,
                         device=f"cuda:{dev}")
        eff, stored_fl, bytes_min = part_model(w, info)
        parts.append(dict(name=name, w=w, h=h, info=info, B=B, dB=dB, dC=dC, eff=eff, stored_flops=stored_fl,
                          bytes_min=bytes_min, launches=2 if w.fmt == "wcsr" else 1,
                          kernel="bcsr_kernel.cu" if w.fmt == "bcsr" else "wcsr_kernel.cu"))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=f"cuda:{dev}")
    for p in parts:
        p["l2_gbs"] = measure_l2_read_gbs(S, stream, dev, p["B"].nbytes) if p["w"].fmt == "wcsr" else None

    def one_step(times):
        for p in parts:
            with torch.cuda.stream(stream):
                flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            S.spmm_run(p["h"], p["dB"].data_ptr(), p["dC"].data_ptr(), p["w"].n, sptr)
            e1.record(stream)
            times.setdefault(p["name"], []).append((e0, e1))

    clk = ClockSampler(dev).__enter__()
    t_first = time.perf_counter()
    while not clk.lines and time.perf_counter() - t_first < 2.0:
        time.sleep(0.05)  # let nvidia-smi produce its first sample
    for _ in range(args.warmup):
        one_step({})
    stream.synchronize()
    for p in parts:
        st = S.spmm_check(p["h"], sptr)
        if st != S.SPMM_OK:
            raise RuntimeError(f"{p['name']}: device status {st}")

    dist = world > 1
    if dist:
        import torch.distributed as tdist
        tdist.barrier()
    torch.cuda.synchronize()
    times = {}
    with clk:
        t_wall0 = time.perf_counter()
        for _ in range(args.steps):
            one_step(times)
        stream.synchronize()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    if dist:
        tdist.barrier()
    for p in parts:
        st = S.spmm_check(p["h"], sptr)
        if st != S.SPMM_OK:
            raise RuntimeError(f"{p['name']}: device status {st}")

    per_part = {}
    for p in parts:
        ms = [a.elapsed_time(b) for a, b in times[p["name"]]]
        per_part[p["name"]] = ms
    step_ms = [sum(per_part[p["name"]][i] for p in parts) for i in range(args.steps)]
    total_ms = max_over_ranks(sum(step_ms), world)
    eff_per_step = sum(p["eff"] for p in parts)
    value = whole_job_tflops(eff_per_step, args.steps, world, total_ms)

    # roofline of each part; the dominant kernel (largest time share) is reported
    breakdown = []
    for p in parts:
        ms = per_part[p["name"]]
        t = statistics.mean(ms) * 1e-3
        t_tc = p["stored_flops"] / (peaks["bf16_tflops"] * 1e12)
        t_hbm = p["bytes_min"] / (peaks["hbm_gbs"] * 1e9)
        bound = "hbm" if t_hbm >= t_tc else "tensor"
        if bound == "hbm":
            achieved, peak, unit = p["bytes_min"] / t / 1e9, peaks["hbm_gbs"], "GB/s"
        else:
            achieved, peak, unit = p["stored_flops"] / t / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        tr = MEASURED_TRAFFIC.get(p["kernel"])
        traffic = tr["bytes_per_launch"] if tr and tr.get("src_sha") == src_sha(p["kernel"]) else None
        breakdown.append({
            "part": p["name"], "workload": p["w"].describe(), "kernel": p["kernel"],
            "ms_mean": round(statistics.mean(ms), 5), "ms_median": round(statistics.median(ms), 5),
            "ms_min": round(min(ms), 5), "eff_tflops": round(p["eff"] / t / 1e12, 3),
            "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "t_roof_us": round(max(t_tc, t_hbm) * 1e6, 2), "t_tensor_us": round(t_tc * 1e6, 2),
                         "t_hbm_us": round(t_hbm * 1e6, 2), "bytes_min": int(p["bytes_min"]),
                         "stored_flops": p["stored_flops"], "peak_source": peaks["source"] + " (burst)"},
            "format": {k: p["info"][k] for k in ("nnz", "stored", "padding", "n_units", "n_tasks",
                                                 "n_split_windows")},
        })
        gb = gather_model(p["w"], p["info"])
        if gb:
            breakdown[-1]["gather"] = {"bytes": int(gb), "achieved": round(gb / t / 1e9, 1), "unit": "GB/s",
                                       "peak": p["l2_gbs"], "frac": round(gb / t / 1e9 / p["l2_gbs"], 4),
                                       "peak_source": L2_PEAK_SOURCE,
                                       "note": "B rows gathered from L2 (one row of N values per packed column)"}
    dom = max(breakdown, key=lambda b: b["ms_mean"])

    # end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        hosts = []
        for p in parts:
            hb = torch.from_numpy(p["B"].view(np.int16)).pin_memory()
            hc = torch.empty(p["dC"].shape, dtype=p["dC"].dtype).pin_memory()
            hosts.append((hb, hc))
        for _ in range(max(1, min(args.warmup, 2))):
            for p, (hb, hc) in zip(parts, hosts):
                S.spmm_run_host_ptr(p["h"], hb.data_ptr(), hc.data_ptr(), p["w"].n, sptr)
        # Each step is timed on its own (every call ends with a synchronize)
        # and the median step gives the figure: the host side of this box
        # shows occasional slow steps (whole runs 25-54 TFLOP/s apart with
        # the link's copy rate unchanged).
        e2e_steps = max(1, min(args.steps, 9))
        if dist:
            tdist.barrier()
        step_s = []
        for _ in range(e2e_steps):
            t0 = time.perf_counter()
            for p, (hb, hc) in zip(parts, hosts):
                S.spmm_run_host_ptr(p["h"], hb.data_ptr(), hc.data_ptr(), p["w"].n, sptr)
            step_s.append(time.perf_counter() - t0)
        t_e2e = max_over_ranks(statistics.median(step_s), world)
        e2e = {"value": round(whole_job_tflops(eff_per_step, 1, world, t_e2e * 1e3), 4), "unit": UNIT,
               "ms_per_step_median": round(t_e2e * 1e3, 3),
               "ms_per_step_all": [round(x * 1e3, 2) for x in step_s],
               "h2d_bytes_per_step": int(sum(hb.numel() * 2 for hb, _ in hosts)),
               "d2h_bytes_per_step": int(sum(hc.numel() * hc.element_size() for _, hc in hosts)),
               "steps": e2e_steps, "host_link": host_link_rates(stream, dev)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(parts_workloads=[p["w"] for p in parts], budget_s=args.cpu_seconds)

    for p in parts:
        S.spmm_destroy(p["h"])

    clocks = clk.summary()
    gpu_launches = args.steps * sum(p["launches"] for p in parts)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate",
        "data": "synthetic (seeded; shapes and distributions of the benchmark configurations)",
        "config": {"workload": " + ".join(p["w"].describe() for p in parts),
                   "parts": [p["name"] for p in parts], "l2": "flushed before every launch (256 MiB write)",
                   "parallelism": f"replicated problem per GPU x{world}"},
        "roofline": {k: dom["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")},
        "roofline_kernel": dom["kernel"],
        "parts": breakdown,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches, "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    return line


# ---------------------------------------------------------------- oracle arm
def cpu_baseline_sample(parts_workloads, budget_s=10.0, offset=0):
    """Time the oracle's fp64 SpMM on a row sample of each part, about
    budget_s seconds of CPU work in total (whole matrices are repeated when
    they take less); returns the cpu_baseline dict."""
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    flops = 0.0
    t = 0.0
    desc = []
    want = budget_s / len(parts_workloads)
    for w in parts_workloads:
        B = w.B()
        per_row = 2.0 * w.nnz / max(w.m, 1) * w.n
        rows = max(1, min(w.m, int(5e7 / max(per_row, 1))))
        while True:
            r0 = (offset * rows) % max(w.m - rows + 1, 1)
            dt = _time_rows(oracle, w, B, r0, rows, threads)
            if rows >= w.m or dt >= 0.25 * want:
                break
            rows = min(w.m, rows * 4)
        reps = 1
        if dt < want:
            if rows < w.m:
                rows = min(w.m, int(rows * want / max(dt, 1e-6)))
                r0 = (offset * rows) % max(w.m - rows + 1, 1)
            else:
                reps = max(1, int(want / max(dt, 1e-6)))
        tt = 0.0
        for _ in range(reps):
            tt += _time_rows(oracle, w, B, r0, rows, threads)
        fl = 2.0 * float(w.row_ptr[r0 + rows] - w.row_ptr[r0]) * w.n * reps
        flops += fl
        t += tt
        desc.append(f"{w.name}: rows {r0}..{r0 + rows - 1} of {w.m} x{reps} "
                    f"({int(w.row_ptr[r0 + rows] - w.row_ptr[r0])} nnz, N={w.n})")
    return {"value": round(flops / t / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "; ".join(desc), "seconds": round(t, 3)}


def _time_rows(oracle, w, B, r0, rows, threads):
    rp = w.row_ptr[r0:r0 + rows + 1] - w.row_ptr[r0]
    ci = w.col_idx[w.row_ptr[r0]:w.row_ptr[r0 + rows]]
    vv = w.vals[w.row_ptr[r0]:w.row_ptr[r0 + rows]]
    t0 = time.perf_counter()
    oracle.spmm_csr(rows, w.k, rp, ci, vv, oracle.BF16 if w.dtype == "bf16" else oracle.F16, B,
                    threads=threads, with_abs=False)
    return time.perf_counter() - t0


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    ws = [fn() for _, fn in STEP_PARTS]
    per_step_s = max(1.0, min(6.0, 150.0 / max(args.steps + args.warmup, 1)))
    for i in range(args.warmup):
        cpu_baseline_sample(ws, budget_s=per_step_s, offset=i)
    fl = 0.0
    tt = 0.0
    last = None
    for i in range(args.steps):
        r = cpu_baseline_sample(ws, budget_s=per_step_s, offset=args.warmup + i)
        fl += r["value"] * 1e12 * r["seconds"]
        tt += r["seconds"]
        last = r
    value = fl / tt / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp64 (oracle)",
        "data": "synthetic (seeded), row samples per step",
        "config": {"workload": " + ".join(w.describe() for w in ws), "parts": [n for n, _ in STEP_PARTS],
                   "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                         "sample": f"per step ~{per_step_s:.1f} s of rows, e.g. " + last["sample"]},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ---------------------------------------------------------------- sweep
SWEEP_SUFFIXES = ("_split", "_dyn", "_h64", "_rcm")  # removed from the end in this order


def parse_config_entry(e):
    """A --sweep entry -> (base configuration, variant flags, sweep point).
    The variant suffixes (see SWEEP_SUFFIXES) may follow a name in the order
    _rcm, _h64, _dyn, _split; the flags dict holds those present (without the
    underscore).  A single sweep point such as bcsr_sweep_95_N256 or
    wcsr_sweep_0.1_N8 gives point = (format, level, N), else point is None."""
    flags = {}
    base = e
    for suf in SWEEP_SUFFIXES:
        if base.endswith(suf):
            base = base[:-len(suf)]
            flags[suf[1:]] = True
    parts = base.split("_")
    point = None
    if len(parts) == 4 and parts[0] in ("bcsr", "wcsr") and parts[1] == "sweep" and parts[3].startswith("N"):
        point = (parts[0], float(parts[2]), int(parts[3][1:]))
    return base, flags, point


def run_sweep(args):
    """One JSON line per benchmark configuration on this GPU (ours only)."""
    import torch
    import sparse_dense_matrix_bcsr_gb300 as S
    from sparse_dense_matrix_bcsr_gb300 import build as lib_build
    lib_build.build()
    peaks = load_peaks()
    stream = torch.cuda.Stream()
    sptr = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    cfgs = []
    # entries: a configuration name, optionally ":N" to change the dense width
    # of a single-workload configuration (e.g. a smaller case for a profiler)
    sel = {}
    for e in (args.sweep.split(",") if args.sweep not in ("all", "") else []):
        name, _, n = e.partition(":")
        sel[name] = int(n) if n else None
    builders = [("bcsr_tiny", lambda n: [W.bcsr_tiny()]),
                ("wcsr_uniform", lambda n: [W.wcsr_uniform(n=n) if n else W.wcsr_uniform()]),
                ("wcsr_irregular", lambda n: [W.wcsr_irregular(n=n) if n else W.wcsr_irregular()]),
                ("bcsr_weight", lambda n: [W.bcsr_weight(n=n) if n else W.bcsr_weight()]),
                ("bcsr_sweep", lambda n: [W.bcsr_sweep(s, k) for s in W.BCSR_SWEEP_SPARSITY for k in W.SWEEP_N]),
                ("wcsr_sweep", lambda n: [W.wcsr_sweep(d, k) for d in W.WCSR_SWEEP_DENSITY for k in W.SWEEP_N])]
    # an entry may end in _rcm (rows in reverse Cuthill-McKee order before the
    # format is built; C comes out in that row order), _h64 (the WCSR matrix
    # in 64-row windows with column padding 8, the paper's WCSR geometry)
    # and/or _dyn (the WCSR dynamic schedule) or _split (the BCSR split
    # schedule), in that order;
    # bcsr_sweep_95_N256 or wcsr_sweep_0.1_N8 name one sweep point
    def variant(ws, h64, dyn, rcm=False, split=False):
        for w in ws:
            if split:
                w.name += "_split"
                w.meta["schedule"] = S.SPMM_SCHEDULE_SPLIT
                w.meta["desc"] = w.describe() + " (split schedule)"
            if rcm:
                from sparse_dense_matrix_bcsr_gb300 import reorder
                t0 = time.perf_counter()
                perm = reorder.rcm_row_order(w.m, w.k, w.row_ptr, w.col_idx)
                w.row_ptr, w.col_idx, w.vals = reorder.permute_rows(w.row_ptr, w.col_idx, w.vals, perm)
                w.name += "_rcm"
                w.meta["desc"] = w.describe() + f" (RCM rows, {time.perf_counter() - t0:.1f} s on the host)"
            if h64:
                w.b_row, w.b_col = 64, 8
                w.name += "_h64"
                w.meta["desc"] = w.describe().replace(" h16 ", " h64 pad8 ")
            if dyn:
                w.name += "_dyn"
                w.meta["schedule"] = S.SPMM_SCHEDULE_DYNAMIC
                w.meta["desc"] = w.describe() + " (dynamic schedule)"
        return ws
    named = dict(builders)
    if not sel:
        cfgs = [(name, lambda b=b: b(None)) for name, b in builders]
    for e, n in sel.items():
        if e == "linear_weight":
            continue
        base, flags, point = parse_config_entry(e)
        h64, dyn, rcm, split = (flags.get(k, False) for k in ("h64", "dyn", "rcm", "split"))
        if base in named:
            fn = (lambda b=named[base], n=n: b(n))
        elif point is not None:
            fmt, lvl, nn = point
            fn = (lambda lvl=lvl, nn=nn: [W.bcsr_sweep(int(lvl), nn)]) if fmt == "bcsr" else \
                (lambda lvl=lvl, nn=nn: [W.wcsr_sweep(lvl, nn)])
        else:
            raise SystemExit(f"unknown configuration {e!r}")
        cfgs.append((e, lambda fn=fn, h64=h64, dyn=dyn, rcm=rcm, split=split: variant(fn(), h64, dyn, rcm, split)))
    if "linear_weight" in sel:
        run_linear_sweep(args, peaks, stream, flush)
    for name, b in cfgs:
        cache = {}
        for w in b():
            key = (w.fmt, w.m, w.k, w.nnz, int(w.row_ptr[w.m // 2]), w.b_row, w.meta.get("schedule"))
            if key not in cache:
                for hh in cache.values():
                    S.spmm_destroy(hh)
                cache.clear()
                create = S.spmm_bcsr_create if w.fmt == "bcsr" else S.spmm_wcsr_create
                cache[key] = create(w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype, w.b_row, w.b_col)
                if w.meta.get("schedule") is not None:
                    S.spmm_set_schedule(cache[key], w.meta["schedule"])
            h = cache[key]
            info = S.spmm_format_info(h)
            dB = torch.from_numpy(w.B().view(np.int16)).cuda().view(torch.bfloat16 if w.dtype == "bf16" else torch.float16)
            dC = torch.empty((w.m, w.n), dtype=torch.float32 if w.out_dtype == "f32" else torch.bfloat16, device="cuda")
            ms_cold, ms_warm = [], []
            for i in range(args.warmup + args.steps):
                with torch.cuda.stream(stream):
                    flush.fill_(1.0)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                S.spmm_run(h, dB.data_ptr(), dC.data_ptr(), w.n, sptr)
                e1.record(stream)
                e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e2.record(stream)
                S.spmm_run(h, dB.data_ptr(), dC.data_ptr(), w.n, sptr)
                e3.record(stream)
                if i >= args.warmup:
                    ms_cold.append((e0, e1))
                    ms_warm.append((e2, e3))
            stream.synchronize()
            assert S.spmm_check(h, sptr) == S.SPMM_OK
            cold = statistics.median(a.elapsed_time(b) for a, b in ms_cold)
            warm = statistics.median(a.elapsed_time(b) for a, b in ms_warm)
            eff, stored_fl, bytes_min = part_model(w, info)
            l2_gbs = measure_l2_read_gbs(S, stream, torch.cuda.current_device(), 2 * w.k * w.n) \
                if w.fmt == "wcsr" else None
            t = cold * 1e-3
            t_tc = stored_fl / (peaks["bf16_tflops"] * 1e12)
            t_hbm = bytes_min / (peaks["hbm_gbs"] * 1e9)
            print(json.dumps({
                "config": w.name, "workload": w.describe(), "fmt": w.fmt, "N": w.n, "nnz": w.nnz,
                "stored": info["stored"], "fill": round(w.nnz / max(info["stored"], 1), 4),
                "ms_cold_median": round(cold, 5), "ms_warm_median": round(warm, 5),
                "eff_tflops": round(eff / t / 1e12, 3), "eff_tflops_warm": round(eff / (warm * 1e-3) / 1e12, 3),
                "roofline_frac": round(max(t_tc, t_hbm) / t, 4), "bound": "hbm" if t_hbm >= t_tc else "tensor",
                "t_roof_us": round(max(t_tc, t_hbm) * 1e6, 2), "n_tasks": info["n_tasks"],
                "n_split_windows": info["n_split_windows"],
                "gather_gbs": round(gather_model(w, info) / t / 1e9, 1) if w.fmt == "wcsr" else None,
                "gather_frac": round(gather_model(w, info) / t / 1e9 / l2_gbs, 4) if w.fmt == "wcsr" else None,
                "l2_read_gbs": l2_gbs}),
                flush=True)
        for hh in cache.values():
            S.spmm_destroy(hh)


def run_linear_sweep(args, peaks, stream, flush):
    """The BCSR product in the layout of a linear layer (Y = X * A^T, X the
    64K-token activations, A the 90 %-block-sparse gate projection), beside
    dense torch.mm on the same box (cuBLAS; context, as the pages' Table III
    sets their kernel beside torch.mm)."""
    import torch
    import sparse_dense_matrix_bcsr_gb300 as S
    w = W.bcsr_weight()
    sptr = stream.cuda_stream
    h = S.spmm_bcsr_create(w.m, w.k, w.row_ptr, w.col_idx, w.vals, w.dtype, w.out_dtype)
    info = S.spmm_format_info(h)
    X = torch.from_numpy(np.ascontiguousarray(w.B().T).view(np.int16)).cuda().view(torch.bfloat16)
    Y = torch.empty((w.n, w.m), dtype=torch.bfloat16, device="cuda")

    def timed(fn):
        ms = []
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= args.warmup:
                ms.append((e0, e1))
        stream.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ms)

    t_ours = timed(lambda: S.spmm_run_linear(h, X.data_ptr(), Y.data_ptr(), w.n, sptr))
    assert S.spmm_check(h, sptr) == S.SPMM_OK
    dense = np.zeros((w.m, w.k), np.uint16)
    rows = np.repeat(np.arange(w.m), np.diff(w.row_ptr))
    dense[rows, w.col_idx] = w.vals
    Wd = torch.from_numpy(dense.view(np.int16)).cuda().view(torch.bfloat16)
    Yd = torch.empty_like(Y)
    with torch.cuda.stream(stream):
        t_mm = timed(lambda: torch.mm(X, Wd.t(), out=Yd))
    S.spmm_destroy(h)
    eff, stored_fl, bytes_min = part_model(w, info)
    t = t_ours * 1e-3
    t_tc = stored_fl / (peaks["bf16_tflops"] * 1e12)
    t_hbm = bytes_min / (peaks["hbm_gbs"] * 1e9)
    print(json.dumps({
        "config": "linear_weight", "workload": "Y = X * A^T, " + w.describe() + " (X: 65536 x 3584 rows)",
        "fmt": "bcsr-linear", "N": w.n, "nnz": w.nnz, "ms_cold_median": round(t_ours, 5),
        "eff_tflops": round(eff / t / 1e12, 3), "roofline_frac": round(max(t_tc, t_hbm) / t, 4),
        "bound": "hbm" if t_hbm >= t_tc else "tensor", "t_roof_us": round(max(t_tc, t_hbm) * 1e6, 2),
        "torch_mm_dense_ms": round(t_mm, 5), "speedup_vs_torch_mm": round(t_mm / t_ours, 3)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", default=None, help="comma list of configs, or 'all'")
    args = ap.parse_args()
    if args.warmup < 3 and args.sweep is None and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: run N > 1 GPUs under "
                         "python -m torch.distributed.run --nproc-per-node N")
    if args.sweep is not None:
        run_sweep(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
