"""Benchmark of the fused pattern out = alpha * X^T (v * (X y)) + beta * z on GB300.

Default workload: dense fp32 X 16,000,000 x 32 row-major, X, y, z ~ N(0, 1),
v ~ U[0.1, 2], alpha = 2, beta = -1 (the full pattern with every step of the path).
A step is one fused call over that input. Inputs (2.1 GB) exceed L2 (129 MB), so no
flush is needed between steps.

Prints one JSON line. ``value`` is effective GB/s: the algorithmic bytes of a call
(X once, y, v, z, out) over its device time, inputs resident in HBM. ``e2e`` is the
same metric with the host-to-device copy of the inputs (pinned memory) and the
device-to-host copy of out inside the timed region. ``roofline`` relates the fused
kernel to the measured HBM copy bandwidth; ``cpu_baseline`` is the C oracle timed on
this host's cores; ``unfused_library`` is the three-call cuBLAS sequence
(gemv, scale, transposed gemv) on the same GPU.

The default run also measures every other configuration of the workload list (dense f64
1000 x 64; the three variants of the tall fp32 X; dense f64 20,000 x 20,000; CSR f64
uniform; CSR f32 power-law) in the same process and nests their figures in the same
line under ``configs``: back-to-back microseconds per call, isolated calls after an L2
flush (p10/p50/p90; hot-L2 too for the small case), GB/s against the measured HBM copy
bandwidth, the fp64 ALU roof where it binds, e2e, the unfused library sequence and the
oracle on a bounded sample. --headline-only skips them.

--impl reference times the oracle (the CPU reference of this pattern) instead, on a
bounded sample of the same workload, and prints the same line with "impl": "reference".
--workload picks one other configuration; --all prints one line per configuration.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fused aX^T(v.*Xy)+bz: effective GB/s and % of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
FP64_PEAK_TFLOPS = 1.259  # 152 SMs x 2 DFMA/clk x 2 flops x 2.07 GHz
FP32_PEAK_TFLOPS = 78.5   # 152 SMs x 124.7 FFMA/clk (measured issue rate) x 2 flops x 2.07 GHz

def _m(kw, m):
    return dict(kw, m=m) if m else kw


WORKLOADS = {
    "dense_small": ("dense f64 1000 x 64, U[-1,1], alpha=1.5, beta=0.5",
                    lambda g, m=None: g.dense_small(**_m({}, m))),
    "dense_tall_a": ("dense f32 16,000,000 x 32, N(0,1) X/y, v U[0.1,2], alpha=1, beta=0, no z",
                     lambda g, m=None: g.dense_tall(**_m({"variant": "a"}, m))),
    "dense_tall_b": ("dense f32 16,000,000 x 32, N(0,1) X/y/z, v U[0.1,2], alpha=2, beta=-1",
                     lambda g, m=None: g.dense_tall(**_m({"variant": "b"}, m))),
    "dense_tall_c": ("dense f32 16,000,000 x 32, N(0,1) X/y, v=1 (X^T X y), alpha=1, beta=0",
                     lambda g, m=None: g.dense_tall(**_m({"variant": "c"}, m))),
    "dense_tall_bf16": ("dense 16,000,000 x 32 with X in bfloat16, fp32 vectors and arithmetic, N(0,1) X/y/z, "
                        "v U[0.1,2], alpha=2, beta=-1",
                        lambda g, m=None: g.dense_tall(**_m({"variant": "b", "x_store": "bf16"}, m))),
    "dense_wide": ("dense f64 20,000 x 20,000, U[-1,1], alpha=0.7, beta=0.3",
                   lambda g, m=None: g.dense_wide(**_m({}, m))),
    "csr_uniform": ("CSR f64 4,000,000 x 10,000, Poisson(50) uniform distinct columns, U[-1,1], alpha=beta=1",
                    lambda g, m=None: g.csr_uniform(**_m({}, m))),
    "dense_multi": ("dense f32 16,000,000 x 32 with k=8 right-hand sides: Y, Z (32 x 8) N(0,1), V (16,000,000 x 8) "
                    "U[0.1,2], alpha=2, beta=-1",
                    lambda g, m=None: g.dense_multi(**_m({}, m))),
    "dense_multi_k16": ("dense f32 16,000,000 x 32 with k=16 right-hand sides: Y, Z (32 x 16) N(0,1), V "
                        "(16,000,000 x 16) U[0.1,2], alpha=2, beta=-1",
                        lambda g, m=None: g.dense_multi(**_m({"k": 16}, m))),
    "dense_multi_k32": ("dense f32 16,000,000 x 32 with k=32 right-hand sides: Y, Z (32 x 32) N(0,1), V "
                        "(16,000,000 x 32) U[0.1,2], alpha=2, beta=-1",
                        lambda g, m=None: g.dense_multi(**_m({"k": 32}, m))),
    "dense_multi_shared": ("dense f32 16,000,000 x 32 with k=8 right-hand sides and one shared v: Y, Z (32 x 8) "
                           "N(0,1), v U[0.1,2], alpha=2, beta=-1",
                           lambda g, m=None: g.dense_multi(**_m({"v_mode": "shared"}, m))),
    "csr_powerlaw": ("CSR f32 2,000,000 x 1,000,000, Zipf(1.5) row lengths (mean 100, cap 50,000), Zipf(1.1) "
                     "columns, N(0,1) vals/y, v U[0,1], alpha=1, beta=0",
                     lambda g, m=None: g.csr_powerlaw(**_m({}, m))),
    "csr_powerlaw_rotated": ("CSR f32 2,000,000 x 1,000,000 as csr_powerlaw with every column index rotated by "
                             "500,000 (the hot columns mid-range)",
                             lambda g, m=None: g.csr_powerlaw(**_m({"col_offset": 500_000}, m))),
}


def dominant_kernel(p) -> str:
    """The kernel that carries the call, from the launch plan the library picks."""
    import dense_linear_algebra_gb300 as fx

    if p.x_store == "bf16":
        return "dense_tile_kernel"
    if is_multi(p):
        vm = "none" if p.v is None else ("full" if p.v.ndim == 2 else "shared")
        plan = fx.multi_plan_describe(dtype_name(p), p.m, p.n, p.y.shape[1], vm, p.ld)
        return "dense_multi_tc_kernel" if " tc=1 " in plan else "dense_multi_kernel"
    if p.kind == "csr":
        # rows longer than the plan's one-warp limit go to the long-row kernel, which dominates
        # when they hold most entries; otherwise the row kernel of the plan (lane groups for
        # fp64, packed batches for fp32)
        desc = fx.plan_describe("csr", dtype_name(p), p.m, p.n, p.nnz)
        f = dict(kv.split("=") for kv in desc.split()[1:] if "=" in kv)
        lens = np.diff(p.row_ptr)
        if lens[lens > int(f["warp_cap"])].sum() > 0.5 * p.nnz:
            return "csr_long_kernel"
        return "csr_group_kernel" if int(f["group_lanes"]) > 0 else "csr_rows_kernel"
    desc = fx.plan_describe("dense", dtype_name(p), p.m, p.n, 0, p.ld)
    kind = dict(kv.split("=") for kv in desc.split()[1:] if "=" in kv)["kind"]
    if kind == "wide" and dtype_name(p) == "f64":
        return "dense_wide_f64_kernel"
    return {"tile_tma": "dense_tile_kernel", "narrow_tma": "dense_narrow_kernel", "narrow_direct": "dense_narrow_kernel",
            "wide": "dense_wide_kernel"}.get(kind, kind)


def is_multi(p) -> bool:
    return p.kind == "dense" and p.y.ndim == 2


def model_estimate(p):
    """The launch model's plan for the call and its roofline estimate of the duration."""
    import dense_linear_algebra_gb300 as fx

    if is_multi(p):
        vm = "none" if p.v is None else ("full" if p.v.ndim == 2 else "shared")
        desc = fx.multi_plan_describe(dtype_name(p), p.m, p.n, p.y.shape[1], vm, p.ld)
        return {"plan": desc, "est_us": float(dict(kv.split("=") for kv in desc.split()[1:])["est_us"])}
    if p.kind == "csr":
        desc = fx.plan_describe("csr", dtype_name(p), p.m, p.n, p.nnz)
    elif p.x_store == "bf16":
        return {"plan": "bfloat16 X: the fp32 model's tile plan with 2-byte elements"}
    else:
        desc = fx.plan_describe("dense", dtype_name(p), p.m, p.n, 0, p.ld)
    f = dict(kv.split("=") for kv in desc.split()[1:] if "=" in kv)
    return {"plan": desc, "est_us": float(f.get("est_us", "nan"))}


def _num(v):
    """A positive number from a peak entry: a number, or a record holding one."""
    if isinstance(v, dict):
        for k in ("value", "burst", "gbs", "GBs", "measured"):
            if k in v:
                return _num(v[k])
        return None
    try:
        f = float(v)
    except (TypeError, ValueError):
        return None
    return f if f > 0 and f == f and f != float("inf") else None


def measured_peaks(path=None):
    """(HBM GB/s, "measured" | "fallback", the file's records) from the measured-peaks file."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
        except Exception:
            d = None
        if isinstance(d, dict):
            keys = ["hbm_gbs", "hbm_GBs", "hbm_copy_gbs"]
            keys += sorted(k for k in d if "hbm" in k.lower() and k not in keys)
            for k in keys:
                f = _num(d.get(k))
                if f is not None:
                    return f, "measured", d
    return FALLBACK_HBM_GBS, "fallback", {}


def fp64_peak_tflops(peaks):
    f = _num(peaks.get("fp64_tflops"))
    return FP64_PEAK_TFLOPS if f is None else f


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout: float):
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


KERNEL_SOURCES = {"dense": ["dense.cu", "common.cuh", "kernels.h"], "csr": ["csr.cu", "common.cuh", "kernels.h"],
                  "multi": ["multi.cu", "multi.h", "common.cuh", "kernels.h"],
                  "multi_tc": ["multi_tc.cu", "multi.h", "common.cuh", "kernels.h"]}


def source_sha(kernel: str) -> str:
    """Hash of the source files that define a kernel (its .cu file and the device headers it includes)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_linear_algebra_gb300", "csrc")
    group = ("csr" if kernel.startswith("csr") else "multi_tc" if kernel.startswith("dense_multi_tc")
             else "multi" if kernel.startswith("dense_multi") else "dense")
    for fn in KERNEL_SOURCES[group]:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, name: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(f"{kernel} {name}")
    except Exception:
        return None
    if not d or d.get("source_sha") != source_sha(kernel):
        return None
    return d.get("dram_bytes_per_launch")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate_over_ranks(ms_step, world, ideal_bytes, dist, device):
    """Whole-job figures for `world` independent replicas: the slowest rank's step time
    (max over ranks) and the bytes of every rank over it, in GB/s."""
    if dist is not None and world > 1:
        import torch

        tt = torch.tensor([ms_step], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_step = float(tt.item())
    return ms_step, world * ideal_bytes / (ms_step * 1e-3) / 1e9


def cpu_oracle_time(p, budget_s: float, min_reps: int = 1, max_reps: int = 5):
    """Times the oracle's double-accumulator pass (one thread) on problem p."""
    import oracle

    times = []
    t_all = time.perf_counter()
    while len(times) < max_reps:
        t0 = time.perf_counter()
        oracle.solve(p, acc="d")
        times.append(time.perf_counter() - t0)
        if len(times) >= min_reps and time.perf_counter() - t_all > budget_s:
            break
    return statistics.median(times), len(times)


def sample_problem(p, rows: int):
    """The first `rows` rows of a problem (same recipe, bounded CPU work)."""
    import inputgen

    if p.kind == "dense" or rows >= p.m:
        if rows >= p.m:
            return p
        return inputgen.Problem(p.name + f"_first{rows}", p.kind, p.dtype, rows, p.n, p.alpha, p.beta, y=p.y,
                                v=None if p.v is None else p.v[:rows], z=p.z, X=p.X[:rows], ld=p.ld)
    rp = p.row_ptr[: rows + 1].copy()
    nnz = int(rp[-1])
    return inputgen.Problem(p.name + f"_first{rows}", p.kind, p.dtype, rows, p.n, p.alpha, p.beta, y=p.y,
                            v=None if p.v is None else p.v[:rows], z=p.z, row_ptr=rp, col_idx=p.col_idx[:nnz],
                            vals=p.vals[:nnz])


def run_reference(args, name, desc, p):
    """--impl reference: the oracle on the host cores, a bounded sample per step."""
    rows = max(1, p.m // 4)
    sp = sample_problem(p, rows)
    for _ in range(args.warmup):
        cpu_oracle_time(sp, 0.0, 1, 1)
    ts = [cpu_oracle_time(sp, 0.0, 1, 1)[0] for _ in range(args.steps)]
    t = statistics.median(ts)
    val = sp.ideal_bytes() / t / 1e9
    sample = f"first {rows} of {p.m} rows of the workload ({sp.ideal_bytes()} algorithmic bytes) per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(p), "data": "synthetic",
        "config": {"workload": desc, "name": name},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def dtype_name(p):
    if p.x_store == "bf16":
        return "bf16 X, f32"
    return "f32" if np.dtype(p.dtype) == np.float32 else "f64"


def time_e2e(args, host, d, call, out, out_host, stream, ideal):
    """End to end: H2D of the step's inputs from pinned memory, the call, D2H of out."""
    import torch

    e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        for k, t in host.items():
            if t is not None:
                d[k].copy_(t, non_blocking=True)
        call()
        out_host.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        for k, t in host.items():
            if t is not None:
                d[k].copy_(t, non_blocking=True)
        call()
        out_host.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    e2e_val = ideal / (e2e_ms * 1e-3) / 1e9

    return e2e_ms, e2e_val


def time_unfused(args, p, d, X, out, dev, stream, ideal, ms_step):
    """The unfused library sequence on the same GPU."""
    import torch

    # the unfused library sequence on the same GPU (dense: cuBLAS gemv, scale, transposed gemv)
    if p.x_store == "bf16":
        return {"error": "no library gemv takes bfloat16 X with fp32 vectors and fp32 accumulation"}
    if is_multi(p):
        try:
            k = p.y.shape[1]
            tz = d["z"] if (d["z"] is not None and p.beta != 0) else torch.zeros((p.n, k), dtype=out.dtype, device=dev)
            vv = None if d["v"] is None else (d["v"] if d["v"].dim() == 2 else d["v"][:, None])

            def lib_seq():
                u = torch.mm(X, d["y"])
                t = u * vv if vv is not None else u
                return torch.addmm(tz, X.t(), t, beta=p.beta, alpha=p.alpha)
            for _ in range(3):
                lib_seq()
            torch.cuda.synchronize()
            u0 = torch.cuda.Event(enable_timing=True)
            u1 = torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            for _ in range(args.steps):
                lib_seq()
            u1.record(stream)
            torch.cuda.synchronize()
            ums = u0.elapsed_time(u1) / args.steps
            return {"what": "torch.mm (cuBLAS GEMM X Y), V scale, torch.addmm on X^T (cuBLAS GEMM)",
                    "ms_per_step": round(ums, 4), "value": round(ideal / (ums * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "fused_speedup": round(ums / ms_step, 3)}
        except Exception as e:  # report, do not fail the bench
            return {"error": str(e)[:200]}
    if p.kind == "dense":
        try:
            Xt = X
            tz = d["z"] if (d["z"] is not None and p.beta != 0) else torch.zeros(p.n, dtype=out.dtype, device=dev)

            def lib_seq():
                u = torch.mv(Xt, d["y"])
                t = u * d["v"] if d["v"] is not None else u
                return torch.addmv(tz, Xt.t(), t, beta=p.beta, alpha=p.alpha)
            for _ in range(3):
                lib_seq()
            torch.cuda.synchronize()
            u0 = torch.cuda.Event(enable_timing=True)
            u1 = torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            for _ in range(args.steps):
                lib_seq()
            u1.record(stream)
            torch.cuda.synchronize()
            ums = u0.elapsed_time(u1) / args.steps
            unfused = {"what": "torch.mv (cuBLAS gemv N), v scale, torch.addmv on X^T (cuBLAS gemv T)",
                       "ms_per_step": round(ums, 4), "value": round(ideal / (ums * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "fused_speedup": round(ums / ms_step, 3)}
        except Exception as e:  # report, do not fail the bench
            unfused = {"error": str(e)[:200]}
    else:
        try:
            # cuSPARSE takes one index type for both arrays: widen col_idx to int64 to match row_ptr
            Xs = torch.sparse_csr_tensor(d["row_ptr"], d["col_idx"].to(torch.int64), d["vals"], size=(p.m, p.n))
            XsT = Xs.t().to_sparse_csr()
            tz = d["z"] if (d["z"] is not None and p.beta != 0) else torch.zeros(p.n, dtype=out.dtype, device=dev)

            def lib_seq():
                u = torch.mv(Xs, d["y"])
                t = u * d["v"] if d["v"] is not None else u
                return torch.addmv(tz, XsT, t, beta=p.beta, alpha=p.alpha)
            for _ in range(3):
                lib_seq()
            torch.cuda.synchronize()
            u0 = torch.cuda.Event(enable_timing=True)
            u1 = torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            for _ in range(args.steps):
                lib_seq()
            u1.record(stream)
            torch.cuda.synchronize()
            ums = u0.elapsed_time(u1) / args.steps
            unfused = {"what": "torch CSR mv (cuSPARSE SpMV), v scale, addmv on a pre-transposed CSR copy of X",
                       "ms_per_step": round(ums, 4), "value": round(ideal / (ums * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "fused_speedup": round(ums / ms_step, 3)}
            del Xs, XsT
        except Exception as e:
            unfused = {"error": str(e)[:200]}

    return unfused


L2_FLUSH_BYTES = 256 << 20  # larger than GB300's 129 MB L2


GATE_CYCLES = 2_000_000  # a ~1 ms spin on the device that holds the stream while a call is enqueued


def time_isolated(call, stream, reps: int, flush=None):
    """Per-call device times (us) of `reps` isolated calls, one CUDA-event pair each. With
    `flush`, a write of L2_FLUSH_BYTES before every call evicts L2 (cold-cache calls).

    Each call is enqueued behind a device-side spin, so the first event and the call are both
    queued before the device reaches them: the pair then times the call alone, not the host's
    enqueue latency (which an idle device would otherwise wait out between the two events)."""
    import torch

    ts = []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        torch.cuda._sleep(GATE_CYCLES)
        if flush is not None:
            flush.fill_(1)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return ts


def percentiles(ts):
    q = np.percentile(np.asarray(ts, dtype=np.float64), [10, 50, 90])
    return {"p10": round(float(q[0]), 2), "p50": round(float(q[1]), 2), "p90": round(float(q[2]), 2),
            "calls": len(ts)}


def run_fused(args, name, desc, p, rank, world, dist):
    import torch

    import dense_linear_algebra_gb300 as fx

    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)

    def pin(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    host = {}
    if p.kind == "dense":
        host["X"] = pin(p.X)
        if p.x_store == "bf16":  # bfloat16-representable values: exact
            host["X"] = host["X"].to(torch.bfloat16).pin_memory()
    else:
        host["row_ptr"], host["col_idx"], host["vals"] = pin(p.row_ptr), pin(p.col_idx), pin(p.vals)
    host["y"], host["v"], host["z"] = pin(p.y), pin(p.v), pin(p.z)
    d = {k: (None if t is None else t.to(dev, non_blocking=False)) for k, t in host.items()}
    out = torch.empty(p.y.shape, dtype=d["y"].dtype, device=dev)
    out_host = torch.empty(p.y.shape, dtype=d["y"].dtype).pin_memory()

    if is_multi(p):
        X = d["X"][:, : p.n]

        def call(o=out):
            return fx.dense_multi(X, d["y"], d["v"], p.alpha, p.beta, d["z"], out=o, stream=stream)
        plan = fx.multi_plan_describe(dtype_name(p), p.m, p.n, p.y.shape[1],
                                      "none" if p.v is None else ("full" if p.v.ndim == 2 else "shared"), p.ld)
        launches = int(dict(kv.split("=") for kv in plan.split()[1:])["passes"])
    elif p.kind == "dense":
        X = d["X"][:, : p.n]

        def call(o=out):
            return fx.dense(X, d["y"], d["v"], p.alpha, p.beta, d["z"], out=o, stream=stream)
        launches = 1 if p.n * p.itemsize <= 2048 else 2
    else:
        analysis = None
        if args.analyze:
            analysis = fx.csr_analyze(d["row_ptr"], d["col_idx"], p.n, dtype_name(p), stream=stream)

        def call(o=out):
            return fx.csr(d["row_ptr"], d["col_idx"], d["vals"], d["y"], p.n, d["v"], p.alpha, p.beta, d["z"],
                          out=o, stream=stream)
        launches = 3

    ideal = p.ideal_bytes()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[dev.index] if vis else str(dev.index)
    with ClockSampler(smi_index) as clk:
        clk.wait_first(3.0)
        for _ in range(max(args.warmup, 3)):
            call()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        # device-timed steps, inputs resident
        wall0 = time.time()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            call()
        t_end.record(stream)
        torch.cuda.synchronize()
        # the same step keeps running until the clock window spans a second
        extra = 0
        while time.time() - wall0 < 1.0:
            for _ in range(20):
                call()
            extra += 20
            torch.cuda.synchronize()
    # the same call in isolation, one event pair per call: after an L2 flush (cold cache, as ncu's
    # serialised launch list sees it), and for inputs that fit in L2 also hot
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    iso_cold = time_isolated(call, stream, max(args.steps, 5), flush)
    del flush
    iso_hot = time_isolated(call, stream, max(args.steps, 5)) if p.ideal_bytes() <= 64e6 else None
    if dist:
        dist.barrier()
    # one event pair around the K back-to-back calls: events between calls would stop
    # consecutive launches from overlapping and add their drain time to every call
    total_ms = t_start.elapsed_time(t_end)
    ms_step = total_ms / args.steps
    ms_step, value = aggregate_over_ranks(ms_step, world, ideal, dist, dev)
    kernel_ms = total_ms / args.steps

    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = out_host.numel() * out_host.element_size()
    e2e_ms = e2e_val = None
    unfused = None
    if not args.no_extras:
        e2e_ms, e2e_val = time_e2e(args, host, d, call, out, out_host, stream, ideal)
        unfused = time_unfused(args, p, d, X if p.kind == "dense" else None, out, dev, stream, ideal, ms_step)

    peak, peak_kind, peaks = measured_peaks()
    kernel = dominant_kernel(p)
    traffic = profiled_traffic(kernel, name)
    achieved = ideal / (kernel_ms * 1e-3) / 1e9
    rec = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(p), "data": "synthetic",
        "config": {"workload": desc, "name": name, "algorithmic_bytes_per_step": ideal,
                   "l2": "inputs larger than L2 (129 MB); no flush" if ideal > 256e6 else
                         "inputs fit in L2: hot-L2 figure",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_call": round(kernel_ms * 1e3, 2),
        "isolated_call_us": dict({"l2_flushed": percentiles(iso_cold)},
                                 **({"hot_l2": percentiles(iso_hot)} if iso_hot is not None else {})),
        "hbm_pct_of_peak": round(100 * value / world / peak, 2),
        "hbm_pct_of_nominal_7900": round(100 * value / world / 7900.0, 2),
        "clocks": dict(clk.summary(), window=f"{args.steps} timed steps + {extra} identical steps (>= 1 s)"),
        "e2e": None if e2e_val is None else {"value": round(e2e_val, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                                             "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "kernel": kernel},
        "unfused_library": unfused,
        "model": model_estimate(p),
    }
    if is_multi(p) and kernel == "dense_multi_tc_kernel":
        # both products on the tensor cores (bfloat16 terms, fp32 accumulation): per 128-row tile
        # 6 + 8 MMAs of M = 128, K = 16 and N = 3 kb rounded up to 16; the kernel is bound by the
        # number of MMAs and shared-memory traffic long before the tensor pipe's flop rate
        k = p.y.shape[1]
        kb = 8 if k <= 8 else (16 if k <= 16 else 32)
        nw = (3 * kb + 15) // 16 * 16
        passes = -(-k // kb)
        tiles = -(-p.m // 128)
        mma_flops = 2.0 * 128 * nw * 16 * 14 * tiles * passes
        bf16_peak = _num(peaks.get("bf16_tflops")) if isinstance(peaks, dict) else None
        rec["roofline_tensor"] = {"bound": "tensor", "algorithmic_flops_per_step": 4.0 * p.m * p.n * k,
                                  "executed_mma_flops_per_step": mma_flops,
                                  "achieved": round(mma_flops / (kernel_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                                  "peak": bf16_peak, "peak_source": "measured cuBLAS bf16 (burst)",
                                  "frac": None if not bf16_peak else round(mma_flops / (kernel_ms * 1e-3) / 1e12 /
                                                                          bf16_peak, 4)}
        rec["config"]["right_hand_sides"] = int(k)
    elif is_multi(p):
        # k right-hand sides: two FMAs (4 flops) per stored element per right-hand side, on the fp32 or fp64 pipe
        flops = 4.0 * p.m * p.n * p.y.shape[1]
        alu_peak = FP32_PEAK_TFLOPS if dtype_name(p) == "f32" else fp64_peak_tflops(peaks)
        rec["roofline_alu"] = {"bound": "alu", "achieved": round(flops / (kernel_ms * 1e-3) / 1e12, 4),
                               "peak": alu_peak, "unit": "TFLOP/s",
                               "frac": round(flops / (kernel_ms * 1e-3) / 1e12 / alu_peak, 4),
                               "peak_source": "152 SMs x 124.7 FFMA/clk (probe) x 2 flops x 2.07 GHz" if alu_peak ==
                               FP32_PEAK_TFLOPS else "152 SMs x 2 DFMA/clk x 2 flops x 2.07 GHz (DFMA probe: 1.254)",
                               "algorithmic_flops_per_step": flops}
        rec["config"]["right_hand_sides"] = int(p.y.shape[1])
        if flops / (alu_peak * 1e12) > ideal / (peak * 1e9):
            rec["roofline"]["bound"] = "alu"
    elif dtype_name(p) == "f64":
        # fp64 runs on GB300's fp64 units: 2 DFMA per clock per SM (measured 1.254 TFLOP/s), and the
        # pattern needs two FMAs (4 flops) per stored element, so the fp64 rate can bind before HBM
        flops = 4.0 * (p.m * p.n if p.kind == "dense" else p.nnz)
        fp64_peak = fp64_peak_tflops(peaks)
        rec["roofline_alu"] = {"bound": "alu", "achieved": round(flops / (kernel_ms * 1e-3) / 1e12, 4),
                               "peak": fp64_peak, "unit": "TFLOP/s",
                               "frac": round(flops / (kernel_ms * 1e-3) / 1e12 / fp64_peak, 4),
                               "peak_source": "152 SMs x 2 DFMA/clk x 2 flops x 2.07 GHz (DFMA probe: 1.254)",
                               "algorithmic_flops_per_step": flops}
        hbm_time = ideal / (peak * 1e9)
        alu_time = flops / (fp64_peak * 1e12)
        rec["roofline"]["bound"] = "alu" if alu_time > hbm_time else "hbm"
    if p.kind == "csr":
        rec["config"]["nnz"] = p.nnz
        if analysis is not None:
            rec["config"]["analysis"] = analysis
            fx.csr_analysis_clear()
    return rec


def run_split(args, name, desc, p, rank, world, dist):
    """--split rows: one problem split by rows across the ranks (strong scaling). Each rank
    holds its row block; a step is its partial (one fused call at alpha = 1, beta = 0), one
    all-reduce of the n-vector and the epilogue kernel, on every rank."""
    import torch

    from dense_linear_algebra_gb300 import distributed as sp

    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)

    def to(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    if p.kind == "dense":
        b = sp.row_bounds(p.m, world)
        shard = sp.shard_dense(to(p.X[b[rank]:b[rank + 1], : p.n]), to(p.v[b[rank]:b[rank + 1]])
                               if p.v is not None else None, [0, b[rank + 1] - b[rank]], 0)
    else:
        b = sp.row_bounds(p.m, world, p.row_ptr)
        hs = sp.shard_csr(p.row_ptr, p.col_idx, p.vals, p.v, p.n, b, rank)
        shard = sp.RowShard("csr", p.n, hs.r0, hs.r1, v=to(hs.v), row_ptr=to(hs.row_ptr), col_idx=to(hs.col_idx),
                            vals=to(hs.vals))
    y, z = to(p.y), to(p.z)

    def step():
        return sp.sharded_call(shard, y, p.alpha, p.beta, z)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms_rank = e0.elapsed_time(e1) / args.steps
    ms_step = ms_rank
    if dist is not None and world > 1:
        tt = torch.tensor([ms_step], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_step = float(tt.item())
    ideal = p.ideal_bytes()
    peak, peak_kind, _ = measured_peaks()
    value = ideal / (ms_step * 1e-3) / 1e9
    per_call = 1 if p.kind == "dense" else 3
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": dtype_name(p), "data": "synthetic",
        "config": {"workload": desc, "name": name, "algorithmic_bytes_per_step": ideal,
                   "parallelism": f"rows split over {world} rank(s): fused partial, all-reduce of n values, epilogue",
                   "rows_this_rank": shard.rows},
        "hbm_pct_of_peak_per_gpu": round(100 * value / world / peak, 2), "peak_source": f"{peak_kind} HBM copy",
        "gpu_launches": (per_call + 1) * args.steps,
    }


def run_solver(args):
    """Ridge regression by CG on the tall workload's X: fused operator vs the cuBLAS pair, per iteration."""
    import torch

    import inputgen
    from dense_linear_algebra_gb300 import solvers

    p = inputgen.dense_tall(variant="c", m=args.rows or 16_000_000)
    dev = torch.device("cuda", 0)
    X = torch.from_numpy(p.X).to(dev)
    w_true = torch.from_numpy(inputgen.normal(0, 7, p.n, np.float32)).to(dev)
    b = torch.mv(X, w_true) + 0.1 * torch.from_numpy(inputgen.normal(0, 8, p.m, np.float32)).to(dev)
    lam = 1.0
    iters = 32
    rhs = solvers.rmatvec(X, b)

    def fused_op(q):
        return solvers.fused(X, q, None, 1.0, lam, q)

    def unfused_op(q):
        return torch.mv(X.t(), torch.mv(X, q)) + lam * q

    out = {}
    for name, op in (("fused", fused_op), ("unfused_cublas", unfused_op)):
        solvers.cg(op, rhs, tol=0.0, max_iter=3, check_every=3)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        w, info = solvers.cg(op, rhs, tol=0.0, max_iter=iters, check_every=iters)
        true_res = float(torch.linalg.vector_norm(rhs - op(w)) / torch.linalg.vector_norm(rhs))
        e1.record()
        torch.cuda.synchronize()
        out[name] = {"ms_per_iteration": round(e0.elapsed_time(e1) / info.iterations, 4),
                     "relative_residual": true_res}
    # k = 8 targets: block CG with one multi-vector call per iteration, against the cuBLAS
    # GEMM pair, per iteration of all eight solves
    k = 8
    B = torch.mm(X, torch.from_numpy(inputgen.normal(0, 9, (p.n, k), np.float32)).to(dev))
    rhs_k = torch.mm(X.t(), B).contiguous()

    def fused_multi_op(P):
        return solvers.fused_multi(X, P.contiguous(), None, 1.0, lam, P.contiguous())

    def unfused_multi_op(P):
        return torch.mm(X.t(), torch.mm(X, P)) + lam * P

    for name, op in (("fused_multi_k8", fused_multi_op), ("unfused_cublas_k8", unfused_multi_op)):
        solvers.cg_block(op, rhs_k, tol=0.0, max_iter=3, check_every=3)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        W, info = solvers.cg_block(op, rhs_k, tol=0.0, max_iter=iters, check_every=iters)
        true_res = float((torch.linalg.vector_norm(rhs_k - op(W), dim=0) / torch.linalg.vector_norm(rhs_k, dim=0)).max())
        e1.record()
        torch.cuda.synchronize()
        out[name] = {"ms_per_iteration": round(e0.elapsed_time(e1) / info.iterations, 4),
                     "relative_residual": true_res}
    rec = {"metric": "ridge regression by conjugate gradients: ms per CG iteration", "unit": "ms",
           "higher_is_better": False, "data": "synthetic",
           "config": {"workload": f"X {p.m} x {p.n} fp32 N(0,1), b = X w + 0.1 noise, lambda = 1, {iters} iterations",
                      "operator": "X^T (X p) + lambda p"},
           "fused": out["fused"], "unfused_cublas": out["unfused_cublas"],
           "speedup": round(out["unfused_cublas"]["ms_per_iteration"] / out["fused"]["ms_per_iteration"], 3),
           "k8": {"operator": "X^T (X P) + lambda P for 8 targets (block CG)", "fused_multi": out["fused_multi_k8"],
                  "unfused_cublas": out["unfused_cublas_k8"],
                  "speedup": round(out["unfused_cublas_k8"]["ms_per_iteration"] /
                                   out["fused_multi_k8"]["ms_per_iteration"], 3),
                  "vs_8_single_solves": round(8 * out["fused"]["ms_per_iteration"] /
                                              out["fused_multi_k8"]["ms_per_iteration"], 3)}}
    print(json.dumps(rec), flush=True)


# the benchmark configurations in order: (label, workload, HBM-fraction target or None)
BENCH_CONFIGS = [("1", "dense_small", None), ("2a", "dense_tall_a", 0.75), ("2b", "dense_tall_b", 0.75),
                    ("2c", "dense_tall_c", 0.75), ("3", "dense_wide", 0.75), ("4", "csr_uniform", 0.5),
                    ("5", "csr_powerlaw", 0.5)]
HEADLINE = "dense_tall_b"
CPU_SAMPLE_BYTES = 256e6  # algorithmic bytes of the oracle's sample for a configuration's cpu_baseline


def cpu_baseline_sample(p, budget_s: float = 3.0):
    """The oracle (double accumulator, one thread) on the first rows of p, about CPU_SAMPLE_BYTES of them."""
    rows = max(1, min(p.m, int(p.m * CPU_SAMPLE_BYTES / max(p.ideal_bytes(), 1))))
    sp = sample_problem(p, rows)
    t, reps = cpu_oracle_time(sp, budget_s=budget_s, min_reps=1, max_reps=3)
    return {"value": round(sp.ideal_bytes() / t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {rows} of {p.m} rows ({sp.ideal_bytes()} algorithmic bytes), double accumulator, "
                      f"single thread, median of {reps} runs of {t:.3f} s",
            "host_cores": os.cpu_count()}


def config_summary(label, target, rec):
    """The figures of one configuration's measurement, for the headline line's `configs` object."""
    peak = rec["roofline"]["peak"]
    frac = rec["roofline"]["achieved"] / peak
    d = {"workload": rec["config"]["workload"], "name": rec["config"]["name"], "dtype": rec["dtype"],
         "us_per_call": rec["us_per_call"], "isolated_call_us": rec["isolated_call_us"],
         "value": rec["roofline"]["achieved"], "unit": "GB/s", "hbm_frac_of_measured": round(frac, 4),
         "hbm_pct_of_nominal_7900": round(100 * rec["roofline"]["achieved"] / 7900.0, 2),
         "algorithmic_bytes_per_call": rec["config"]["algorithmic_bytes_per_step"],
         "roofline": rec["roofline"], "e2e": rec["e2e"], "clocks": rec["clocks"], "model": rec["model"]}
    for key in ("roofline_alu", "roofline_tensor"):
        if key in rec:
            d[key] = rec[key]
    if "nnz" in rec["config"]:
        d["nnz"] = rec["config"]["nnz"]
    u = rec.get("unfused_library") or {}
    if "ms_per_step" in u:
        d["unfused_library"] = {"what": u["what"], "us_per_call": round(u["ms_per_step"] * 1e3, 2),
                                "fused_speedup": u["fused_speedup"]}
    elif u:
        d["unfused_library"] = u
    if "cpu_baseline" in rec:
        d["cpu_baseline"] = rec["cpu_baseline"]
    if target is None:
        d["target"] = "parity; launch-bound and L2-resident, so microseconds per call (hot and L2-flushed)"
    else:
        d["target"] = f">= {int(target * 100)} % of HBM peak"
        d["meets_target"] = bool(frac >= target)
    return d


# rows beyond the benchmark configurations measured in the default run: the multi-vector form
NEXT_WORKLOADS = [("multi_k8", "dense_multi"), ("multi_k16", "dense_multi_k16"), ("multi_k32", "dense_multi_k32")]


def next_summary(rec):
    """The figures of one multi-vector measurement, for the headline line's `next` object."""
    d = {"workload": rec["config"]["workload"], "name": rec["config"]["name"], "dtype": rec["dtype"],
         "right_hand_sides": rec["config"].get("right_hand_sides"), "us_per_call": rec["us_per_call"],
         "isolated_call_us": rec["isolated_call_us"], "value": rec["roofline"]["achieved"], "unit": "GB/s",
         "hbm_frac_of_measured": rec["roofline"]["frac"], "roofline": rec["roofline"]}
    for key in ("roofline_alu", "roofline_tensor"):
        if key in rec:
            d[key] = rec[key]
    u = rec.get("unfused_library") or {}
    if "ms_per_step" in u:
        d["unfused_library"] = {"what": u["what"], "us_per_call": round(u["ms_per_step"] * 1e3, 2),
                                "fused_speedup": u["fused_speedup"]}
    return d


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fused", choices=["fused", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(WORKLOADS),
                    help="one workload only (default: the headline, with every benchmark configuration nested)")
    ap.add_argument("--headline-only", action="store_true", help="skip the nested configurations")
    ap.add_argument("--all", action="store_true", help="one line per workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=0, help="override the row count (same recipe), for profiling")
    ap.add_argument("--no-extras", action="store_true", help="skip the e2e and unfused-library legs")
    ap.add_argument("--analyze", action="store_true",
                    help="CSR: sample the matrix once (fxtx_csr_analyze) before timing, so the plan reads it")
    ap.add_argument("--solver", action="store_true", help="time ridge-regression CG on the tall X instead")
    ap.add_argument("--split", default=None, choices=["rows"],
                    help="rows: split one problem by rows across the ranks (all-reduce of n values) "
                         "instead of running independent replicas")
    args = ap.parse_args()

    import inputgen

    rank, world, local = dist_env()
    names = sorted(WORKLOADS) if args.all else [args.workload or HEADLINE]
    # the default run nests every benchmark configuration in the headline's line
    nest = not args.all and args.workload is None and not args.headline_only and args.impl == "fused"
    if args.solver:
        if rank == 0:
            run_solver(args)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        for name in names:
            desc, mk = WORKLOADS[name]
            print(json.dumps(run_reference(args, name, desc, mk(inputgen, args.rows or None))), flush=True)
        return

    import torch

    dist = None
    if world > 1:
        import torch.distributed as tdist

        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)

    if args.split == "rows":
        for name in names:
            desc, mk = WORKLOADS[name]
            p = mk(inputgen, args.rows or None)
            if is_multi(p) or p.x_store == "bf16":
                raise SystemExit("--split rows takes the single-vector fp32/fp64 workloads")
            rec = run_split(args, name, desc, p, rank, world, dist)
            if rank == 0:
                print(json.dumps(rec), flush=True)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    for name in names:
        desc, mk = WORKLOADS[name]
        p = mk(inputgen, args.rows or None)
        if args.rows:
            desc = f"{desc} [rows overridden: {p.m}]"
        rec = run_fused(args, name, desc, p, rank, world, dist)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            t, reps = cpu_oracle_time(p, budget_s=10.0, min_reps=1, max_reps=3)
            rec["cpu_baseline"] = {"value": round(p.ideal_bytes() / t / 1e9, 4), "unit": "GB/s", "cores": 1,
                                   "kind": "oracle",
                                   "sample": f"the whole workload ({p.ideal_bytes()} algorithmic bytes), double "
                                             f"accumulator, single thread, median of {reps} runs of {t:.2f} s",
                                   "host_cores": os.cpu_count()}
        del p
        if nest:
            rec["configs"] = {}
            for label, wl, target in BENCH_CONFIGS:
                if wl == name:
                    rec["configs"][label] = config_summary(label, target, rec)
                    continue
                wdesc, wmk = WORKLOADS[wl]
                q = wmk(inputgen, None)
                r = run_fused(args, wl, wdesc, q, rank, world, dist)
                if rank == 0 and world == 1 and not args.no_cpu_baseline:
                    r["cpu_baseline"] = cpu_baseline_sample(q)
                rec["configs"][label] = config_summary(label, target, r)
                del q, r
                torch.cuda.empty_cache()
            rec["config"]["configs_note"] = ("headline: configuration 2 (dense f32 16,000,000 x 32, "
                                             "alpha=2, beta=-1); every configuration, the headline included, "
                                             "under `configs`, each measured in this run; the multi-vector form "
                                             "(k = 8, 16, 32 on the same X) under `next`")
            rec["next"] = {}
            for label, wl in NEXT_WORKLOADS:
                wdesc, wmk = WORKLOADS[wl]
                q = wmk(inputgen, None)
                r = run_fused(args, wl, wdesc, q, rank, world, dist)
                rec["next"][label] = next_summary(r)
                del q, r
                torch.cuda.empty_cache()
        if rank == 0:
            print(json.dumps(rec), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
