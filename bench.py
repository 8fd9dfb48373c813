#!/usr/bin/env python
"""Benchmark of the INT4 weight-only linear layer on GB300.

A step is one decode pass over the four 7B projections at M=1 (fused QKV
4608x3584, O 3584x3584, fused gate|up 37888x3584, down 3584x18944; G=128,
symmetric), each a w4a16_linear call.  `value` is the algorithmic bytes of a
step (packed weights + scales + activations + outputs) divided by the device
time of a step, summed over ranks (each rank runs its own replica: weak
scaling, no collective on the data path).  The same run also measures the
other workloads (prefill GEMM in TFLOP/s, the W4A8 integer path, batched
asymmetric decode), reported as sub-objects of the one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as WL  # noqa: E402

METRIC = "W4A16 GEMV HBM GB/s (M=1) & prefill TFLOP/s (M=2048) vs GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------- helpers
def algorithmic_bytes(lin: WL.Linear, M: int) -> int:
    """Bytes a linear must move at least once: packed codes, scales, zero
    points (asymmetric), activations and outputs (+ bias)."""
    Kp = -(-lin.K // lin.group_size) * lin.group_size
    Ng = Kp // lin.group_size
    b = lin.N * Kp // 2 + 4 * lin.N * Ng
    if not lin.symmetric:
        b += lin.N * Ng
    if lin.kind == "w4a8":
        b += M * Kp + 4 * M
    else:
        b += 2 * M * lin.K
    b += 2 * M * lin.N
    if lin.bias:
        b += 4 * lin.N
    return b


def load_peaks():
    """(hbm GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, kind)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def _code_only(src: str) -> str:
    """C/C++/CUDA source without comments, blank lines and trailing spaces:
    what the compiler sees, so that comment edits keep a recorded capture."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] in "\"'":
            q, j = src[i], i + 1
            while j < n and src[j] != q:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    lines = ("".join(out)).split("\n")
    return "\n".join(l.rstrip() for l in lines if l.strip())


def source_digest(files) -> str:
    """Digest of the code (not the comments) of the given sources."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


DECODE_SOURCES = ["int4_weight_only_gb300/csrc/gemv.cu",
                  "int4_weight_only_gb300/csrc/gemv_split.cu",
                  "int4_weight_only_gb300/csrc/gemv_impl.cuh",
                  "int4_weight_only_gb300/csrc/w4_device.cuh",
                  "int4_weight_only_gb300/csrc/w4_internal.h"]


PREFILL_SOURCES = ["int4_weight_only_gb300/csrc/gemm_tc.cu",
                   "int4_weight_only_gb300/csrc/w4_device.cuh",
                   "int4_weight_only_gb300/csrc/w4_internal.h"]


def recorded_traffic(kernel: str, digest: str):
    """DRAM bytes from a committed ncu summary (profiles/traffic.json), if
    it was taken on the current kernel source; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("source_digest") == digest:
            return e
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"] + sel
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.15)
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
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_graph(fn, nsteps: int):
    """Capture `nsteps` calls fn(i) into one CUDA graph."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
            for i in range(nsteps):
                fn(i)
    torch.cuda.current_stream().wait_stream(s)
    return g


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """The slowest rank's time: the job is done when every replica is."""
    if world <= 1:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank_step: float, steps: int, world: int, sec: float) -> float:
    """Whole-job throughput: the bytes all `world` replicas streamed over
    `steps` steps, divided by the slowest rank's time (weak scaling)."""
    return bytes_per_rank_step * steps * world / sec / 1e9


def time_graph_steps(step_fn, K, R, world, reps=1, warm_s=0.0):
    """Replay graphs holding exactly K calls step_fn(i); returns seconds.

    reps > 1: the K-step region is timed `reps` times (each bracketed by a
    barrier and a synchronize) and the list of the `reps` times is returned.
    warm_s: untimed replays for that long first, so that the clocks sampled
    during the timed regions are those of a loaded GPU."""
    g_full = make_graph(step_fn, R)
    g_rem = make_graph(step_fn, K % R) if K % R else None
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if warm_s > 0:
        t_end = time.perf_counter() + warm_s
        while time.perf_counter() < t_end:
            for _ in range(max(1, K // R)):
                g_full.replay()
            torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        barrier(world)
        torch.cuda.synchronize()
        ev0.record()
        for _ in range(K // R):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record()
        torch.cuda.synchronize()
        barrier(world)
        out.append(ev0.elapsed_time(ev1) / 1e3)
    return out if reps > 1 else out[0]


# ---------------------------------------------------------------- our arm
class DecodeSet:
    """Device-resident rotated copies of a set of linears (M <= 16) so that a
    sequence of steps never re-reads weights from L2."""

    def __init__(self, w4, lins, M, min_bytes):
        self.w4, self.lins, self.M = w4, lins, M
        self.bytes_step = sum(algorithmic_bytes(l, M) for l in lins)
        self.R = max(2, math.ceil(min_bytes / self.bytes_step))
        base = []
        for lin in lins:
            inp = WL.make_inputs(lin, M)
            p, s, z = w4.w4_pack_rtn(inp.W.cuda(), lin.group_size, lin.symmetric)
            b = inp.bias.cuda() if inp.bias is not None else None
            base.append((p, s, z, b))
        torch.cuda.synchronize()
        self.copies = []
        for r in range(self.R):
            cp = []
            for li, (p, s, z, b) in enumerate(base):
                lin = lins[li]
                xr = WL.make_activations(lin.K, M, seed=10_000 + 97 * r + li).cuda()
                cp.append(dict(p=p.clone(), s=s.clone(), z=None if z is None else z.clone(),
                               b=b, x=xr,
                               y=torch.empty(M, lin.N, dtype=torch.bfloat16, device="cuda")))
            self.copies.append(cp)
        del base
        torch.cuda.synchronize()

    def call(self, li, r):
        lin, d = self.lins[li], self.copies[r % self.R][li]
        self.w4.w4a16_linear(d["x"], d["p"], d["s"], d["z"], d["b"], lin.N, lin.K,
                             lin.group_size, y=d["y"])

    def step(self, i):
        for li in range(len(self.lins)):
            self.call(li, i)


def measure_linears(ds: DecodeSet, reps: int):
    out = []
    for li, lin in enumerate(ds.lins):
        n = reps * ds.R
        sec = time_graph_steps(lambda i, li=li: ds.call(li, i), n, ds.R, 1)
        us = sec / n * 1e6
        b = algorithmic_bytes(lin, ds.M)
        out.append({"name": lin.name, "N": lin.N, "K": lin.K, "M": ds.M,
                    "group_size": lin.group_size, "symmetric": lin.symmetric,
                    "us": round(us, 3), "GB/s": round(b / (us * 1e-6) / 1e9, 1)})
    return out


def measure_e2e(w4, ds: DecodeSet, K: int):
    """Same metric through the public API, per step: the step's activations
    copied in from pinned host memory (one copy of all four inputs), the four
    w4a16_linear calls back to back, and the four outputs copied back to
    pinned host memory (one copy); no graphs, host overhead included.  The
    weights keep rotating over the device copies, so they stay cold."""
    xs = [d["x"] for d in ds.copies[0]]
    ys = [d["y"] for d in ds.copies[0]]
    nx = [t.numel() for t in xs]
    ny = [t.numel() for t in ys]
    dx = torch.empty(sum(nx), dtype=torch.bfloat16, device="cuda")
    dy = torch.empty(sum(ny), dtype=torch.bfloat16, device="cuda")
    hx = torch.cat([t.flatten().cpu() for t in xs]).pin_memory()
    hy = torch.empty(sum(ny), dtype=torch.bfloat16).pin_memory()
    xv = [v.view(t.shape) for v, t in zip(torch.split(dx, nx), xs)]
    yv = [v.view(t.shape) for v, t in zip(torch.split(dy, ny), ys)]
    h2d = hx.numel() * hx.element_size()
    d2h = hy.numel() * hy.element_size()

    def step(i):
        c = ds.copies[i % ds.R]
        dx.copy_(hx, non_blocking=True)
        for lin, d, x, y in zip(ds.lins, c, xv, yv):
            w4.w4a16_linear(x, d["p"], d["s"], d["z"], d["b"], lin.N, lin.K, lin.group_size, y=y)
        hy.copy_(dy, non_blocking=True)

    for i in range(5):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        step(i)
    torch.cuda.synchronize()
    return time.perf_counter() - t0, h2d, d2h


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def _oracle_row_sample(lins, frac, seed):
    """Oracle packing of a fixed random row sample of each linear (RTN is
    row-independent, so the sampled rows pack exactly as in the full
    matrix)."""
    import oracle as O
    out = []
    rng = np.random.default_rng(seed)
    for lin in lins:
        inp = WL.make_inputs(lin)
        n = max(1, int(round(lin.N * frac)))
        rows = np.sort(rng.choice(lin.N, n, replace=False))
        W = inp.W.numpy()[rows]
        out.append((lin, inp.x, O.pack_rtn(W, lin.group_size, lin.symmetric),
                    algorithmic_bytes(lin, 1) * n / lin.N))
    return out


def _oracle_step(sample):
    import oracle as O
    by = 0.0
    for lin, x, (op, os_, oz), b in sample:
        O.w4a16_linear(x, op, os_, oz, None, lin.K, lin.group_size)
        by += b
    return by


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _time_oracle_decode(lins, frac, budget_s, seed=7):
    sample = _oracle_row_sample(lins, frac, seed=seed)
    by, t, n = 0.0, 0.0, 0
    while t < budget_s and n < 2000:
        t0 = time.perf_counter()
        by += _oracle_step(sample)
        t += time.perf_counter() - t0
        n += 1
    return by / t / 1e9, n, t


def _time_oracle_w4a8(budget_s, frac=1 / 64):
    """Oracle W4A8 (per-token INT8 quantize + int64 dot products) on a fixed
    row sample of the three W4A8 linears at M = 1."""
    import oracle as O
    rng = np.random.default_rng(11)
    sample = []
    for lin in WL.w4a8_7b():
        inp = WL.make_inputs(lin)
        n = max(1, int(round(lin.N * frac)))
        rows = np.sort(rng.choice(lin.N, n, replace=False))
        op, os_, _ = O.pack_rtn(inp.W.numpy()[rows], lin.group_size, True)
        sample.append((lin, inp.x, op, os_, algorithmic_bytes(lin, 1) * n / lin.N))
    by, t, n = 0.0, 0.0, 0
    while t < budget_s and n < 2000:
        t0 = time.perf_counter()
        for lin, x, op, os_, b in sample:
            qx, sx = O.w4a8_quantize_act(x, lin.group_size)
            O.w4a8_linear(qx, sx, op, os_, None)
            by += b
        t += time.perf_counter() - t0
        n += 1
    return by / t / 1e9, n, t


def _time_oracle_prefill(budget_s, rows=16):
    """Oracle prefill at M = 2048 on a fixed sample of output rows of the
    two 7B MLP linears (fp64 dequantize + library matmul)."""
    import oracle as O
    rng = np.random.default_rng(13)
    sample = []
    for lin in WL.prefill_7b(2048):
        inp = WL.make_inputs(lin)
        r = np.sort(rng.choice(lin.N, rows, replace=False))
        sample.append((lin, inp.x, O.pack_rtn(inp.W.numpy()[r], lin.group_size, True)))
    fl, t, n = 0.0, 0.0, 0
    while t < budget_s and n < 200:
        t0 = time.perf_counter()
        for lin, x, (op, os_, oz) in sample:
            O.w4a16_linear(x, op, os_, oz, None, lin.K, lin.group_size)
            fl += 2.0 * 2048 * rows * lin.K
        t += time.perf_counter() - t0
        n += 1
    return fl / t / 1e12, n, t


def cpu_baseline(lins, frac=1 / 16):
    """The oracle as it stands, timed on bounded samples on the host cores:
    the headline is the four 7B decode linears at M = 1 on a fixed 1/16 row
    sample (oracle packing outside the timing; fp64 dequantize + matvec
    inside) with the library's default threads; the same with one thread
    (a child process with the BLAS/OpenMP thread counts set to 1), the W4A8
    oracle and the prefill oracle are reported beside it."""
    v, n, t = _time_oracle_decode(lins, frac, budget_s=8.0)
    out = {"value": round(v, 4), "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
           "sample": f"{n} passes of oracle w4a16_linear (numpy, fp64 dequantize + matvec) over "
                     f"a fixed {frac:.4f} row sample of each of the four 7B decode linears, "
                     f"M=1; {t:.1f} s",
           "cpu_model": cpu_model(), "nproc": os.cpu_count()}
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker"],
                           capture_output=True, text=True, timeout=300, env=env)
        st = json.loads(r.stdout.strip().splitlines()[-1])
        out["single_thread"] = {"value": st["value"], "unit": "GB/s", "cores": 1,
                                "sample": st["sample"]}
    except Exception as e:       # noqa: BLE001 - reported, not hidden
        out["single_thread"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    v8, n8, t8 = _time_oracle_w4a8(budget_s=3.0)
    out["w4a8"] = {"value": round(v8, 4), "unit": "GB/s", "cores": blas_threads(),
                   "sample": f"{n8} passes of oracle w4a8_quantize_act + w4a8_linear (int64) "
                             f"over a fixed 1/64 row sample of the three W4A8 linears; {t8:.1f} s"}
    vp, npf, tp = _time_oracle_prefill(budget_s=3.0)
    out["prefill_m2048"] = {"value": round(vp, 5), "unit": "TFLOP/s", "cores": blas_threads(),
                            "sample": f"{npf} passes of oracle w4a16_linear at M=2048 over 16 "
                                      f"sampled rows of each 7B MLP linear; {tp:.1f} s"}
    return out


def cpu_worker():
    """Child process of cpu_baseline: the decode oracle sample with the
    thread counts the parent set in the environment."""
    v, n, t = _time_oracle_decode(WL.decode_7b(1), 1 / 16, budget_s=4.0)
    print(json.dumps({"value": round(v, 4),
                      "sample": f"{n} passes over the same 1/16 row sample, one thread; "
                                f"{t:.1f} s"}))


def measure_prefill(w4, M, bf16_peak, peak_kind, reps=20):
    """Prefill GEMM at the 7B MLP shapes, TFLOP/s = 2*M*N*K / time."""
    lins = WL.prefill_7b(M)
    ds = DecodeSet(w4, lins, M, min_bytes=2 * L2_BYTES)
    for i in range(3):
        ds.step(i)
    torch.cuda.synchronize()
    out, tot_f, tot_s = [], 0.0, 0.0
    for li, lin in enumerate(lins):
        n = reps * ds.R
        sec = time_graph_steps(lambda i, li=li: ds.call(li, i), n, ds.R, 1) / n
        fl = 2.0 * M * lin.N * lin.K
        tot_f += fl
        tot_s += sec
        out.append({"name": lin.name, "M": M, "N": lin.N, "K": lin.K, "us": round(sec * 1e6, 2),
                    "TFLOP/s": round(fl / sec / 1e12, 1)})
    del ds
    torch.cuda.empty_cache()
    tf = tot_f / tot_s / 1e12
    tr = recorded_traffic("k_w4a16_gemm_tc", source_digest(PREFILL_SOURCES))
    traffic = None
    if tr is not None and str(M) in tr.get("dram_bytes_per_launch", {}):
        traffic = tr["dram_bytes_per_launch"][str(M)]
    return {"M": M, "value": round(tf, 1), "unit": "TFLOP/s", "per_linear": out,
            "roofline": {"kernel": "k_w4a16_gemm_tc", "bound": "tensor", "achieved": round(tf, 1),
                         "peak": bf16_peak, "unit": "TFLOP/s", "frac": round(tf / bf16_peak, 4),
                         "peak_kind": f"{peak_kind} bf16_tflops (burst, kernel timed alone)",
                         "traffic": traffic,
                         "traffic_note": "DRAM bytes of one launch per linear (gate_up, down) "
                                         "from an ncu capture of this source" if traffic else
                                         "no ncu capture recorded for this source"}}


def measure_mid_m(w4, hbm, bf16_peak, reps=20):
    """The 7B gate_up and down linears from M = 16 (the largest decode size)
    through the tensor-core path at M = 17 .. 128: per M and linear, time,
    algorithmic GB/s and TFLOP/s (where the decode/prefill threshold sits)."""
    out = []
    for M in (16, 17, 32, 64, 128):
        lins = [l for l in WL.decode_7b(M) if l.name.endswith(("gate_up", "down"))]
        ds = DecodeSet(w4, lins, M, min_bytes=3 * L2_BYTES)
        ds.step(0)
        torch.cuda.synchronize()
        per = measure_linears(ds, reps)
        for p, lin in zip(per, lins):
            sec = p["us"] * 1e-6
            out.append({"M": M, "name": lin.name.replace("decode7b_", ""), "us": p["us"],
                        "GB/s": p["GB/s"], "hbm_frac": round(p["GB/s"] / hbm, 4),
                        "TFLOP/s": round(2.0 * M * lin.N * lin.K / sec / 1e12, 1)})
        del ds
        torch.cuda.empty_cache()
    return out


class W4A8Set:
    """Rotated copies of the W4A8 linears: per call, dynamic INT8 activation
    quantization then the integer GEMV."""

    def __init__(self, w4, lins, min_bytes):
        self.w4, self.lins = w4, lins
        self.bytes_lin = [algorithmic_bytes(l, 1) for l in lins]
        self.R = max(2, math.ceil(min_bytes / sum(self.bytes_lin)))
        self.copies = []
        base = []
        for lin in lins:
            inp = WL.make_inputs(lin)
            p, sc, _ = w4.w4_pack_rtn(inp.W.cuda(), lin.group_size, True)
            base.append((p, sc, inp.bias.cuda() if inp.bias is not None else None))
        for r in range(self.R):
            cp = []
            for li, (p, sc, b) in enumerate(base):
                lin = lins[li]
                x = WL.make_activations(lin.K, 1, seed=20_000 + 31 * r + li,
                                        outlier_frac=lin.x_outlier_frac).cuda()
                qx, sx = w4.w4a8_quantize_act(x, lin.group_size)
                cp.append(dict(p=p.clone(), s=sc.clone(), b=b, x=x, qx=qx, sx=sx,
                               y=torch.empty(1, lin.N, dtype=torch.bfloat16, device="cuda")))
            self.copies.append(cp)
        torch.cuda.synchronize()

    def call(self, li, r, quant=True):
        lin, d = self.lins[li], self.copies[r % self.R][li]
        if quant:
            self.w4.w4a8_quantize_act(d["x"], lin.group_size, qx=d["qx"], sx=d["sx"])
        self.w4.w4a8_linear(d["qx"], d["sx"], d["p"], d["s"], d["b"], lin.N, lin.K,
                            lin.group_size, y=d["y"])


def measure_w4a8(w4, hbm, reps=200, group_size=None):
    """W4A8 linears at M=1: integer GEMV alone (GB/s) and quantize + GEMV."""
    lins = WL.w4a8_7b()
    if group_size is not None:
        # group-wise weight scales (one per group_size columns) instead of one per row
        lins = [WL.Linear(l.name + f"_g{group_size}", l.M, l.N, l.K, group_size, True, l.seed,
                          x_outlier_frac=l.x_outlier_frac, x_outlier_scale=l.x_outlier_scale,
                          bias=l.bias, kind="w4a8") for l in lins[:2]]
    ws = W4A8Set(w4, lins, min_bytes=3 * L2_BYTES)
    out = []
    for li, lin in enumerate(lins):
        n = reps * ws.R
        for q in (False, True):
            ws.call(li, 0, q)
        t_lin = time_graph_steps(lambda i, li=li: ws.call(li, i, False), n, ws.R, 1) / n
        t_all = time_graph_steps(lambda i, li=li: ws.call(li, i, True), n, ws.R, 1) / n
        b = ws.bytes_lin[li]
        out.append({"name": lin.name, "N": lin.N, "K": lin.K, "group_size": lin.group_size,
                    "linear_us": round(t_lin * 1e6, 3), "linear_GB/s": round(b / t_lin / 1e9, 1),
                    "quant+linear_us": round(t_all * 1e6, 3)})
    tb = sum(ws.bytes_lin)
    tt = sum(o["linear_us"] for o in out) * 1e-6
    del ws
    torch.cuda.empty_cache()
    v = tb / tt / 1e9
    return {"value": round(v, 1), "unit": "GB/s", "per_linear": out,
            "roofline": {"kernel": "k_w4a8_gemv" if group_size is None else "k_w4a8g_gemv",
                         "bound": "hbm", "achieved": round(v, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(v / hbm, 4)}}


def measure_decode_12b(w4, hbm, reps=100):
    """Batched asymmetric G=32 decode at 12B-class shapes, M in {1,4,8,16}."""
    out = []
    for M in (1, 4, 8, 16):
        lins = WL.decode_12b(M)
        ds = DecodeSet(w4, lins, M, min_bytes=3 * L2_BYTES)
        ds.step(0)
        torch.cuda.synchronize()
        per = measure_linears(ds, reps)
        tb = sum(algorithmic_bytes(l, M) for l in lins)
        tt = sum(p["us"] for p in per) * 1e-6
        out.append({"M": M, "GB/s": round(tb / tt / 1e9, 1), "frac": round(tb / tt / 1e9 / hbm, 4),
                    "per_linear": per})
        del ds
        torch.cuda.empty_cache()
    return out


def measure_swiglu(w4, hbm, reps=200):
    """Fused gate|up + SiLU (w4a16_linear_swiglu, F = 18944, K = 3584) next
    to the plain gate|up linear on the same rotated weight copies: the fused
    call writes M x F outputs instead of M x 2F and needs no separate SiLU
    kernel."""
    out = []
    for M in (1, 8):
        lin = [l for l in WL.decode_7b(M) if l.name.endswith("gate_up")][0]
        F = lin.N // 2
        ds = DecodeSet(w4, [lin], M, min_bytes=3 * L2_BYTES)
        yF = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")

        def fused(i):
            d = ds.copies[i % ds.R][0]
            w4.w4a16_linear_swiglu(d["x"], d["p"], d["s"], d["z"], d["b"], F, lin.K,
                                   lin.group_size, y=yF)
        # the same with the INT8 activations of the W4A8 down projection
        # (one scale per row, Fp = F): fused, and as two launches
        qx = torch.empty(M, F, dtype=torch.int8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")

        def fused_q8(i):
            d = ds.copies[i % ds.R][0]
            w4.w4a16_linear_swiglu_q8(d["x"], d["p"], d["s"], d["z"], d["b"], F, lin.K,
                                      lin.group_size, F, y=yF, qx=qx, sx=sx)

        def two_launch_q8(i):
            fused(i)
            w4.w4a8_quantize_act(yF, F, qx=qx, sx=sx)
        for i in range(3):
            fused(i)
            ds.call(0, i)
            fused_q8(i)
            two_launch_q8(i)
        torch.cuda.synchronize()
        n = reps * ds.R
        t_lin = time_graph_steps(lambda i: ds.call(0, i), n, ds.R, 1) / n
        t_fus = time_graph_steps(fused, n, ds.R, 1) / n
        t_q8 = time_graph_steps(fused_q8, n, ds.R, 1) / n
        t_2l = time_graph_steps(two_launch_q8, n, ds.R, 1) / n
        b = algorithmic_bytes(lin, M) - 2 * M * lin.N + 2 * M * F
        out.append({"M": M, "F": F, "K": lin.K, "fused_us": round(t_fus * 1e6, 3),
                    "gate_up_linear_us": round(t_lin * 1e6, 3),
                    "GB/s": round(b / t_fus / 1e9, 1), "frac": round(b / t_fus / 1e9 / hbm, 4),
                    "fused_int8_us": round(t_q8 * 1e6, 3),
                    "swiglu_then_quantize_us": round(t_2l * 1e6, 3)})
        del ds
        torch.cuda.empty_cache()
    return out


def measure_moe(w4, hbm, reps=100):
    """Expert layer at decode (128 experts, 8 per token, G = 32 symmetric):
    the grouped call per projection over rotated copies of the stacked
    expert weights, GB/s over the bytes of the experts that have tokens.
    For context, the same gate|up work as one w4a16_linear call per active
    expert (the host knows the counts here; a serving loop would not)."""
    out = []
    E = WL.MOE_EXPERTS
    for batch in (16, 4):
        counts = WL.moe_route_counts(batch, seed=batch)
        T, gmax = sum(counts), max(counts)
        act = [e for e in range(E) if counts[e]]
        goff = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
        goff[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32, device="cuda"), 0,
                                dtype=torch.int32)
        lins = WL.moe_decode(batch)
        per_copy = sum(E * l.N * l.K * 0.6 for l in lins)
        R = max(2, math.ceil(3 * L2_BYTES / per_copy))
        copies = []
        for r in range(R):
            cp = []
            for lin in lins:
                # random codes and scales drawn on the device (timing only)
                Kp = -(-lin.K // lin.group_size) * lin.group_size
                g = torch.Generator(device="cuda")
                g.manual_seed(lin.seed + r)
                p = torch.randint(0, 256, (E * lin.N, Kp // 2), generator=g, device="cuda",
                                  dtype=torch.int32).to(torch.uint8)
                s = torch.rand(E * lin.N, Kp // lin.group_size, generator=g,
                               device="cuda") * 0.01 + 1e-4
                x = WL.make_activations(lin.K, T, seed=30_000 + 7 * r + lin.seed)
                cp.append(dict(p=p, s=s, x=x.cuda(),
                               y=torch.empty(T, lin.N, dtype=torch.bfloat16, device="cuda")))
            copies.append(cp)
        torch.cuda.synchronize()

        def call(li, i):
            lin, d = lins[li], copies[i % R][li]
            w4.w4a16_grouped_linear(d["x"], goff, d["p"], d["s"], None, None, E, lin.N, lin.K,
                                    lin.group_size, gmax, y=d["y"])
        for i in range(3):
            call(0, i)
            call(1, i)
        torch.cuda.synchronize()
        res = {"batch": batch, "tokens_routed": T, "active_experts": len(act), "max_per_expert": gmax}
        tot_b = tot_t = 0.0
        for li, lin in enumerate(lins):
            n = reps * R
            sec = time_graph_steps(lambda i, li=li: call(li, i), n, R, 1) / n
            Kp = -(-lin.K // lin.group_size) * lin.group_size
            b = len(act) * (lin.N * Kp // 2 + 4 * lin.N * (Kp // lin.group_size)) \
                + 2 * T * lin.K + 2 * T * lin.N
            tot_b += b
            tot_t += sec
            res[lin.name.split("_b")[0] + "_us"] = round(sec * 1e6, 3)
            res[lin.name.split("_b")[0] + "_GB/s"] = round(b / sec / 1e9, 1)
        res["GB/s"] = round(tot_b / tot_t / 1e9, 1)
        res["frac"] = round(tot_b / tot_t / 1e9 / hbm, 4)
        # context: one w4a16_linear per active expert (gate|up)
        lin = lins[0]
        rows = {e: (int(sum(counts[:e])), counts[e]) for e in act}

        def per_expert(i):
            d = copies[i % R][0]
            for e in act:
                t0, c = rows[e]
                w4.w4a16_linear(d["x"][t0:t0 + c], d["p"][e * lin.N:(e + 1) * lin.N],
                                d["s"][e * lin.N:(e + 1) * lin.N], None, None, lin.N, lin.K,
                                lin.group_size, y=d["y"][t0:t0 + c])
        per_expert(0)
        torch.cuda.synchronize()
        n = 5 * R
        res["gate_up_one_call_per_expert_us"] = round(
            time_graph_steps(per_expert, n, R, 1) / n * 1e6, 2)
        out.append(res)
        del copies
        torch.cuda.empty_cache()
    return out


def measure_moe_prefill(w4, hbm, batch=512, reps=20):
    """Expert layer at prefill (batch 512, 8 of 128 experts per token: 4096
    routed rows, 32 per expert on average): the grouped call per projection
    with 64-token tiles on the tensor-core kernel, TFLOP/s over 2 T N K and
    GB/s over the active experts' bytes; for context the same call with
    16-token tiles (the decode kernel, which re-reads each expert's weights
    once per tile)."""
    E = WL.MOE_EXPERTS
    counts = WL.moe_route_counts(batch, seed=batch)
    T = sum(counts)
    act = sum(1 for c in counts if c)
    goff = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    goff[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32, device="cuda"), 0,
                            dtype=torch.int32)
    lins = WL.moe_decode(batch)
    per_copy = sum(E * l.N * l.K * 0.6 for l in lins)
    R = max(2, math.ceil(3 * L2_BYTES / per_copy))
    copies = []
    for r in range(R):
        cp = []
        for lin in lins:
            Kp = -(-lin.K // lin.group_size) * lin.group_size
            g = torch.Generator(device="cuda")
            g.manual_seed(lin.seed + 50 + r)
            p = torch.randint(0, 256, (E * lin.N, Kp // 2), generator=g, device="cuda",
                              dtype=torch.int32).to(torch.uint8)
            s = torch.rand(E * lin.N, Kp // lin.group_size, generator=g,
                           device="cuda") * 0.01 + 1e-4
            x = WL.make_activations(lin.K, T, seed=40_000 + 7 * r + lin.seed)
            cp.append(dict(p=p, s=s, x=x.cuda(),
                           y=torch.empty(T, lin.N, dtype=torch.bfloat16, device="cuda")))
        copies.append(cp)
    torch.cuda.synchronize()
    res = {"batch": batch, "tokens_routed": T, "active_experts": act,
           "max_per_expert": max(counts)}
    for tile in (64, 16):
        def call(li, i, tile=tile):
            lin, d = lins[li], copies[i % R][li]
            w4.w4a16_grouped_linear(d["x"], goff, d["p"], d["s"], None, None, E, lin.N, lin.K,
                                    lin.group_size, tile, y=d["y"])
        for i in range(3):
            call(0, i)
            call(1, i)
        torch.cuda.synchronize()
        tot_f = tot_t = 0.0
        for li, lin in enumerate(lins):
            n = reps * R
            sec = time_graph_steps(lambda i, li=li: call(li, i), n, R, 1) / n
            f = 2.0 * T * lin.N * lin.K
            Kp = -(-lin.K // lin.group_size) * lin.group_size
            b = act * (lin.N * Kp // 2 + 4 * lin.N * (Kp // lin.group_size)) \
                + 2 * T * lin.K + 2 * T * lin.N
            tot_f += f
            tot_t += sec
            key = f"{lin.name.split('_b')[0]}_tile{tile}"
            res[key + "_us"] = round(sec * 1e6, 2)
            res[key + "_TFLOP/s"] = round(f / sec / 1e12, 1)
            res[key + "_GB/s"] = round(b / sec / 1e9, 1)
        res[f"tile{tile}_TFLOP/s"] = round(tot_f / tot_t / 1e12, 1)
    del copies
    torch.cuda.empty_cache()
    return res


def measure_bf16p(w4, hbm, reps=200):
    """The 7B decode step with the bf16 parameter layout (bf16 scales; the
    step's linears are symmetric, so no offsets): per linear and per step,
    GB/s over its own algorithmic bytes (2-byte scales)."""
    lins = WL.decode_7b(1)
    per_copy = sum(algorithmic_bytes(l, 1) for l in lins)
    R = max(2, math.ceil(3 * L2_BYTES / per_copy))
    base = []                                   # (packed, bf16 scales) per linear
    for lin in lins:
        p, sb, _ = w4.w4_pack_rtn_bf16(WL.make_inputs(lin).W.cuda(), lin.group_size, True)
        base.append((p, sb))
    copies = []
    for r in range(R):
        copies.append([dict(p=p.clone(), sb=sb.clone(),
                            x=WL.make_activations(lin.K, 1, seed=10_000 + 97 * r + li).cuda(),
                            y=torch.empty(1, lin.N, dtype=torch.bfloat16, device="cuda"))
                       for li, (lin, (p, sb)) in enumerate(zip(lins, base))])
    del base
    torch.cuda.synchronize()

    def call(li, i):
        lin, d = lins[li], copies[i % R][li]
        w4.w4a16_linear_bf16p(d["x"], d["p"], d["sb"], None, None, lin.N, lin.K, lin.group_size,
                              y=d["y"])

    def step(i):
        for li in range(len(lins)):
            call(li, i)
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    out, tb = [], 0
    for li, lin in enumerate(lins):
        n = reps * R
        sec = time_graph_steps(lambda i, li=li: call(li, i), n, R, 1) / n
        b = algorithmic_bytes(lin, 1) - 2 * lin.N * (lin.K // lin.group_size)   # 2-byte scales
        tb += b
        out.append({"name": lin.name, "us": round(sec * 1e6, 3), "GB/s": round(b / sec / 1e9, 1)})
    n = reps * R
    sec = time_graph_steps(step, n, R, 1) / n
    return {"step_us": round(sec * 1e6, 2), "GB/s": round(tb / sec / 1e9, 1),
            "frac": round(tb / sec / 1e9 / hbm, 4), "per_linear": out}


def measure_gptq(w4, reps=3):
    """GPTQ of the 7B fused QKV projection (4608 x 3584, G = 128,
    symmetric) from 512 calibration tokens, on the device: Hessian, Cholesky,
    triangular inverse, the column loop and packing, per layer."""
    g = torch.Generator().manual_seed(9)
    N, K, T, G = 4608, 3584, 512, 128
    X = torch.randn(T, K, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(N, K, generator=g) * 0.02).cuda()
    w4.w4_gptq(X, W, G, True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        w4.w4_gptq(X, W, G, True)
    e1.record()
    torch.cuda.synchronize()
    return {"workload": f"GPTQ {N}x{K}, G={G}, {T} calibration tokens",
            "ms_per_layer": round(e0.elapsed_time(e1) / reps, 2)}


HEADLINE_REPS = 10        # timed regions of --steps steps; the median is reported


def run_ours(args, world, rank):
    import int4_weight_only_gb300 as w4
    from int4_weight_only_gb300 import build as b
    b.build()
    w4.load()
    dev = torch.cuda.current_device()
    hbm, bf16, bf16_sus, peak_kind = load_peaks()

    lins = WL.decode_7b(1)
    ds = DecodeSet(w4, lins, 1, min_bytes=3 * L2_BYTES)
    for i in range(max(args.warmup, 3)):
        ds.step(i)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        secs = time_graph_steps(ds.step, args.steps, ds.R, world, reps=HEADLINE_REPS,
                                warm_s=0.3)
    # per rank: the median of the timed regions; the job: the slowest rank
    sec = max_over_ranks(statistics.median(secs), world)
    sec_min = max_over_ranks(min(secs), world)
    sec_max = max_over_ranks(max(secs), world)
    value = aggregate_gbs(ds.bytes_step, args.steps, world, sec)
    tr = recorded_traffic("k_w4a16_gemv", source_digest(DECODE_SOURCES))
    roofline = {
        "kernel": "k_w4a16_gemv (all four launches of a step)", "bound": "hbm",
        "achieved": round(value / world, 1), "peak": hbm, "unit": "GB/s",
        "frac": round(value / world / hbm, 4), "peak_kind": f"{peak_kind} hbm_gbs",
        "traffic": None if tr is None else tr["dram_bytes_per_step"],
        "algorithmic_bytes_per_step": ds.bytes_step,
    }
    per_linear = measure_linears(ds, reps=200)
    ke = max(200, min(args.steps, 2000))     # enough steps for a stable host-side rate
    dt, h2d, d2h = measure_e2e(w4, ds, ke)
    dt = max_over_ranks(dt, world)
    e2e = {"value": round(aggregate_gbs(ds.bytes_step, ke, world, dt), 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(dt / ke * 1e3, 4), "steps": ke}
    del ds
    torch.cuda.empty_cache()

    subs = {}
    if not args.decode_only:
        # the other workloads: a failure is recorded in its own field and
        # does not take the headline measurement with it
        for name, fn in [
                ("prefill", lambda: [measure_prefill(w4, M, bf16, peak_kind) for M in (2048, 512)]),
                ("w4a8", lambda: measure_w4a8(w4, hbm)),
                ("w4a8_g128", lambda: measure_w4a8(w4, hbm, group_size=128)),
                ("decode_12b", lambda: measure_decode_12b(w4, hbm)),
                ("mid_m", lambda: measure_mid_m(w4, hbm, bf16)),
                ("swiglu_7b", lambda: measure_swiglu(w4, hbm)),
                ("moe_decode", lambda: measure_moe(w4, hbm)),
                ("moe_prefill", lambda: measure_moe_prefill(w4, hbm)),
                ("gptq", lambda: measure_gptq(w4)),
                ("decode7b_bf16_params", lambda: measure_bf16p(w4, hbm))]:
            try:
                subs[name] = fn()
            except Exception as e:          # noqa: BLE001 - reported, not hidden
                subs[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
            torch.cuda.empty_cache()

    # The line: the headline and the short per-config figures first (the
    # second half of the metric, prefill at M = 2048, included), the long
    # sub-objects last.
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian weights and activations, 7B decode shapes)",
        "hbm_frac": round(value / world / hbm, 4),
    }
    pf = subs.get("prefill")
    if isinstance(pf, list):
        for p in pf:
            tf = p["value"]
            res[f"prefill_m{p['M']}_tflops"] = tf
            res[f"prefill_m{p['M']}_frac_burst"] = round(tf / bf16, 4)
            res[f"prefill_m{p['M']}_frac_sustained"] = round(tf / bf16_sus, 4)
    res["per_linear_us"] = {p["name"].replace("decode7b_", ""): p["us"] for p in per_linear}
    res["headline_timing"] = {
        "regions": HEADLINE_REPS, "steps_per_region": args.steps, "reported": "median",
        "ms_per_step_min": round(sec_min / args.steps * 1e3, 5),
        "ms_per_step_max": round(sec_max / args.steps * 1e3, 5)}
    res["config"] = {
        "workload": "decode_7b M=1: qkv 4608x3584, o 3584x3584, gate_up 37888x3584, "
                    "down 3584x18944; int4 G=128 symmetric; bf16 activations",
        "M": 1, "bytes_per_step": int(sum(algorithmic_bytes(l, 1) for l in lins)),
        "l2": "rotating weight/activation copies (> 3x L2) so every step reads cold HBM",
        "timing": f"CUDA graphs of the w4a16_linear calls, CUDA events; median of "
                  f"{HEADLINE_REPS} timed regions of --steps steps, max over ranks",
        "parallelism": f"replicas x{world}",
    }
    res["gpu_launches"] = 4 * args.steps * HEADLINE_REPS
    res["clocks"] = clk.summary()
    res["roofline"] = roofline
    res["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(lins)
    res["per_linear"] = per_linear
    res.update(subs)
    return res


def run_sharded(args, world, rank):
    """The 7B decode step (M = 1) with every linear split over the `world`
    ranks: --shard n splits the output rows (no exchange), --shard k the
    input columns in group-aligned slices, with one NCCL all-reduce of the
    fp32 partials per linear.  Strong scaling: the job is one whole step per
    iteration, so `value` is the unsharded step's algorithmic bytes per
    second.  Eager launches (the all-reduce sits between the kernels),
    CUDA events, median of the timed regions, max over ranks."""
    import int4_weight_only_gb300 as w4
    from int4_weight_only_gb300 import build as b
    from int4_weight_only_gb300.shard import (column_parallel_linear, pack_shard,
                                              row_parallel_linear)
    b.build()
    w4.load()
    hbm, _, _, peak_kind = load_peaks()
    lins = WL.decode_7b(1)
    bytes_step = sum(algorithmic_bytes(l, 1) for l in lins)
    base = []
    for lin in lins:
        inp = WL.make_inputs(lin)
        sh = pack_shard(inp.W.cuda(), lin.group_size, True, args.shard, world, rank)
        base.append((lin, sh, inp.x.cuda()))
        torch.cuda.synchronize()
    shard_bytes = sum(sh.packed.numel() + 4 * sh.scales.numel() for _, sh, _ in base)
    R = max(2, math.ceil(3 * L2_BYTES / max(shard_bytes, 1)))
    copies = []
    for r in range(R):
        cp = []
        for lin, sh, x in base:
            c = type(sh)(**{**sh.__dict__, "packed": sh.packed.clone(), "scales": sh.scales.clone()})
            xl = x if args.shard == "n" else x[:, sh.lo:sh.hi].contiguous()
            y = torch.empty(1, lin.N if args.shard == "k" else sh.width, dtype=torch.bfloat16,
                            device="cuda")
            y32 = torch.empty(1, lin.N, dtype=torch.float32, device="cuda")
            cp.append((c, xl, y, y32))
        copies.append(cp)
    torch.cuda.synchronize()

    def step(i):
        for c, xl, y, y32 in copies[i % R]:
            if args.shard == "n":
                column_parallel_linear(xl, c, y=y)
            else:
                row_parallel_linear(xl, c, y=y, y32=y32)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    secs = []
    dev = torch.cuda.current_device()
    with ClockSampler(dev) as clk:
        for _ in range(HEADLINE_REPS):
            barrier(world)
            torch.cuda.synchronize()
            ev0.record()
            for i in range(args.steps):
                step(i)
            ev1.record()
            torch.cuda.synchronize()
            barrier(world)
            secs.append(ev0.elapsed_time(ev1) / 1e3)
    sec = max_over_ranks(statistics.median(secs), world)
    value = bytes_step * args.steps / sec / 1e9
    launches = 4 * args.steps * HEADLINE_REPS * (2 if args.shard == "k" else 1)
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec / args.steps * 1e3, 5), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian weights and activations, 7B decode shapes)",
        "config": {"workload": "decode_7b M=1, every linear sharded over the ranks",
                   "M": 1, "bytes_per_step": bytes_step,
                   "parallelism": (f"tp{world} column-parallel (output rows), no exchange"
                                   if args.shard == "n" else
                                   f"tp{world} row-parallel (group-aligned K slices), "
                                   f"one fp32 all-reduce per linear"),
                   "timing": f"eager launches, CUDA events, median of {HEADLINE_REPS} timed "
                             f"regions of --steps steps, max over ranks",
                   "l2": f"rotating {R} copies of each rank's shard (> 3x L2)"},
        "gpu_launches": launches, "clocks": clk.summary(),
        "roofline": {"kernel": "k_w4a16_gemv (shards)", "bound": "hbm",
                     "achieved": round(value / world, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(value / world / hbm, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "traffic": None},
    }


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle, as it stands, on the same workload and metric: each
    step runs the four decode linears at M=1 on a fixed row sample, sized so
    that warm-up plus timed steps take about two minutes."""
    lins = WL.decode_7b(1)
    total = args.steps + args.warmup
    probe = _oracle_row_sample(lins, 1 / 256, seed=3)
    t0 = time.perf_counter()
    _oracle_step(probe)
    t1 = max(time.perf_counter() - t0, 1e-4)
    frac = min(1 / 8, (1 / 256) * (120.0 / total) / t1)
    frac = max(frac, 1.0 / min(l.N for l in lins))
    sample = _oracle_row_sample(lins, frac, seed=5)
    for _ in range(args.warmup):
        _oracle_step(sample)
    t0 = time.perf_counter()
    by = 0.0
    for _ in range(args.steps):
        by += _oracle_step(sample)
    dt = time.perf_counter() - t0
    v = by / dt / 1e9
    desc = (f"oracle w4a16_linear (numpy fp64) on a fixed {frac:.5f} row sample of each of the "
            f"four 7B decode linears per step, M=1")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode_7b M=1: qkv 4608x3584, o 3584x3584, gate_up "
                                   "37888x3584, down 3584x18944; int4 G=128 symmetric "
                                   "(row sample per step)", "M": 1},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": blas_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_case(args):
    """A few calls of one named linear: the small command profilers run."""
    import int4_weight_only_gb300 as w4
    from int4_weight_only_gb300 import build as b
    b.build()
    if args.case.startswith("moe_"):
        # expert layer, --M = batch of tokens (8 experts each): grouped calls
        lin = next(l for l in WL.moe_decode(args.M) if l.name.startswith(args.case))
        E = WL.MOE_EXPERTS
        counts = WL.moe_route_counts(args.M, seed=args.M)
        goff = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
        goff[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32, device="cuda"), 0,
                                dtype=torch.int32)
        Kp = -(-lin.K // lin.group_size) * lin.group_size
        g = torch.Generator(device="cuda")
        g.manual_seed(lin.seed)
        p = torch.randint(0, 256, (E * lin.N, Kp // 2), generator=g, device="cuda",
                          dtype=torch.int32).to(torch.uint8)
        sc = torch.rand(E * lin.N, Kp // lin.group_size, generator=g, device="cuda") * 0.01 + 1e-4
        x = WL.make_activations(lin.K, sum(counts), seed=lin.seed).cuda()
        for _ in range(args.reps):
            w4.w4a16_grouped_linear(x, goff, p, sc, None, None, E, lin.N, lin.K, lin.group_size,
                                    max(counts))
        torch.cuda.synchronize()
        print(json.dumps({"case": lin.name, "batch": args.M, "reps": args.reps,
                          "device_error": w4.w4_get_device_error()}))
        return
    allw = (WL.tiny() + WL.decode_7b(args.M) + WL.decode_12b(args.M) + WL.prefill_7b(args.M)
            + WL.w4a8_7b())
    lin = next(l for l in allw if l.name.startswith(args.case))
    if args.G:                                 # e.g. the W4A8 linear with G = 128 scales
        lin = dataclasses.replace(lin, group_size=args.G)
    inp = WL.make_inputs(lin, args.M)
    p, sc, z = w4.w4_pack_rtn(inp.W.cuda(), lin.group_size, lin.symmetric)
    x = inp.x.cuda()
    bias = inp.bias.cuda() if inp.bias is not None else None
    for _ in range(args.reps):
        if lin.kind == "w4a8":
            qx, sx = w4.w4a8_quantize_act(x, lin.group_size)
            w4.w4a8_linear(qx, sx, p, sc, bias, lin.N, lin.K, lin.group_size)
        else:
            w4.w4a16_linear(x, p, sc, z, bias, lin.N, lin.K, lin.group_size)
    torch.cuda.synchronize()
    print(json.dumps({"case": lin.name, "M": args.M, "reps": args.reps,
                      "device_error": w4.w4_get_device_error()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode step (skip the other workloads)")
    ap.add_argument("--case", default=None,
                    help="run --reps calls of the workload linear whose name starts with this")
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--G", type=int, default=0, help="--case: override the group size")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--shard", choices=["n", "k"], default=None,
                    help="time the decode step with every linear split over the ranks: "
                         "n = output rows, k = group-aligned input columns + all-reduce")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker:
        cpu_worker()
        return
    if args.case:
        run_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    res = run_sharded(args, world, rank) if args.shard else run_ours(args, world, rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
