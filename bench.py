"""Benchmark of the forward FP8 MLP down-projection on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gpt2xl] [--rows M] [--no-extras]
                    [--profile [--mx | --group | --unfused]]

One step is one pass of the forward path over one batch: cast W [K,N] to
E4M3 (transposed operand), fused ReLU^2 + BF16 copy + E4M3 cast + amax of H
[M,K], FP8 GEMM Y = X_q W_q / (s_x s_w) -> BF16, and the two delayed-scale
history updates.  The default workload is the largest one, the GPT-2-XL
down-projection (M = 131072 tokens, K = 6400, N = 1600, margin 2.0, history
length 1), where the step is one kernel (fp8_downproj_fwd_ex).

Timing: W untimed warm-up steps, then exactly K steps; before each step a
256 MiB buffer is written and read back to flush L2 (outside the timed
events); each step (a CUDA graph of the step's launches) is timed on its
stream with CUDA events.  `value` is whole-job TFLOP/s (2 M N K per step and
GPU) over the mean step time, max over ranks.  `e2e` repeats the step
through the same public API with H and W copied in from pinned host memory
and Y copied back inside the timed region.  `extras` holds the other
workloads' steps (each with its dominant kernel's roofline), the per-step
delayed-scaling metrics of the GPT-2-small batch, the outlier workload's
zero-flush rates, the comparators (unfused three-pass quantize, cuBLAS BF16,
cuBLASLt FP8) and the path's other rows.

`--impl reference` times the CPU oracle (the plain C reference the tests check
against) on a bounded sample of rows of the same workload and reports it in the
same metric and unit.  `--rows M` runs the workload with M rows (a smaller
case for counter captures); `--profile` runs a few eager steps only, without
timing, for `ncu` (with `--mx` the MXFP8 path, with `--group` the 1x128 /
128x128 group-scaled path, with `--unfused` the two-launch path).

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from quantize_fp8_gemm_gb300 import workloads as WL  # noqa: E402

METRIC = "FP8 down-proj fwd TFLOP/s (fused quant+GEMM); quant kernel HBM GB/s"
UNIT = "TFLOP/s"
PROFILES = os.path.join(ROOT, "profiles")
L2_FLUSH_BYTES = 256 << 20
DEFAULT_WORKLOAD = "gpt2xl"


def flush_l2(buf: torch.Tensor) -> None:
    """Write, then read back, a buffer twice the size of L2: the next step
    starts with none of its inputs in L2 and no dirty lines left to write back."""
    buf.zero_()
    buf.sum()


# ----------------------------------------------------------------- helpers --
def fp8_peak(dev) -> dict:
    """Dense FP8 peak for the GEMM rooflines: the stricter (larger) of 2 x the
    measured BF16 burst (the nominal FP8:BF16 ratio) and a cuBLASLt E4M3 GEMM
    (torch._scaled_mm, BF16 out) at 8192^3 timed here as a burst."""
    peaks = measured_peaks()
    nominal = 2.0 * peaks["bf16_tflops"]
    meas = None
    try:
        n = 8192
        g = torch.Generator(device=dev).manual_seed(5)
        a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()  # column-major operand
        one = torch.ones((), device=dev)
        t = timed_b2b([lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)], 20)
        meas = 2.0 * n ** 3 / (t * 1e-3) / 1e12
        del a, b
    except (RuntimeError, TypeError, AttributeError) as e:  # no FP8 GEMM in this torch / cuBLASLt
        return {"tflops": nominal, "cublaslt_e4m3_8192_tflops": None,
                "source": f"{peaks['source']} bf16 burst x 2 (cuBLASLt E4M3 unavailable: {type(e).__name__})"}
    if meas > nominal:
        return {"tflops": meas, "cublaslt_e4m3_8192_tflops": meas,
                "source": "cuBLASLt E4M3 GEMM burst at 8192^3 (torch._scaled_mm), above 2 x the bf16 burst"}
    return {"tflops": nominal, "cublaslt_e4m3_8192_tflops": meas,
            "source": f"{peaks['source']} bf16 burst x 2 (nominal FP8:BF16 ratio), above cuBLASLt E4M3 at 8192^3"}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(local_ms: float, local_units: float, world: int):
    """Max step time over ranks and the units all ranks processed (weak scaling)."""
    if world == 1:
        return local_ms, local_units
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self) -> dict:
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s in sm if smax and s >= 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def file_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_key: str, source: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since the capture (profiles/<key>.txt: 'source_sha' and
    'dram_bytes_per_launch' lines)."""
    p = os.path.join(PROFILES, f"{kernel_key}.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha") != file_sha(source):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def workload(name: str, rows: int | None):
    w = WL.WORKLOADS[name]
    return w if not rows else dataclasses.replace(w, M=int(rows))


# -------------------------------------------------------------- reference --
def run_reference(args, world, rank):
    """The CPU oracle, timed on this host's cores on a bounded sample of rows."""
    if rank != 0:
        return
    import oracle as O
    w = workload(args.workload, args.rows)
    threads = O.default_threads()
    rows_per_step = max(1, min(args.ref_rows, w.M))
    h = WL.h_preact(dataclasses.replace(w, M=min(w.M, 4096)), 0)  # the rows a step samples from
    Wb = WL.w_down(w)
    sw = O.delayed_scale(O.amax(Wb, O.ACT_IDENTITY), w.margin, O.E4M3)
    wq = O.quant(Wb, O.ACT_IDENTITY, O.E4M3, sw, want_act=False, nthreads=threads)["q"]
    sx = O.delayed_scale(O.amax(h, O.ACT_RELU2), w.margin, O.E4M3)
    rng = np.random.default_rng(0)

    def one_step():
        r0 = int(rng.integers(0, h.shape[0] - rows_per_step + 1))
        hs = h[r0:r0 + rows_per_step]
        rq = O.quant(hs, O.ACT_RELU2, O.E4M3, sx, nthreads=threads)
        O.gemm_fwd(rq["q"], wq, sx, sw, nthreads=threads)

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / dt / 1e12
    sample = (f"{rows_per_step} random rows of H per step (fused quantize + double-precision GEMM "
              f"over those rows against all {w.N} columns); W cast once outside the timed steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy normals rounded to BF16)",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "act": "relu2",
                   "margin": w.margin, "l2": "sampled rows on the CPU"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, h_bits, w_bits, gemm_rows: int) -> dict:
    """The oracle on this host's cores, in the two parts the step has: the
    fused quantize of the full H (and the W cast), as GB/s of the 5 bytes per
    element the kernel moves; and the double-precision GEMM on a sample of rows,
    per row, with the full GEMM's time extrapolated from it.  value = the
    metric (TFLOP/s of the whole step) with that extrapolated time."""
    import oracle as O
    threads = O.default_threads()
    sw = O.delayed_scale(O.amax(w_bits, O.ACT_IDENTITY), w.margin, O.E4M3)
    sx = O.delayed_scale(O.amax(h_bits[:4096], O.ACT_RELU2), w.margin, O.E4M3)
    t0 = time.perf_counter()
    wq = O.quant(w_bits, O.ACT_IDENTITY, O.E4M3, sw, want_act=False, nthreads=threads)["q"]
    rq = O.quant(h_bits, O.ACT_RELU2, O.E4M3, sx, nthreads=threads)
    t_quant = time.perf_counter() - t0
    rows = np.arange(min(gemm_rows, w.M), dtype=np.int64)
    t0 = time.perf_counter()
    O.gemm_fwd(rq["q"], wq, sx, sw, rows=rows, nthreads=threads)
    t_rows = time.perf_counter() - t0
    del rq
    per_row = t_rows / rows.size
    t_gemm_full = per_row * w.M
    qbytes = 5.0 * w.M * w.K + 3.0 * w.K * w.N
    return {"value": 2.0 * w.M * w.N * w.K / (t_quant + t_gemm_full) / 1e12, "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "quant_gbs": qbytes / t_quant / 1e9, "quant_s": t_quant,
            "gemm_ms_per_row": per_row * 1e3, "gemm_full_extrapolated_s": t_gemm_full,
            "sample": (f"quantize of the full H [{w.M},{w.K}] and the W cast: {t_quant:.2f} s; double-precision "
                       f"GEMM of the first {rows.size} rows against all {w.N} columns: {t_rows:.2f} s, "
                       f"{per_row * 1e3:.2f} ms per row, the full {w.M}-row GEMM extrapolated to "
                       f"{t_gemm_full:.1f} s; value = 2MNK / (quantize + extrapolated GEMM)")}


# --------------------------------------------------------------------- ours --
def timed_b2b(fns, reps: int) -> float:
    """Average device ms per launch of `reps` back-to-back calls cycling through
    fns (each reading its own inputs): the calls are captured into one CUDA
    graph and a replay is timed between one pair of events, so the host's
    launch rate does not enter (tiny kernels).  Eager launches if capture fails."""
    for f in fns:
        f()
    torch.cuda.synchronize()

    def run():
        for i in range(reps):
            fns[i % len(fns)]()

    graph = None
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                run()
        torch.cuda.current_stream().wait_stream(side)
        graph.replay()
    except RuntimeError:
        graph = None
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    if graph is not None:
        graph.replay()
    else:
        run()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def timed_steps(run_step, flush, steps: int) -> np.ndarray:
    """Device ms of each of `steps` calls of run_step(i), L2 flushed before each."""
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush_l2(flush)
        pairs[i][0].record()
        run_step(i)
        pairs[i][1].record()
    torch.cuda.synchronize()
    return np.array([a.elapsed_time(b) for a, b in pairs])


def kernel_times(dp, H, Wt, w, dev, reps: int) -> dict:
    """Device ms per launch of the step's kernels.  Inputs rotate over copies
    that together exceed L2 (4 x H for the casts, 8 x X_q for the GEMM), so no
    launch finds its input in L2; outputs go to scratch buffers (the step's
    state is not touched)."""
    from quantize_fp8_gemm_gb300 import binding as B
    M, K, N = w.M, w.K, w.N
    Hs = list(H) + [torch.empty_like(H[0]).copy_(H[i % len(H)]) for i in range(4 - len(H))]
    act = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    xq = torch.empty(M, K, dtype=torch.uint8, device=dev)
    wtq = torch.empty(N, K, dtype=torch.uint8, device=dev)
    ax, aw = torch.zeros(1, device=dev), torch.zeros(1, device=dev)
    sat = torch.zeros(1, dtype=torch.int64, device=dev)
    sx, sw = dp.x.scale.clone(), dp.w.scale.clone()
    batches = [[B.quant_args(Wt, B.ACT_IDENTITY, B.E4M3, sw, q_t_out=wtq, amax_out=aw, flags=B.ACCUMULATE),
                B.quant_args(h, dp.act, B.E4M3, sx, act_out=act, q_out=xq, amax_out=ax, sat_count=sat,
                             flags=B.ACCUMULATE)] for h in Hs]
    out = {"quant": timed_b2b([lambda e=e: B.fp8_quant_fused_batch(e) for e in batches], reps)}
    out["quant_h_only"] = timed_b2b([lambda h=h: B.fp8_quant_fused_ex(
        h, dp.act, B.E4M3, sx, act_out=act, q_out=xq, amax_out=ax, sat_count=sat, flags=B.ACCUMULATE)
        for h in Hs], reps)
    out["w_cast"] = timed_b2b([lambda: B.fp8_quant_fused_ex(Wt, B.ACT_IDENTITY, B.E4M3, sw, q_t_out=wtq,
                                                            amax_out=aw, flags=B.ACCUMULATE)], reps)
    del act
    nx = max(2, min(8, -(-(256 << 20) // (M * K))))
    xqs = [torch.empty_like(dp.x_q).copy_(dp.x_q) for _ in range(nx)]
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    out["gemm"] = timed_b2b([lambda x=x: B.fp8_gemm_fwd(x, dp.wt_q, sx, sw, y) for x in xqs], reps)
    del xqs
    if dp.fused:
        # the one-launch step kernel (W cast + quantize + GEMM), on its own scratch
        ws = torch.zeros(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device=dev)
        xq1 = torch.empty(M, K, dtype=torch.uint8, device=dev)
        act1 = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        out["fused_step_kernel"] = timed_b2b([lambda h=h: B.fp8_downproj_fwd_ex(
            h, wtq, sx, sw, xq1, y, ws, w=Wt, amax_w=aw, act=dp.act, act_out=act1, amax_out=ax, sat_count=sat,
            flags=B.ACCUMULATE) for h in Hs], reps)
        del ws, xq1, act1
    del Hs
    hist = torch.zeros_like(dp.x.history)
    head = torch.zeros(1, dtype=torch.int32, device=dev)
    scl = torch.ones(1, device=dev)
    out["history (one tensor)"] = timed_b2b([lambda: B.amax_history_update(hist, head, ax, w.margin, B.E4M3, scl)],
                                            reps)
    return out


def rooflines(w, kern_ms: dict, peaks: dict, fp8: dict, workload_key: str, step_ms=None) -> dict:
    """The rooflines of a per-tensor step's kernels: the one-launch cast (HBM),
    the FP8 GEMM (tensor) and, where the step runs it, the one-launch step
    kernel, which is bound by both: its roofline time is the larger of its
    algorithmic bytes over the HBM peak and its FLOPs over the FP8 peak.
    step_ms: the timed steps' mean event time when each step is that one
    launch; its duration is then taken over the timed region (the
    back-to-back figure is kept beside it as b2b_ms)."""
    M, K, N = w.M, w.K, w.N
    flops = 2.0 * M * N * K
    quant_bytes = 5.0 * M * K + 3.0 * K * N  # H in, BF16 act + E4M3 out; W in, W_q^T out
    quant_gbs = quant_bytes / (kern_ms["quant"] * 1e-3) / 1e9
    gemm_tflops = flops / (kern_ms["gemm"] * 1e-3) / 1e12
    quant_src = os.path.join(ROOT, "quantize_fp8_gemm_gb300", "csrc", "quant.cu")
    gemm_src = os.path.join(ROOT, "quantize_fp8_gemm_gb300", "csrc", "gemm.cu")
    out = {
        "quant": {"bound": "hbm", "kernel": "quant_batch_kernel (fp8_quant_fused_batch: W cast + H quantize)",
                  "achieved": quant_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                  "frac": quant_gbs / peaks["hbm_gbs"],
                  "traffic": profiled_traffic(f"quant_batch_{workload_key}", quant_src),
                  "algorithmic_bytes": quant_bytes, "peak_source": peaks["source"] + " (burst copy)"},
        "gemm": {"bound": "tensor", "kernel": "fp8_gemm_kernel (fp8_gemm_fwd)", "achieved": gemm_tflops,
                 "peak": fp8["tflops"], "unit": "TFLOP/s", "frac": gemm_tflops / fp8["tflops"],
                 "traffic": profiled_traffic(f"fp8_gemm_{workload_key}", gemm_src),
                 "algorithmic_flops": flops, "peak_source": fp8["source"]},
    }
    out["dominant"] = out["quant"] if kern_ms["quant"] >= kern_ms["gemm"] else out["gemm"]
    if "fused_step_kernel" in kern_ms:
        t = (step_ms if step_ms is not None else kern_ms["fused_step_kernel"]) * 1e-3
        fbytes = quant_bytes + 2.0 * M * N  # + Y
        t_hbm = fbytes / (peaks["hbm_gbs"] * 1e9)
        t_mma = flops / (fp8["tflops"] * 1e12)
        hbm_bound = t_hbm >= t_mma
        f = {"bound": "hbm" if hbm_bound else "tensor",
             "kernel": "fp8_gemm_kernel<FUSED> (fp8_downproj_fwd_ex: the one-launch step)",
             "achieved": fbytes / t / 1e9 if hbm_bound else flops / t / 1e12,
             "peak": peaks["hbm_gbs"] if hbm_bound else fp8["tflops"],
             "unit": "GB/s" if hbm_bound else "TFLOP/s", "frac": max(t_hbm, t_mma) / t,
             "traffic": profiled_traffic(f"fp8_fused_{workload_key}", gemm_src),
             "algorithmic_bytes": fbytes, "algorithmic_flops": flops,
             "hbm_gbs": fbytes / t / 1e9, "hbm_frac": t_hbm / t,
             "tensor_tflops": flops / t / 1e12, "tensor_frac": t_mma / t,
             "roofline_ms": max(t_hbm, t_mma) * 1e3,
             "duration_ms": t * 1e3,
             "duration_source": ("the timed steps (one launch per step; CUDA events around each step's "
                                 "graph replay on the launching stream)" if step_ms is not None else
                                 "back-to-back launches over input copies larger than L2"),
             "b2b_ms": kern_ms["fused_step_kernel"],
             "peak_source": f"HBM: {peaks['source']} copy; FP8: {fp8['source']}"}
        out["fused"] = f
        out["dominant"] = f
    return out


def measure_step(w, dev, steps: int, warmup: int, flush, eager: bool = False, group: bool = False):
    """Build the step's state for workload w, calibrate, capture the step as CUDA
    graphs, run `warmup` untimed steps and time `steps` steps (L2 flushed before
    each).  Returns the state, the inputs, the per-step ms, the timing mode and
    the wall time of the timed loop."""
    from quantize_fp8_gemm_gb300.downproj import Fp8DownProj
    h_bits = [WL.h_preact(w, s) for s in range(2)]
    w_bits = WL.w_down(w)
    H = [WL.bf16_tensor(b).to(dev) for b in h_bits]
    Wt = WL.bf16_tensor(w_bits).to(dev)
    dp = Fp8DownProj(w.M, w.K, w.N, margin=w.margin, history_len=w.history_len, group=group, device=dev)
    dp.calibrate(H[0], Wt)
    for i in range(warmup):
        flush_l2(flush)
        dp.step(H[i % 2], Wt)
    torch.cuda.synchronize()
    graphs, mode = None, "eager"
    if not eager:
        try:
            graphs = dp.capture(H[0], Wt, H_next=H[1])  # replays alternate H[0] / H[1]
            mode = "cuda-graph"
        except RuntimeError as exc:  # capture refused
            mode = f"eager (graph capture unavailable: {exc})"[:200]

    def run_step(i):
        if graphs is not None:
            graphs.replay()
        else:
            dp.step(H[i % 2], Wt)

    for i in range(warmup):
        flush_l2(flush)
        run_step(i)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    step_ms = timed_steps(run_step, flush, steps)
    wall = time.perf_counter() - wall0
    st = int(dp.gemm_status.item())
    if st != 0:
        raise RuntimeError(f"GEMM reported device status {st} on {w.name}")
    return dict(dp=dp, H=H, Wt=Wt, h_bits=h_bits, w_bits=w_bits, step_ms=step_ms, mode=mode, wall=wall,
                graphs=graphs)


def step_desc(dp) -> tuple[str, int]:
    if dp.fused:
        return "W cast, quantize of H, FP8 GEMM and the 2 history updates in one kernel", 1
    if dp.group:
        return ("128x128 block cast of W, 1x128 group quantize of H, group-scaled FP8 GEMM "
                "(no delayed scales to update)"), 3
    if dp.chunks == 1:
        return "W cast + quantize of H in one launch, then the FP8 GEMM, which also runs the 2 history updates", 2
    return f"W cast, {dp.chunks} x (row-block quantize + its GEMM), 2 history updates", 3 + 2 * dp.chunks


def run_profile(args, local):
    """A few eager steps of the workload, nothing timed: the command ncu wraps.
    With --rows the step takes the path and the GEMM tile the full-size
    workload takes (the one-launch kernel, or with --unfused or below the
    one-launch size the two-launch cast + GEMM), so a smaller capture shows
    the same kernels."""
    from quantize_fp8_gemm_gb300.downproj import FUSED_MIN_ROWS, Fp8DownProj
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload(args.workload, args.rows)
    H = WL.bf16_tensor(WL.h_preact(w, 0)).to(dev)
    Wt = WL.bf16_tensor(WL.w_down(w)).to(dev)
    full = WL.WORKLOADS[args.workload]
    if args.mx:
        return run_profile_mx(args, w, H, Wt, dev)
    fused = full.M >= FUSED_MIN_ROWS and not args.unfused and not args.group
    if w.M != full.M:
        # the full size's tile too (the tile choice depends on M)
        from quantize_fp8_gemm_gb300 import binding as B
        B.fp8q_gemm_set_tile(*B.fp8q_test_gemm_tile(full.M, full.N, fused))
    dp = Fp8DownProj(w.M, w.K, w.N, margin=w.margin, history_len=w.history_len, fused=fused, group=args.group,
                     device=dev)
    dp.calibrate(H, Wt)
    for _ in range(max(1, args.steps)):
        dp.step(H, Wt)
    torch.cuda.synchronize()
    st = int(dp.gemm_status.item())
    print(json.dumps({"profile": w.name, "M": w.M, "K": w.K, "N": w.N, "fused": dp.fused, "steps": args.steps,
                      "status": st}), flush=True)
    if w.M != full.M:
        B.fp8q_gemm_set_tile(-1)
    if st != 0:
        raise SystemExit(1)


def run_profile_mx(args, w, H, Wt, dev):
    """--profile --mx: the MXFP8 path on the workload, nothing timed: the
    activation's block quantize, the weight's transposed block cast and the
    block-scaled GEMM, --steps times."""
    from quantize_fp8_gemm_gb300 import binding as B
    M, K, N = w.M, w.K, w.N
    q = torch.empty(M, K, dtype=torch.uint8, device=dev)
    sf = torch.empty(B.fp8_mx_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    qt = torch.empty(N, K, dtype=torch.uint8, device=dev)
    sft = torch.empty(B.fp8_mx_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(max(1, args.steps)):
        B.fp8_quant_mx(H, B.ACT_RELU2, B.E4M3, q_out=q, sf_out=sf)
        B.fp8_quant_mx(Wt, B.ACT_IDENTITY, B.E4M3, q_t_out=qt, sf_t_out=sft)
        B.fp8_gemm_mx(q, sf, qt, sft, y, status=st)
    torch.cuda.synchronize()
    print(json.dumps({"profile": w.name + " (MXFP8)", "M": M, "K": K, "N": N, "steps": args.steps,
                      "status": int(st.item())}), flush=True)
    if st.item() != 0:
        raise SystemExit(1)


def run_ours(args, world, rank, local):
    from quantize_fp8_gemm_gb300 import binding as B  # noqa: F401  (fails loudly without the library)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload(args.workload, args.rows)
    M, K, N = w.M, w.K, w.N
    peaks = measured_peaks()
    fp8 = fp8_peak(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    barrier(world)
    torch.cuda.synchronize()
    # clocks sampled while the steps and then the kernel rooflines run (the
    # latter keep the GPU loaded for a few seconds, so the samples see it busy)
    with ClockSampler(local) as clk:
        r = measure_step(w, dev, args.steps, args.warmup, flush, eager=args.eager)
        barrier(world)
        dp, H, Wt = r["dp"], r["H"], r["Wt"]
        kern_ms = kernel_times(dp, H, Wt, w, dev, reps=max(24, min(args.steps, 400)))
    clocks = clk.summary()
    local_ms = float(r["step_ms"].mean())
    flops_step = 2.0 * M * N * K
    ms, total_flops = reduce_over_ranks(local_ms, flops_step, world)
    value = total_flops / (ms * 1e-3) / 1e12
    kern_ms["step"] = local_ms
    desc, launches_per_step = step_desc(dp)
    roof = rooflines(w, kern_ms, peaks, fp8, w.name if not args.rows else f"{w.name}_m{w.M}",
                     step_ms=local_ms if launches_per_step == 1 and r["graphs"] is not None else None)

    extras = {}
    if not args.no_extras:
        extras = measure_extras(args, dp, H, Wt, flush, kern_ms, w, dev, fp8, peaks)

    e2e = measure_e2e(args, dp, r["h_bits"], r["w_bits"], flush, w, dev, use_graph=r["graphs"] is not None)
    wall, mode = r["wall"], r["mode"]
    del r
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        h0 = WL.h_preact(w, 0)
        cpu = cpu_baseline(w, h0, WL.w_down(w), args.cpu_rows)
        del h0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32 accumulate -> bf16",
        "data": "synthetic (seeded numpy normals rounded to BF16, uploaded before timing)",
        "config": {"workload": w.name, "M": M, "K": K, "N": N, "act": "relu2",
                   "scaling": "per-tensor delayed", "margin": w.margin, "history": w.history_len,
                   "l2": "flushed before every step (256 MiB write + read, untimed)",
                   "step": desc},
        "kernel_ms": kern_ms,
        "quant_hbm_gbs": roof["quant"]["achieved"],
        "gemm_tflops": roof["gemm"]["achieved"],
        "roofline": roof["dominant"],
        "roofline_quant": roof["quant"],
        "roofline_gemm": roof["gemm"],
        "roofline_fused": roof.get("fused"),
        "fp8_peak": fp8,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "kernel_ms_note": ("each kernel as back-to-back launches over input copies larger than L2, "
                           "captured in one CUDA graph (average device time per launch, one event pair)"),
        "timing": f"{mode}: one event pair around each step on the launching stream",
        "clocks": clocks,
        "wall_s_timed_loop": wall,
        "extras": extras,
    }
    print(json.dumps(line), flush=True)


def measure_other_config(name: str, dev, flush, fp8: dict, peaks: dict, steps: int, group: bool = False) -> dict:
    """One of the smaller workloads' steps, timed like the headline (CUDA-graph
    replays, L2 flushed before each), with its kernels' rooflines."""
    from quantize_fp8_gemm_gb300 import binding as B
    w = WL.WORKLOADS[name]
    r = measure_step(w, dev, steps, 3, flush, group=group)
    dp = r["dp"]
    ms = float(r["step_ms"].mean())
    flops = 2.0 * w.M * w.N * w.K
    desc, launches = step_desc(dp)
    row = {"shape": f"H [{w.M},{w.K}] x W [{w.K},{w.N}]", "step": desc, "launches_per_step": launches,
           "step_ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12, "timing": r["mode"]}
    reps = max(24, min(steps, 200))
    if not group:
        km = kernel_times(dp, r["H"], r["Wt"], w, dev, reps)
        roof = rooflines(w, km, peaks, fp8, name,
                         step_ms=ms if launches == 1 and r["graphs"] is not None else None)
        row["kernel_ms"] = km
        row["roofline"] = roof["dominant"]
        row["roofline_quant"] = roof["quant"]
        row["roofline_gemm"] = roof["gemm"]
        if "fused" in roof:
            row["roofline_fused"] = roof["fused"]
    else:
        M, K, N = w.M, w.K, w.N
        Hs = r["H"] + [r["H"][0].clone(), r["H"][1].clone()]
        act = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        amax = torch.zeros(1, device=dev)
        t_q = timed_b2b([lambda h=h: B.fp8_quant_fused_ex(h, dp.act, B.E4M3, None, act_out=act, q_out=dp.x_q,
                                                          amax_out=amax, group_scales_out=dp.x_gscale,
                                                          group_rows=1, flags=B.ACCUMULATE) for h in Hs], reps)
        xqs = [dp.x_q.clone() for _ in range(4)]
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        t_g = timed_b2b([lambda x=x: B.fp8_gemm_fwd(x, dp.wt_q, dp.x_gscale, dp.w_gscale, y, group_mode=1)
                         for x in xqs], reps)
        qb = 5.0 * M * K + 4.0 * M * (K // 128)
        row["kernel_ms"] = {"group_quant": t_q, "group_gemm": t_g}
        rq = {"bound": "hbm", "kernel": "quant_stream_kernel<GROUP> (1x128)", "achieved": qb / (t_q * 1e-3) / 1e9,
              "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": qb / (t_q * 1e-3) / 1e9 / peaks["hbm_gbs"],
              "algorithmic_bytes": qb}
        tf = flops / (t_g * 1e-3) / 1e12
        rg = {"bound": "tensor", "kernel": "fp8_gemm_kernel<GROUP>", "achieved": tf, "peak": fp8["tflops"],
              "unit": "TFLOP/s", "frac": tf / fp8["tflops"], "algorithmic_flops": flops}
        row["roofline_quant"], row["roofline_gemm"] = rq, rg
        row["roofline"] = rq if t_q >= t_g else rg
        del Hs, act, xqs, y
    del r, dp
    torch.cuda.empty_cache()
    return row


def drift_metrics(dev, max_steps: int) -> dict:
    """The GPT-2-small batch's delayed-scaling record: per step, the scale the
    step used, its amax and its saturation count, over the workload's 20 steps
    of drifting H (fresh seeded draws each step)."""
    from quantize_fp8_gemm_gb300.downproj import Fp8DownProj
    w = WL.WORKLOADS["gpt2s_batch"]
    Wt = WL.bf16_tensor(WL.w_down(w)).to(dev)
    dp = Fp8DownProj(w.M, w.K, w.N, margin=w.margin, history_len=w.history_len, keep_act=False, device=dev)
    H = WL.bf16_tensor(WL.h_preact(w, 0, WL.drift_std(w, 0))).to(dev)
    dp.calibrate(H, Wt)
    rec = {"step": [], "std": [], "scale_x": [], "amax_x": [], "saturated_x": [], "scale_w": [], "amax_w": [],
           "saturated_w": []}
    for t in range(min(w.steps, max_steps)):
        std = WL.drift_std(w, t)
        H.copy_(WL.bf16_tensor(WL.h_preact(w, t, std)))
        sx, sw = float(dp.x.scale.item()), float(dp.w.scale.item())
        dp.step(H, Wt)
        torch.cuda.synchronize()
        rec["step"].append(t)
        rec["std"].append(std)
        rec["scale_x"].append(sx)
        rec["scale_w"].append(sw)
        rec["amax_x"].append(float(dp.x.last_amax.item()))
        rec["amax_w"].append(float(dp.w.last_amax.item()))
        rec["saturated_x"].append(int(dp.x.last_sat.item()))
        rec["saturated_w"].append(int(dp.w.last_sat.item()))
    rec["step_path"] = step_desc(dp)[0]
    del dp, H, Wt
    torch.cuda.empty_cache()
    return rec


def outlier_flush_rates(dev) -> dict:
    """The outlier workload's zero flush: the share of non-zero BF16 inputs to
    the cast (the activation) whose E4M3 code is +-0, with one per-tensor scale
    (the current amax, margin 1) against 1x128 group scales, for ReLU^2 and the
    identity (whose +-1e5 entries keep their signs)."""
    from quantize_fp8_gemm_gb300 import binding as B
    w = WL.WORKLOADS["outlier"]
    M, K = w.M, w.K
    H = WL.bf16_tensor(WL.h_preact(w)).to(dev)
    act = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    q = torch.empty(M, K, dtype=torch.uint8, device=dev)
    amax = torch.zeros(1, device=dev)
    gs = torch.empty(M, K // 128, device=dev)
    out = {}
    for name, a in (("relu2", B.ACT_RELU2), ("identity", B.ACT_IDENTITY)):
        one = torch.ones(1, device=dev)
        B.fp8_quant_fused(H, a, B.E4M3, one, act_out=act, amax_out=amax)  # amax pass
        scale = (448.0 / amax).to(torch.float32)  # the current amax, margin 1 (the pages' experiment)
        nz = (act.view(torch.int16) & 0x7FFF) != 0
        n_nz = int(nz.sum().item())
        B.fp8_quant_fused(H, a, B.E4M3, scale, q_out=q)
        pt = int((nz & ((q & 0x7F) == 0)).sum().item()) / n_nz
        B.fp8_quant_fused(H, a, B.E4M3, None, q_out=q, group_scales_out=gs, group_rows=1)
        gr = int((nz & ((q & 0x7F) == 0)).sum().item()) / n_nz
        out[name] = {"per_tensor_scale": float(scale.item()), "flushed_per_tensor": pt, "flushed_1x128": gr,
                     "nonzero_inputs": n_nz}
    del H, act, q, gs
    torch.cuda.empty_cache()
    return out


def measure_extras(args, dp, H, Wt, flush, kern_ms, w, dev, fp8: dict, peaks: dict) -> dict:
    """Comparators at the headline workload, timed like kern_ms (back-to-back
    over 4 rotating copies of H): the unfused three-pass quantize (write the
    activation, an amax pass, a cast pass) against the fused quantize of H
    alone, cuBLAS BF16 on the BF16 activation against the FP8 GEMM, and the
    BF16 path against the FP8 step; then the other workloads and rows."""
    from quantize_fp8_gemm_gb300 import binding as B
    M, K, N = w.M, w.K, w.N
    reps = max(24, min(400, args.steps))
    Hs = list(H) + [torch.empty_like(H[0]).copy_(H[i % len(H)]) for i in range(4 - len(H))]
    a_naive = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    q_naive = torch.empty(M, K, dtype=torch.uint8, device=dev)
    amax = torch.zeros(1, device=dev)

    def naive(h):
        B.fp8q_naive_act(h, B.ACT_RELU2, a_naive)
        B.fp8q_naive_amax(a_naive, amax)
        B.fp8q_naive_cast(a_naive, B.E4M3, amax, w.margin, q_naive)

    t_naive = timed_b2b([lambda h=h: naive(h) for h in Hs], reps)
    del q_naive
    acts = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    for h, act in zip(Hs, acts):
        B.fp8q_naive_act(h, B.ACT_RELU2, act)
    y16 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    t_bf16_gemm = timed_b2b([lambda a=a: torch.matmul(a, Wt, out=y16) for a in acts], reps)
    t_bf16_path = timed_b2b([lambda h=h: (B.fp8q_naive_act(h, B.ACT_RELU2, a_naive),
                                          torch.matmul(a_naive, Wt, out=y16)) for h in Hs], reps)
    del acts, Hs, a_naive
    # the library's FP8 GEMM (cuBLASLt E4M3 x E4M3 -> BF16 via torch._scaled_mm) on the same
    # operands, over rotating copies of X_q like the FP8 GEMM's own timing
    t_lib_fp8 = None
    try:
        xqs = [dp.x_q.clone().view(torch.float8_e4m3fn) for _ in range(2)]
        wtq = dp.wt_q.view(torch.float8_e4m3fn).t()  # [K,N], column-major
        s_x, s_w = (1.0 / dp.x.scale).reshape(()), (1.0 / dp.w.scale).reshape(())  # dequantisation factors
        t_lib_fp8 = timed_b2b([lambda x=x: torch._scaled_mm(x, wtq, scale_a=s_x, scale_b=s_w,
                                                            out_dtype=torch.bfloat16) for x in xqs], reps)
        del xqs
    except (RuntimeError, TypeError, AttributeError):
        pass
    torch.cuda.empty_cache()
    t_fused = kern_ms["quant_h_only"]
    t_fp8_step = kern_ms.get("fused_step_kernel", kern_ms["quant"] + kern_ms["gemm"])
    flops = 2.0 * M * N * K
    out = {
        "naive_3pass_ms": t_naive, "fused_quant_ms": t_fused,
        "fused_vs_naive_speedup": t_naive / t_fused, "fused_vs_naive_ideal": 9.0 / 5.0,
        "bf16_gemm_ms": t_bf16_gemm, "bf16_gemm_tflops": flops / (t_bf16_gemm * 1e-3) / 1e12,
        "fp8_vs_bf16_gemm_speedup": t_bf16_gemm / kern_ms["gemm"],
        "cublaslt_fp8_gemm_ms": t_lib_fp8,
        "cublaslt_fp8_gemm_tflops": flops / (t_lib_fp8 * 1e-3) / 1e12 if t_lib_fp8 else None,
        "fp8_gemm_vs_cublaslt_fp8_speedup": t_lib_fp8 / kern_ms["gemm"] if t_lib_fp8 else None,
        "bf16_path_ms (BF16 activation write + cuBLAS BF16 GEMM)": t_bf16_path,
        "fp8_path_ms (the FP8 step's kernels)": t_fp8_step,
        "fp8_vs_bf16_end_to_end_speedup": t_bf16_path / t_fp8_step,
        "fp8_unfused_path_ms (one-launch W + H cast, then the FP8 GEMM)": kern_ms["quant"] + kern_ms["gemm"],
        "timing": "back-to-back launches over rotating input copies (> L2) in one CUDA graph, one event pair",
        "workload": w.name,
    }
    out["fused_layouts"] = measure_fused_layouts(dp, H, Wt, w, dev, 10)
    cfg_steps = max(20, min(100, args.steps))
    out["configs"] = {}
    for name in ("gpt2s", "gpt2s_batch", "outlier"):
        if name != w.name:
            out["configs"][name] = measure_other_config(name, dev, flush, fp8, peaks, cfg_steps)
    out["configs"]["outlier (1x128 / 128x128 group scales)"] = measure_other_config(
        "outlier", dev, flush, fp8, peaks, cfg_steps, group=True)
    out["gpt2s_batch_delayed_scaling_per_step"] = drift_metrics(dev, 20)
    out["outlier_zero_flush"] = outlier_flush_rates(dev)
    out["other_rows"] = measure_other_rows(dev, max(16, min(64, args.steps)), fp8["tflops"])
    return out


def measure_fused_layouts(dp, H, Wt, w, dev, reps: int) -> dict:
    """The one-launch step kernel with each layout of its quantize warps pinned
    (1: quantize-first, 24 warps; 2: GEMM-first, 9 working warps off the MMA
    issuer's scheduler), timed like the rooflines' kernels: back-to-back
    launches over copies of H that together exceed L2."""
    from quantize_fp8_gemm_gb300 import binding as B
    if not dp.fused:
        return {}
    M, K, N = w.M, w.K, w.N
    Hs = list(H) + [torch.empty_like(H[0]).copy_(H[i % len(H)]) for i in range(4 - len(H))]
    ws = torch.zeros(B.fp8_downproj_workspace_bytes(M), dtype=torch.uint8, device=dev)
    xq = torch.empty(M, K, dtype=torch.uint8, device=dev)
    act = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    wtq = torch.empty(N, K, dtype=torch.uint8, device=dev)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ax, aw = torch.zeros(1, device=dev), torch.zeros(1, device=dev)
    sx, sw = dp.x.scale.clone(), dp.w.scale.clone()
    out = {}
    try:
        for layout, name in ((1, "quantize-first"), (2, "GEMM-first")):
            B.fp8q_test_set_fused_layout(layout)
            out[name + " ms"] = timed_b2b([lambda h=h: B.fp8_downproj_fwd_ex(
                h, wtq, sx, sw, xq, y, ws, w=Wt, amax_w=aw, act=dp.act, act_out=act, amax_out=ax,
                flags=B.ACCUMULATE) for h in Hs], reps)
    finally:
        B.fp8q_test_set_fused_layout(0)
    out["default"] = "GEMM-first" if 2.0 * N * 6.45e12 > 5.0 * 3.7e15 else "quantize-first"
    del Hs, ws, xq, act, wtq, y
    torch.cuda.empty_cache()
    return out

def measure_other_rows(dev, reps: int, fp8_tflops: float) -> dict:
    """The path's other rows, each on the workload it belongs to and timed like
    the step's kernels (back-to-back launches captured in one CUDA graph, the
    inputs larger than L2 or rotated over copies that together exceed it):
    the weight cast in both layouts, the E5M2 gradient cast (row-major and
    transposed), the dgrad GEMM dX = dY W^T and the weight-gradient GEMM
    dW = X^T dY on the GPT-2-XL shapes, the 1x128 group quantize and the
    group-scaled GEMM on the outlier shapes.  Each row carries its roofline
    fraction of the measured peaks."""
    from quantize_fp8_gemm_gb300 import binding as B
    peaks = measured_peaks()
    hbm, fp8 = peaks["hbm_gbs"], fp8_tflops
    l2_bytes = 256 << 20  # rotate copies until the inputs exceed L2 twice over

    def copies(t):
        n = max(1, -(-l2_bytes // (t.numel() * t.element_size())))
        return [t] + [t.clone() for _ in range(n - 1)]

    def mem_row(ms, nbytes, shape):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"shape": shape, "ms": ms, "GB/s": gbs, "bound": "hbm", "frac": gbs / hbm,
                "algorithmic_bytes": nbytes}

    def mma_row(ms, flops, shape):
        tf = flops / (ms * 1e-3) / 1e12
        return {"shape": shape, "ms": ms, "TFLOP/s": tf, "bound": "tensor", "frac": tf / fp8,
                "algorithmic_flops": flops}

    out = {}
    amax = torch.zeros(1, device=dev)
    one = torch.ones(1, device=dev)
    xl = WL.WORKLOADS["gpt2xl"]
    M, K, N = xl.M, xl.K, xl.N
    W = WL.bf16_tensor(WL.w_down(xl)).to(dev)  # [K,N]
    w_q = torch.empty(K, N, dtype=torch.uint8, device=dev)   # dgrad operand
    wt_q = torch.empty(N, K, dtype=torch.uint8, device=dev)  # forward operand
    Ws = copies(W)
    t = timed_b2b([lambda x=x: B.fp8_quant_fused_ex(x, B.ACT_IDENTITY, B.E4M3, one, q_out=w_q, q_t_out=wt_q,
                                                    amax_out=amax, flags=B.ACCUMULATE) for x in Ws], reps)
    out["a7 weight cast, both layouts"] = mem_row(t, 4.0 * K * N, f"W [{K},{N}]")
    del Ws
    dY = WL.bf16_tensor(WL.dy_grad(xl)).to(dev)
    dyq = torch.empty(M, N, dtype=torch.uint8, device=dev)
    sdy = torch.full((1,), 4096.0, device=dev)  # 57344 / (margin * ~7): the spikes stay below the E5M2 max
    t = timed_b2b([lambda: B.fp8_quant_fused_ex(dY, B.ACT_IDENTITY, B.E5M2, sdy, q_out=dyq, amax_out=amax,
                                                flags=B.ACCUMULATE)], max(4, reps // 4))
    out["a10 dY cast E5M2"] = mem_row(t, 3.0 * M * N, f"dY [{M},{N}]")
    # the weight gradient's operand: dY's transposed E5M2 copy (token-contiguous)
    dyqt = torch.empty(N, M, dtype=torch.uint8, device=dev)
    t = timed_b2b([lambda: B.fp8_quant_fused_ex(dY, B.ACT_IDENTITY, B.E5M2, sdy, q_t_out=dyqt, amax_out=amax,
                                                flags=B.ACCUMULATE)], max(4, reps // 4))
    out["next: dY cast E5M2, transposed copy"] = mem_row(t, 3.0 * M * N, f"dY [{M},{N}] -> dY_q^T [{N},{M}]")
    del dY, W
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    t = timed_b2b([lambda: B.fp8_gemm_dgrad(dyq, w_q, sdy, one, dx)], max(4, reps // 8))
    out["a11 dgrad GEMM"] = mma_row(t, 2.0 * M * N * K, f"dY_q [{M},{N}] x W_q [{K},{N}]^T")
    # next: the ReLU^2 backward in the dgrad epilogue, dH = dX * 2 max(H, 0) (H read, dX never stored)
    g = torch.Generator(device=dev).manual_seed(xl.seed)
    Hb = torch.randn(M, K, device=dev, generator=g).to(torch.bfloat16)
    t = timed_b2b([lambda: B.fp8_gemm_dgrad_act(dyq, w_q, sdy, one, Hb, dx, act=B.ACT_RELU2)], max(4, reps // 8))
    row = mma_row(t, 2.0 * M * N * K, f"dY_q [{M},{N}] x W_q [{K},{N}]^T, H [{M},{K}] -> dH")
    row["vs_dgrad_alone"] = out["a11 dgrad GEMM"]["ms"] / t
    # the unfused pair it replaces: the dgrad writing dX, then dH = dX * 2 relu(H) elementwise (torch)
    dh, tmp = torch.empty_like(dx), torch.empty_like(dx)

    def unfused():
        B.fp8_gemm_dgrad(dyq, w_q, sdy, one, dx)
        torch.clamp(Hb, min=0, out=tmp)
        tmp.mul_(2.0)
        torch.mul(dx, tmp, out=dh)

    t2 = timed_b2b([unfused], max(4, reps // 8))
    row["unfused_ms (dgrad writing dX, then dH = dX * 2 relu(H) elementwise)"] = t2
    row["speedup_vs_unfused"] = t2 / t
    out["next: dgrad with the ReLU^2 backward epilogue"] = row
    # the same with H read from its E4M3 cache (1 byte per element instead of 2)
    hq = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device=dev, generator=g)
    s_h = torch.full((1,), 38.0, device=dev)
    t3 = timed_b2b([lambda: B.fp8_gemm_dgrad_act_q(dyq, w_q, sdy, one, hq, s_h, dh, act=B.ACT_RELU2)],
                   max(4, reps // 8))
    row = mma_row(t3, 2.0 * M * N * K, f"dY_q [{M},{N}] x W_q [{K},{N}]^T, H's E4M3 cache [{M},{K}] -> dH")
    row["vs_bf16_h"] = t / t3
    out["next: dgrad with the ReLU^2 backward epilogue, H from its FP8 cache"] = row
    del Hb, dx, dh, tmp, dyq, w_q, wt_q, hq
    # wgrad dW = X^T dY: X_q^T [K,M] (E4M3 codes; the GEMM's time does not depend on their values)
    g = torch.Generator(device=dev).manual_seed(xl.seed)
    xqt = torch.randint(0, 120, (K, M), dtype=torch.uint8, device=dev, generator=g)
    dw = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
    t = timed_b2b([lambda: B.fp8_gemm_wgrad(xqt, dyqt, one, sdy, dw)], max(4, reps // 8))
    out["next: wgrad GEMM"] = mma_row(t, 2.0 * M * N * K, f"X_q^T [{K},{M}] x dY_q^T [{N},{M}]^T")
    del xqt, dyqt, dw
    ol = WL.WORKLOADS["outlier"]
    M, K, N = ol.M, ol.K, ol.N
    H = WL.bf16_tensor(WL.h_preact(ol)).to(dev)
    xq = torch.empty(M, K, dtype=torch.uint8, device=dev)
    act = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    gsx = torch.empty(M, K // 128, device=dev)
    Hs = copies(H)
    t = timed_b2b([lambda x=x: B.fp8_quant_fused_ex(x, B.ACT_RELU2, B.E4M3, None, act_out=act, q_out=xq,
                                                    amax_out=amax, group_scales_out=gsx, group_rows=1,
                                                    flags=B.ACCUMULATE) for x in Hs], reps)
    out["a8 group quantize 1x128"] = mem_row(t, 5.0 * M * K + 4.0 * M * (K // 128), f"H [{M},{K}]")
    del Hs, H, act
    W = WL.bf16_tensor(WL.w_down(ol)).to(dev)
    wt_q = torch.empty(N, K, dtype=torch.uint8, device=dev)
    gsw = torch.empty(K // 128, (N + 127) // 128, device=dev)
    B.fp8_quant_fused(W, B.ACT_IDENTITY, B.E4M3, None, q_t_out=wt_q, amax_out=amax, group_scales_out=gsw,
                      group_rows=128)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    xqs = copies(xq)
    t = timed_b2b([lambda x=x: B.fp8_gemm_fwd(x, wt_q, gsx, gsw, y, group_mode=1) for x in xqs], reps)
    out["a12 group-scaled GEMM"] = mma_row(t, 2.0 * M * N * K, f"X_q [{M},{K}] x W_q^T [{N},{K}]")
    del xqs, xq, W, wt_q, y
    # next: MXFP8 (one power-of-two scale per 32 values) at the outlier and GPT-2-XL shapes: the
    # quantize of H (row blocks), the weight cast (column blocks, transposed) and the block-scaled GEMM
    for wl_name in ("outlier", "gpt2xl"):
        wl = WL.WORKLOADS[wl_name]
        Mx, Kx, Nx = wl.M, wl.K, wl.N
        g = torch.Generator(device=dev).manual_seed(wl.seed)
        Hx = copies(torch.randn(Mx, Kx, device=dev, generator=g).to(torch.bfloat16))
        Wx = torch.randn(Kx, Nx, device=dev, generator=g).mul_(0.02).to(torch.bfloat16)
        qx = torch.empty(Mx, Kx, dtype=torch.uint8, device=dev)
        sfx = torch.empty(B.fp8_mx_scale_bytes(Mx, Kx), dtype=torch.uint8, device=dev)
        ax = torch.empty(Mx, Kx, dtype=torch.bfloat16, device=dev)
        r = max(4, reps // (1 if wl_name == "outlier" else 8))
        # MX scales are per block, so no per-tensor amax is asked for (it would add a zeroing memset per call)
        t = timed_b2b([lambda h=h: B.fp8_quant_mx(h, B.ACT_RELU2, B.E4M3, act_out=ax, q_out=qx, sf_out=sfx)
                       for h in Hx], r)
        out[f"next: MX quantize of H, 32-value blocks ({wl_name})"] = mem_row(
            t, 5.0 * Mx * Kx + Mx * Kx / 32, f"H [{Mx},{Kx}] -> act + E4M3 + scale bytes")
        del Hx, ax
        qwt = torch.empty(Nx, Kx, dtype=torch.uint8, device=dev)
        sfw = torch.empty(B.fp8_mx_scale_bytes(Nx, Kx), dtype=torch.uint8, device=dev)
        Wxs = copies(Wx)
        t = timed_b2b([lambda w=w: B.fp8_quant_mx(w, B.ACT_IDENTITY, B.E4M3, q_t_out=qwt, sf_t_out=sfw) for w in Wxs],
                      r)
        del Wxs
        out[f"next: MX weight cast, transposed ({wl_name})"] = mem_row(
            t, 3.0 * Kx * Nx + Kx * Nx / 32, f"W [{Kx},{Nx}] -> W_q^T + scale bytes")
        B.fp8_quant_mx(Wx, B.ACT_IDENTITY, B.E4M3, q_t_out=qwt, sf_t_out=sfw)
        yx = torch.empty(Mx, Nx, dtype=torch.bfloat16, device=dev)
        xs = copies(qx)
        t = timed_b2b([lambda x=x: B.fp8_gemm_mx(x, sfx, qwt, sfw, yx) for x in xs], r)
        out[f"next: MX GEMM, block-scaled tcgen05 ({wl_name})"] = mma_row(
            t, 2.0 * Mx * Nx * Kx, f"X_q [{Mx},{Kx}] x W_q^T [{Nx},{Kx}], scales per 32 values")
        del xs, qx, sfx, Wx, qwt, sfw, yx
    # next: the up-projection H = X_in W_up with the activation quantize in its epilogue, against
    # the same outputs from the unfused pair (the GEMM writing H, then the quantize of H); operands
    # are E4M3 codes (the GEMM's time does not depend on their values)
    for wl_name in ("gpt2s", "gpt2xl"):
        wl = WL.WORKLOADS[wl_name]
        Mu, Du, Fu = wl.M, wl.N, wl.K  # tokens, model width (the up-projection's K), hidden width
        g = torch.Generator(device=dev).manual_seed(wl.seed)
        xs = copies(torch.randint(0, 120, (Mu, Du), dtype=torch.uint8, device=dev, generator=g))
        wu = torch.randint(0, 100, (Fu, Du), dtype=torch.uint8, device=dev, generator=g)
        sx_u, sw_u = torch.full((1,), 16.0, device=dev), torch.full((1,), 448.0, device=dev)
        s_h = torch.full((1,), 100.0, device=dev)
        act_u = torch.empty(Mu, Fu, dtype=torch.bfloat16, device=dev)
        q_u = torch.empty(Mu, Fu, dtype=torch.uint8, device=dev)
        sat_u = torch.zeros(1, dtype=torch.int64, device=dev)
        r = max(4, reps // (1 if wl_name == "gpt2s" else 8))
        t = timed_b2b([lambda x=x: B.fp8_upproj_fwd(x, wu, sx_u, sw_u, s_h, q_u, act=B.ACT_RELU2, act_out=act_u,
                                                    amax_out=amax, sat_count=sat_u, flags=B.ACCUMULATE)
                       for x in xs], r)
        nbytes = Mu * Du + Fu * Du + 3.0 * Mu * Fu  # X, W in; activation (BF16) + E4M3 out
        row = mem_row(t, nbytes, f"X [{Mu},{Du}] x W_up^T [{Fu},{Du}] -> act + E4M3 [{Mu},{Fu}]")
        row["TFLOP/s"] = 2.0 * Mu * Du * Fu / (t * 1e-3) / 1e12
        row["tensor_frac"] = row["TFLOP/s"] / fp8
        row["hbm_frac"] = row["frac"]
        # bound by whichever of its bytes over the copy rate and its FLOPs over the FP8 peak is longer
        if row["tensor_frac"] > row["hbm_frac"]:
            row["bound"], row["frac"] = "tensor", row["tensor_frac"]
        h_u = torch.empty(Mu, Fu, dtype=torch.bfloat16, device=dev)
        t2 = timed_b2b([lambda x=x: (B.fp8_gemm_fwd(x, wu, sx_u, sw_u, h_u),
                                     B.fp8_quant_fused_ex(h_u, B.ACT_RELU2, B.E4M3, s_h, act_out=act_u, q_out=q_u,
                                                          amax_out=amax, sat_count=sat_u, flags=B.ACCUMULATE))
                        for x in xs], r)
        row["unfused_ms (GEMM writing H, then the quantize of H)"] = t2
        row["speedup_vs_unfused"] = t2 / t
        out[f"next: up-projection + activation quantize epilogue ({wl_name})"] = row
        del xs, wu, act_u, q_u, h_u
    torch.cuda.empty_cache()
    return out


def measure_e2e(args, dp, h_bits, w_bits, flush, w, dev, use_graph=True) -> dict:
    """The step through the public API with host buffers, fed the way a
    training loop's data feed runs: while step i computes, step i + 1's H and
    W go up from pinned memory on a copy stream (into the other of two
    device buffer pairs, once the step that last read it has finished) and
    step i's Y comes down to pinned memory on a second stream.  Every step's
    copies are inside the timed region: one event pair around K steps, from
    the first upload to the last download.  (Issued one after another on one
    stream the same step took 11.4 ms instead of 8.0 ms at GPT-2-XL size; the
    host link, ~210 GB/s up, bounds either.)"""
    M, K, N = w.M, w.K, w.N
    H_host = [WL.bf16_tensor(b).pin_memory() for b in h_bits]
    W_host = WL.bf16_tensor(w_bits).pin_memory()
    Y_host = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    Hd = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    Wd = [torch.empty(K, N, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    for b in range(2):
        Hd[b].copy_(H_host[b % len(H_host)])
        Wd[b].copy_(W_host)
    g = dp.capture(Hd[0], Wd[0], H_next=Hd[1], W_next=Wd[1]) if use_graph else None
    steps = max(3, min(args.steps, 200))
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_down = torch.cuda.Event()

    def upload(i, b):
        with torch.cuda.stream(up):
            up.wait_event(ev_done[b])  # the step that last read buffer b has finished
            Hd[b].copy_(H_host[i % len(H_host)], non_blocking=True)
            Wd[b].copy_(W_host, non_blocking=True)
            ev_up[b].record(up)

    def run(n):
        main = torch.cuda.current_stream()
        b = g.buffer() if g is not None else 0
        upload(0, b)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1, b ^ 1)
            main.wait_event(ev_up[b])
            main.wait_event(ev_down)  # the previous Y has left the output buffer
            y = g.replay() if g is not None else dp.step(Hd[b], Wd[b])
            ev_done[b].record(main)
            with torch.cuda.stream(down):
                down.wait_event(ev_done[b])
                Y_host[i % 2].copy_(y, non_blocking=True)
                ev_down.record(down)
            b ^= 1
        main.wait_stream(down)
        main.wait_stream(up)

    run(3)
    torch.cuda.synchronize()
    flush_l2(flush)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    run(steps)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    del g, Hd, Wd
    return {"value": 2.0 * M * N * K / (ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": 2 * M * K + 2 * K * N, "d2h_bytes_per_step": 2 * M * N,
            "ms_per_step": ms, "steps": steps,
            "schedule": "step i+1's inputs uploaded while step i computes; Y downloaded on a second stream"}

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WL.WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--rows", type=int, default=0, help="run the workload with this many rows of H (0: its own)")
    ap.add_argument("--cpu-rows", type=int, default=256, help="rows of the GEMM the CPU baseline times")
    ap.add_argument("--ref-rows", type=int, default=16, help="rows of H per reference-arm step")
    ap.add_argument("--no-extras", action="store_true", help="skip the comparator measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle timing")
    ap.add_argument("--eager", action="store_true",
                    help="launch the step kernel by kernel instead of as a CUDA graph")
    ap.add_argument("--profile", action="store_true",
                    help="run --steps eager steps without timing (the command an ncu capture wraps)")
    ap.add_argument("--mx", action="store_true",
                    help="with --profile: the MXFP8 path (block quantize, block cast, block-scaled GEMM)")
    ap.add_argument("--group", action="store_true",
                    help="with --profile: 1x128 / 128x128 group scales (block cast, group quantize, group-scaled GEMM)")
    ap.add_argument("--unfused", action="store_true",
                    help="with --profile: the two-launch path (batched cast, then the GEMM) instead of the one-launch step")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not args.profile:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" and torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.profile:
            run_profile(args, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
