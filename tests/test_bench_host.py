"""Host-side logic of bench.py on the CPU: the max-over-ranks / sum-of-units
reduction under a world-size-2 gloo group, the reference (oracle) arm, alone
and under torchrun with two ranks (rank 0 prints the only line), and the
roofline of the one-launch step kernel."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms, units = bench.reduce_over_ranks(1.0 + rank * 2.5, 10.0 * (rank + 1), world)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, units in got:
        assert ms == 3.5      # max of 1.0 and 3.5
        assert units == 30.0  # all ranks' units


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.strip().startswith("{")]


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=500, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def test_fused_roofline_duration_source():
    """The one-launch step kernel's roofline takes the timed steps' own time
    when each step is that one launch, else the back-to-back figure; its
    fraction is max(HBM time, tensor time) over that duration, and its
    algorithmic bytes are 5 M K + 3 K N + 2 M N."""
    sys.path.insert(0, ROOT)
    import bench
    from quantize_fp8_gemm_gb300 import workloads as WL
    w = WL.WORKLOADS["gpt2xl"]
    km = {"quant": 0.67, "gemm": 0.72, "fused_step_kernel": 1.2}
    peaks = {"hbm_gbs": 6788.6, "source": "measured"}
    fp8 = {"tflops": 3900.0, "source": "burst"}
    M, K, N = w.M, w.K, w.N
    fbytes = 5.0 * M * K + 3.0 * K * N + 2.0 * M * N
    t_roof = max(fbytes / (6788.6e9), 2.0 * M * N * K / 3900e12)
    timed = bench.rooflines(w, km, peaks, fp8, "gpt2xl", step_ms=1.05)["fused"]
    assert timed["duration_ms"] == 1.05 and timed["b2b_ms"] == 1.2
    assert timed["frac"] == pytest.approx(t_roof / 1.05e-3)
    assert timed["algorithmic_bytes"] == fbytes
    b2b = bench.rooflines(w, km, peaks, fp8, "gpt2xl")["fused"]
    assert b2b["duration_ms"] == 1.2 and b2b["frac"] == pytest.approx(t_roof / 1.2e-3)
    assert bench.rooflines(w, km, peaks, fp8, "gpt2xl")["dominant"]["kernel"].startswith("fp8_gemm_kernel<FUSED>")
