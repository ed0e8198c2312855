"""Seeded synthetic inputs for the FP8 down-projection workloads.

This module only draws random numbers and rounds them to BF16 input tensors.
It holds none of the method's arithmetic, so both the CUDA path and the CPU
oracle may consume what it produces.

Generation is chunked: chunk c of a stream draws from
``numpy.random.default_rng(SeedSequence([seed, stream, c]))``, so the values
depend only on (seed, stream, shape), not on how many threads fill them.
BF16 rounding of the float32 draws is done by torch's conversion.

Workloads (the FP8 down-projection of a GPT-2-style MLP; H is the BF16
pre-activation, W_down is [K, N]):

========== ======= ===== ===== ==================================================
name        M       K     N     recipe
========== ======= ===== ===== ==================================================
tiny        64      256   64    seed 0, H~N(0,1), W~N(0,0.02), previous amax 4.0,
                                margin 2.0, one step
gpt2s       8192    3072  768   seed 1, H~N(0,1) fresh every step, W fixed,
                                margin 2.0, 10 steps, history length 1
gpt2s_batch 65536   3072  768   seed 2, 20 steps, std of H drifts linearly
                                1.0 -> 1.5 (std_t = 1 + 0.5 t / 19)
outlier     16384   4096  1024  seed 3, H~N(0,1) with M*K/4096 seeded positions
                                set to +-1e5 (random sign)
gpt2xl      131072  6400  1600  seed 4, H~N(0,1); W~N(0,0.02); dY~N(0,1e-3) [M,N]
                                with 0.1% of entries multiplied by 100
========== ======= ===== ===== ==================================================
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

CHUNK = 1 << 22


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    seed: int
    steps: int
    margin: float
    history_len: int = 1
    w_std: float = 0.02
    prev_amax: float | None = None  # given previous-step amax (tiny case)


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 64, seed=0, steps=1, margin=2.0, prev_amax=4.0),
    "gpt2s": Workload("gpt2s", 8192, 3072, 768, seed=1, steps=10, margin=2.0),
    "gpt2s_batch": Workload("gpt2s_batch", 65536, 3072, 768, seed=2, steps=20, margin=2.0),
    "outlier": Workload("outlier", 16384, 4096, 1024, seed=3, steps=1, margin=1.0),
    "gpt2xl": Workload("gpt2xl", 131072, 6400, 1600, seed=4, steps=1, margin=2.0),
}

# stream ids: one independent random stream per tensor role
STREAM_H, STREAM_W, STREAM_DY, STREAM_OUTLIER, STREAM_DY_SPIKE = 0, 1, 2, 3, 4


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return 4


def normal_f32(n: int, seed: int, stream: int, step: int = 0) -> np.ndarray:
    """n standard-normal float32 draws, reproducible from (seed, stream, step)."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(c: int) -> None:
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        rng = np.random.default_rng(np.random.SeedSequence([seed, stream, step, c]))
        rng.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks <= 1:
        fill(0) if n else None
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to BF16 (torch's conversion); return the uint16 patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    """A torch.bfloat16 CPU tensor that shares the given uint16 patterns."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def h_preact(w: Workload, step: int = 0, std: float = 1.0) -> np.ndarray:
    """BF16 pre-activation H [M,K] for one step, as uint16 patterns."""
    x = normal_f32(w.M * w.K, w.seed, STREAM_H, step)
    if std != 1.0:
        x *= np.float32(std)
    if w.name == "outlier":
        rng = np.random.default_rng(np.random.SeedSequence([w.seed, STREAM_OUTLIER, step]))
        n_out = (w.M * w.K) // 4096
        pos = rng.choice(w.M * w.K, size=n_out, replace=False)
        sign = rng.integers(0, 2, size=n_out).astype(np.float32) * 2.0 - 1.0
        x[pos] = sign * np.float32(1e5)
    return to_bf16_bits(x).reshape(w.M, w.K)


def drift_std(w: Workload, step: int) -> float:
    """Standard deviation of H at a step: a linear drift 1.0 -> 1.5 for gpt2s_batch."""
    if w.name == "gpt2s_batch":
        return 1.0 + 0.5 * step / max(1, w.steps - 1)
    return 1.0


def w_down(w: Workload) -> np.ndarray:
    """BF16 down-projection weight W [K,N] ~ N(0, w_std), as uint16 patterns."""
    x = normal_f32(w.K * w.N, w.seed, STREAM_W)
    x *= np.float32(w.w_std)
    return to_bf16_bits(x).reshape(w.K, w.N)


def dy_grad(w: Workload) -> np.ndarray:
    """BF16 output gradient dY [M,N] ~ N(0, 1e-3), 0.1% of entries times 100."""
    x = normal_f32(w.M * w.N, w.seed, STREAM_DY)
    x *= np.float32(1e-3)
    rng = np.random.default_rng(np.random.SeedSequence([w.seed, STREAM_DY_SPIKE]))
    n_sp = (w.M * w.N) // 1000
    pos = rng.choice(w.M * w.N, size=n_sp, replace=False)
    x[pos] *= np.float32(100.0)
    return to_bf16_bits(x).reshape(w.M, w.N)


def sample_rows(M: int, n: int, seed: int, tile: int = 128, edge_tiles: int = 8) -> np.ndarray:
    """A seeded, sorted set of output rows: n random rows plus the first and
    last row of a few 128-row tiles (the first two, the last two and up to
    edge_tiles - 4 random ones)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 99]))
    ntiles = (M + tile - 1) // tile
    picks = {0, 1, ntiles - 2, ntiles - 1}
    if ntiles > 4:
        picks |= set(rng.choice(ntiles, size=min(ntiles, max(0, edge_tiles - 4)), replace=False).tolist())
    edges = []
    for t in sorted(p for p in picks if 0 <= p < ntiles):
        edges += [t * tile, min(M - 1, t * tile + tile - 1)]
    pick = rng.choice(M, size=min(n, M), replace=False)
    return np.unique(np.concatenate([pick, np.array(edges, dtype=np.int64)])).astype(np.int64)
