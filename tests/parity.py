"""Helpers shared by the GPU parity tests: device/host transfers and the GEMM
tolerance.

GEMM tolerance (floating point): an output passes when
    |y_gpu - y_ref| <= ulp_bf16(y_ref) + 1e-5 * S,
where y_ref is the oracle's double-precision result, S the same sum taken over
|terms|, and ulp_bf16(y) = 2^(max(floor(log2|y|), -126) - 7) the BF16 spacing
at y.  The first term covers the final rounding to BF16 (half an ulp) plus
slack for a result that sits near a rounding boundary; the second covers the
FP32 accumulation and the float32 dequantisation factor 1/(s_a s_b).
"""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy().view(np.uint8)


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_f32(x) -> torch.Tensor:
    return torch.tensor(np.atleast_1d(np.asarray(x, dtype=np.float32)), device="cuda")


def bf16_ulp(y: np.ndarray) -> np.ndarray:
    a = np.abs(y)
    with np.errstate(divide="ignore"):
        e = np.where(a > 0, np.floor(np.log2(np.where(a > 0, a, 1.0))), -126.0)
    e = np.maximum(e, -126.0)
    return np.exp2(e - 7.0)


def gemm_within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, S: np.ndarray):
    """Return (ok_mask, err, tol) for the GEMM tolerance above."""
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    tol = bf16_ulp(y_ref) + 1e-5 * S
    return err <= tol, err, tol


def assert_gemm_close(y_gpu_bf16: torch.Tensor, y_ref: np.ndarray, S: np.ndarray, rows=None):
    y = y_gpu_bf16.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        y = y[rows]
    ok, err, tol = gemm_within_tolerance(y, y_ref, S)
    if not ok.all():
        idx = np.argwhere(~ok)
        i, j = idx[0]
        raise AssertionError(
            f"{(~ok).sum()} of {ok.size} outputs outside tolerance; first at {tuple(idx[0])}: "
            f"gpu={y[i, j]!r} ref={y_ref[i, j]!r} err={err[i, j]:.3e} tol={tol[i, j]:.3e}; "
            f"max err/tol={np.max(err / tol):.3f}")
