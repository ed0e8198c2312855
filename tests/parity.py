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


# The MX scale layout (include/fp8q.h, fp8_quant_mx): atoms of 128 rows x 4
# blocks, 512 bytes; (row 128 i + 32 j + l, block 4 g + k) at byte
# 512 (i G + g) + 16 l + 4 j + k, G = ceil(KB / 4).  Written out here from that
# definition, as a plain reshape and transpose.
def mx_scale_bytes(rows: int, KB: int) -> int:
    return -(-rows // 128) * -(-KB // 4) * 512


def mx_untile(sf: np.ndarray, rows: int, KB: int, pad=False):
    """The [rows, KB] scale bytes of a tiled buffer (and, with pad=True, also the
    padding blocks KB .. 4G - 1 of each row)."""
    RB, G = -(-rows // 128), -(-KB // 4)
    a = np.asarray(sf, dtype=np.uint8).reshape(-1)[:RB * G * 512].reshape(RB, G, 32, 4, 4)  # [i, g, l, j, k]
    full = a.transpose(0, 3, 2, 1, 4).reshape(RB * 128, G * 4)                                # [i j l, g k]
    return (full[:rows, :KB], full[:rows, KB:]) if pad else full[:rows, :KB]


def mx_tile(sf_rows: np.ndarray) -> np.ndarray:
    """The tiled buffer of a [rows, KB] array of scale bytes (padding blocks 127,
    rows past the grid 127)."""
    rows, KB = sf_rows.shape
    RB, G = -(-rows // 128), -(-KB // 4)
    full = np.full((RB * 128, G * 4), 127, np.uint8)
    full[:rows, :KB] = sf_rows
    return np.ascontiguousarray(full.reshape(RB, 4, 32, G, 4).transpose(0, 3, 2, 1, 4)).reshape(-1)


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
