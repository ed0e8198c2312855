"""ctypes binding of libfp8q.so: the C ABI of include/fp8q.h, same names.

Argument marshalling only.  Each function checks that the tensors it is given
are CUDA tensors of the byte sizes the C call will touch (so a wrong shape is
a Python error, not an out-of-bounds access on the GPU), passes raw device
pointers and the current CUDA stream, and raises ``Fp8qError`` on a non-zero
status.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback: if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfp8q.so")
NAIVE_LIB_PATH = os.path.join(PKG, "libfp8q_naive.so")  # the unfused comparator (include/fp8q_naive.h)

E4M3, E5M2 = 0, 1
ACT_IDENTITY, ACT_RELU, ACT_RELU2 = 0, 1, 2
DEV_TIMEOUT, DEV_BAD_AMAX = 1, 2
ACCUMULATE = 1  # fp8_quant_fused_ex flag
BATCH_MAX = 4  # FP8Q_BATCH_MAX
GROUP = 128
NOALLOC_MAX_M = 262144  # FP8Q_NOALLOC_MAX_M

_lib = None
_naive = None


class Fp8qError(RuntimeError):
    """A libfp8q call returned a non-zero fp8q_status."""

    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: status {status} ({msg})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libfp8q.so (built in-tree); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built: run quantize_fp8_gemm_gb300.build.build() "
                "(or python -c 'import __graft_entry__ as g; g.build()') first")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        L.fp8_quant_fused.argtypes = [P, i64, i64, i32, i32, P, P, P, P, P, P, P, i32, P]
        L.fp8_quant_fused_ex.argtypes = [P, i64, i64, i32, i32, P, P, P, P, P, P, P, i32, ctypes.c_uint, P]
        L.fp8_gemm_fwd.argtypes = [P, P, P, P, i32, P, i64, i64, i64, P, P]
        L.fp8_gemm_fwd_update.argtypes = [P, P, P, P, P, i64, i64, i64, P, P, P, P, P, P]
        L.fp8_quant_fused_batch.argtypes = [P, i32, P]
        L.fp8_cast_f32.argtypes = [P, P, i64, i32, P]
        L.fp8_gemm_dgrad.argtypes = [P, P, P, P, P, i64, i64, i64, P, P]
        L.fp8_gemm_wgrad.argtypes = [P, P, P, P, P, i64, i64, i64, P, P]
        L.fp8_gemm_dgrad_act.argtypes = [P, P, P, P, P, i32, P, i64, i64, i64, P, P]
        L.fp8_gemm_dgrad_act_q.argtypes = [P, P, P, P, P, P, i32, P, i64, i64, i64, P, P]
        L.fp8_upproj_fwd.argtypes = [P, P, P, P, i32, P, P, P, P, P, P, i64, i64, i64, ctypes.c_uint, P, P]
        L.amax_history_update.argtypes = [P, i32, P, P, f32, i32, P, P, P]
        L.amax_history_update_ex.argtypes = [P, i32, P, P, f32, i32, P, P, P, P, P, P]
        L.fp8_downproj_workspace_bytes.argtypes = [i64]
        L.fp8_downproj_workspace_bytes.restype = ctypes.c_size_t
        L.fp8_downproj_fwd.argtypes = [P, P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
        L.fp8_downproj_fwd_ex.argtypes = [P, P, P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, P, P, P,
                                          ctypes.c_size_t, P, P, ctypes.c_uint, P, P]
        L.fp8_downproj_fwd_noalloc.argtypes = [P, P, i64, i64, i64, i32, P, P, P, P, P, P, P, P, P]
        L.fp8q_status_string.argtypes = [i32]
        L.fp8q_status_string.restype = ctypes.c_char_p
        L.fp8q_version.restype = i32
        L.fp8q_gemm_test_hold_loads.argtypes = [i32]
        L.fp8q_gemm_test_hold_loads.restype = None
        L.fp8q_gemm_set_tile.argtypes = [i32, i32]
        L.fp8q_gemm_set_tile.restype = i32
        L.fp8q_test_set_fused_grid.argtypes = [i32]
        L.fp8q_test_set_fused_grid.restype = i32
        L.fp8q_test_set_fused_layout.argtypes = [i32]
        L.fp8q_test_set_fused_layout.restype = i32
        L.fp8q_test_gemm_tile.argtypes = [i64, i64, i32, P, P]
        L.fp8q_test_gemm_tile.restype = i32
        L.fp8q_test_noalloc_fill.argtypes = [i32, P]
        L.fp8q_test_noalloc_fill.restype = i32
        L.fp8q_mx_set_tile.argtypes = [i32, i32]
        L.fp8q_mx_set_tile.restype = i32
        L.fp8_quant_mx.argtypes = [P, i64, i64, i32, i32, P, P, P, P, P, P, P, P]
        L.fp8_gemm_mx.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, P, P]
        L.fp8_mx_scale_bytes.argtypes = [i64, i64]
        L.fp8_mx_scale_bytes.restype = i64
        for fn in ("fp8_quant_fused", "fp8_quant_fused_ex", "fp8_quant_fused_batch", "fp8_downproj_fwd",
                   "fp8_downproj_fwd_noalloc", "fp8_downproj_fwd_ex", "fp8_gemm_fwd", "fp8_gemm_fwd_update", "fp8_gemm_dgrad", "fp8_gemm_wgrad", "fp8_gemm_dgrad_act", "fp8_gemm_dgrad_act_q", "fp8_upproj_fwd", "amax_history_update",
                   "amax_history_update_ex", "fp8_quant_mx", "fp8_gemm_mx"):
            getattr(L, fn).restype = i32
        _lib = L
    return _lib


def naive_lib() -> ctypes.CDLL:
    """Load libfp8q_naive.so, the unfused three-pass comparator; raise if it is missing."""
    global _naive
    if _naive is None:
        lib()  # the status strings live in the main library
        if not os.path.exists(NAIVE_LIB_PATH):
            raise RuntimeError(f"{NAIVE_LIB_PATH} is not built: run quantize_fp8_gemm_gb300.build.build() first")
        L = ctypes.CDLL(NAIVE_LIB_PATH)
        P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        L.fp8q_naive_act.argtypes = [P, i64, i64, i32, P, P]
        L.fp8q_naive_amax.argtypes = [P, i64, P, P]
        L.fp8q_naive_cast.argtypes = [P, i64, i32, P, f32, P, P, P]
        for fn in ("fp8q_naive_act", "fp8q_naive_amax", "fp8q_naive_cast"):
            getattr(L, fn).restype = i32
        _naive = L
    return _naive


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise Fp8qError(fn, status, lib().fp8q_status_string(status).decode())


def _ptr(t, nbytes: int | None, name: str):
    """Device pointer of an optional CUDA tensor holding at least nbytes."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    have = t.numel() * t.element_size()
    if nbytes is not None and have < nbytes:
        raise ValueError(f"{name} holds {have} bytes, the call needs {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def fp8_quant_fused(h: torch.Tensor, act: int, fmt: int, scale: torch.Tensor | None = None, *,
                    act_out=None, q_out=None, q_t_out=None, amax_out=None, sat_count=None,
                    group_scales_out=None, group_rows: int = 1, stream=None) -> None:
    """Fused activation + BF16 copy + FP8 cast + amax of a [M,K] BF16 tensor."""
    fp8_quant_fused_ex(h, act, fmt, scale, act_out=act_out, q_out=q_out, q_t_out=q_t_out,
                       amax_out=amax_out, sat_count=sat_count, group_scales_out=group_scales_out,
                       group_rows=group_rows, flags=0, stream=stream)


def fp8_quant_fused_ex(h: torch.Tensor, act: int, fmt: int, scale: torch.Tensor | None = None, *,
                       act_out=None, q_out=None, q_t_out=None, amax_out=None, sat_count=None,
                       group_scales_out=None, group_rows: int = 1, flags: int = 0, stream=None) -> None:
    """fp8_quant_fused with flags (ACCUMULATE: fold into amax_out / sat_count)."""
    M, K = h.shape
    n = M * K
    ng = ((M + group_rows - 1) // max(group_rows, 1)) * (K // GROUP) if group_scales_out is not None else 0
    name = "fp8_quant_fused" if flags == 0 else "fp8_quant_fused_ex"
    st = lib().fp8_quant_fused_ex(
        _ptr(h, 2 * n, "h"), M, K, act, fmt, _ptr(scale, 4, "scale"),
        _ptr(act_out, 2 * n, "act_out"), _ptr(q_out, n, "q_out"), _ptr(q_t_out, n, "q_t_out"),
        _ptr(amax_out, 4, "amax_out"), _ptr(sat_count, 8, "sat_count"),
        _ptr(group_scales_out, 4 * ng, "group_scales_out"), group_rows, flags, _stream(stream))
    _check(name, st)


class QuantArgs(ctypes.Structure):
    """fp8q_quant_args: the arguments of one quantize call in fp8_quant_fused_batch."""
    _fields_ = [("h", ctypes.c_void_p), ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("act", ctypes.c_int),
                ("fmt", ctypes.c_int), ("scale", ctypes.c_void_p), ("act_out", ctypes.c_void_p),
                ("q_out", ctypes.c_void_p), ("q_t_out", ctypes.c_void_p), ("amax_out", ctypes.c_void_p),
                ("sat_count", ctypes.c_void_p), ("group_scales_out", ctypes.c_void_p),
                ("group_rows", ctypes.c_int), ("flags", ctypes.c_uint), ("hq_out", ctypes.c_void_p),
                ("scale_h", ctypes.c_void_p), ("amax_h", ctypes.c_void_p), ("sat_h", ctypes.c_void_p)]


def quant_args(h: torch.Tensor, act: int, fmt: int, scale: torch.Tensor, *, act_out=None, q_out=None,
               q_t_out=None, amax_out=None, sat_count=None, flags: int = 0, hq_out=None, scale_h=None,
               amax_h=None, sat_h=None) -> QuantArgs:
    """One entry of fp8_quant_fused_batch (per-tensor scale), with the byte-size
    checks of fp8_quant_fused; hq_out / scale_h / amax_h / sat_h: the E4M3 cache
    of the pre-activation h itself.  The entry holds references to its tensors,
    so temporaries passed here live as long as the entry."""
    M, K = h.shape
    n = M * K
    v = lambda t, nb, name: (lambda p: None if p is None else p.value)(_ptr(t, nb, name))
    a = QuantArgs(v(h, 2 * n, "h"), M, K, act, fmt, v(scale, 4, "scale"), v(act_out, 2 * n, "act_out"),
                  v(q_out, n, "q_out"), v(q_t_out, n, "q_t_out"), v(amax_out, 4, "amax_out"),
                  v(sat_count, 8, "sat_count"), None, 1, flags, v(hq_out, n, "hq_out"), v(scale_h, 4, "scale_h"),
                  v(amax_h, 4, "amax_h"), v(sat_h, 8, "sat_h"))
    a._tensors = (h, scale, act_out, q_out, q_t_out, amax_out, sat_count, hq_out, scale_h, amax_h, sat_h)
    return a


def fp8_quant_fused_batch(entries, stream=None) -> None:
    """Several per-tensor quantize calls (QuantArgs from quant_args) in one launch."""
    arr = (QuantArgs * len(entries))(*entries)
    _check("fp8_quant_fused_batch", lib().fp8_quant_fused_batch(arr, len(entries), _stream(stream)))


def fp8_cast_f32(x: torch.Tensor, fmt: int, q: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q = FP8(x) elementwise (round to nearest even, saturating): the quantize kernels' conversion."""
    if x.dtype != torch.float32:
        raise TypeError("x must be float32")
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    n = x.numel()
    _check("fp8_cast_f32", lib().fp8_cast_f32(_ptr(x, 4 * n, "x"), _ptr(q, n, "q"), n, fmt, _stream(stream)))
    return q


def fp8_gemm_fwd(x_q: torch.Tensor, wt_q: torch.Tensor, scale_x: torch.Tensor, scale_w: torch.Tensor,
                 y: torch.Tensor, *, group_mode: int = 0, amax_x=None, hist_x=None, amax_w=None, hist_w=None,
                 status=None, stream=None) -> None:
    """y[M,N] = BF16((x_q[M,K] . wt_q[N,K]^T) / (s_x s_w)) on the tensor cores.  With
    hist_x / hist_w (HistoryArgs, per-tensor scales only) the call is
    fp8_gemm_fwd_update: the GEMM also runs those delayed-scale updates on
    amax_x / amax_w."""
    M, K = x_q.shape
    N = wt_q.shape[0]
    if wt_q.shape[1] != K:
        raise ValueError("x_q [M,K] and wt_q [N,K] disagree on K")
    if hist_x is not None or hist_w is not None:
        if group_mode:
            raise ValueError("the delayed-scale updates go with per-tensor scales")
        st = lib().fp8_gemm_fwd_update(
            _ptr(x_q, M * K, "x_q"), _ptr(wt_q, N * K, "wt_q"), _ptr(scale_x, 4, "scale_x"),
            _ptr(scale_w, 4, "scale_w"), _ptr(y, 2 * M * N, "y"), M, N, K, _ptr(amax_x, 4, "amax_x"),
            None if hist_x is None else ctypes.byref(hist_x), _ptr(amax_w, 4, "amax_w"),
            None if hist_w is None else ctypes.byref(hist_w), _ptr(status, 4, "status"), _stream(stream))
        _check("fp8_gemm_fwd_update", st)
        return
    if group_mode:
        sx, sw = 4 * M * (K // GROUP), 4 * (K // GROUP) * ((N + GROUP - 1) // GROUP)
    else:
        sx, sw = 4, 4
    st = lib().fp8_gemm_fwd(
        _ptr(x_q, M * K, "x_q"), _ptr(wt_q, N * K, "wt_q"), _ptr(scale_x, sx, "scale_x"),
        _ptr(scale_w, sw, "scale_w"), group_mode, _ptr(y, 2 * M * N, "y"), M, N, K,
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_gemm_fwd", st)


def fp8_gemm_dgrad(dy_q: torch.Tensor, w_q: torch.Tensor, scale_dy: torch.Tensor, scale_w: torch.Tensor,
                   dx: torch.Tensor, *, status=None, stream=None) -> None:
    """dx[M,K] = BF16((dy_q[M,N] . w_q[K,N]^T) / (s_dy s_w)) on the tensor cores."""
    M, N = dy_q.shape
    K = w_q.shape[0]
    if w_q.shape[1] != N:
        raise ValueError("dy_q [M,N] and w_q [K,N] disagree on N")
    st = lib().fp8_gemm_dgrad(
        _ptr(dy_q, M * N, "dy_q"), _ptr(w_q, K * N, "w_q"), _ptr(scale_dy, 4, "scale_dy"),
        _ptr(scale_w, 4, "scale_w"), _ptr(dx, 2 * M * K, "dx"), M, N, K,
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_gemm_dgrad", st)


def fp8_gemm_dgrad_act(dy_q: torch.Tensor, w_q: torch.Tensor, scale_dy: torch.Tensor, scale_w: torch.Tensor,
                       h: torch.Tensor, dh: torch.Tensor, *, act: int = ACT_RELU2, status=None, stream=None) -> None:
    """dh[M,K] = BF16(dX * act'(h)): the dgrad dX = dy_q . w_q^T / (s_dy s_w) times the
    activation derivative at the BF16 pre-activation h [M,K], in the GEMM's epilogue."""
    M, N = dy_q.shape
    K = w_q.shape[0]
    if w_q.shape[1] != N:
        raise ValueError("dy_q [M,N] and w_q [K,N] disagree on N")
    st = lib().fp8_gemm_dgrad_act(
        _ptr(dy_q, M * N, "dy_q"), _ptr(w_q, K * N, "w_q"), _ptr(scale_dy, 4, "scale_dy"),
        _ptr(scale_w, 4, "scale_w"), _ptr(h, 2 * M * K, "h"), act, _ptr(dh, 2 * M * K, "dh"), M, N, K,
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_gemm_dgrad_act", st)


def fp8_gemm_dgrad_act_q(dy_q: torch.Tensor, w_q: torch.Tensor, scale_dy: torch.Tensor, scale_w: torch.Tensor,
                         h_q: torch.Tensor, scale_h: torch.Tensor, dh: torch.Tensor, *, act: int = ACT_RELU2,
                         status=None, stream=None) -> None:
    """fp8_gemm_dgrad_act with the pre-activation from its E4M3 cache h_q [M,K] (cast with scale_h)."""
    M, N = dy_q.shape
    K = w_q.shape[0]
    if w_q.shape[1] != N:
        raise ValueError("dy_q [M,N] and w_q [K,N] disagree on N")
    st = lib().fp8_gemm_dgrad_act_q(
        _ptr(dy_q, M * N, "dy_q"), _ptr(w_q, K * N, "w_q"), _ptr(scale_dy, 4, "scale_dy"),
        _ptr(scale_w, 4, "scale_w"), _ptr(h_q, M * K, "h_q"), _ptr(scale_h, 4, "scale_h"), act,
        _ptr(dh, 2 * M * K, "dh"), M, N, K, _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_gemm_dgrad_act_q", st)


def fp8_gemm_wgrad(x_q_t: torch.Tensor, dy_q_t: torch.Tensor, scale_x: torch.Tensor, scale_dy: torch.Tensor,
                   dw: torch.Tensor, *, status=None, stream=None) -> None:
    """dw[K,N] = BF16((x_q_t[K,M] . dy_q_t[N,M]^T) / (s_x s_dy)): the weight gradient X^T dY."""
    K, M = x_q_t.shape
    N = dy_q_t.shape[0]
    if dy_q_t.shape[1] != M:
        raise ValueError("x_q_t [K,M] and dy_q_t [N,M] disagree on M")
    st = lib().fp8_gemm_wgrad(
        _ptr(x_q_t, K * M, "x_q_t"), _ptr(dy_q_t, N * M, "dy_q_t"), _ptr(scale_x, 4, "scale_x"),
        _ptr(scale_dy, 4, "scale_dy"), _ptr(dw, 2 * K * N, "dw"), M, N, K,
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_gemm_wgrad", st)


def fp8_upproj_fwd(x_q: torch.Tensor, wt_q: torch.Tensor, scale_x: torch.Tensor, scale_w: torch.Tensor,
                   scale_h: torch.Tensor, h_q: torch.Tensor, *, act: int = ACT_RELU2, h_out=None, act_out=None,
                   amax_out=None, sat_count=None, flags: int = 0, status=None, stream=None) -> None:
    """Up-projection H = x_q[M,K] . wt_q[N,K]^T / (s_x s_w) with the activation quantize in its
    epilogue: h_q[M,N] = E4M3(BF16(act(BF16(H))) * s_h), and optionally H, the activation, amax, saturations."""
    M, K = x_q.shape
    N = wt_q.shape[0]
    if wt_q.shape[1] != K:
        raise ValueError("x_q [M,K] and wt_q [N,K] disagree on K")
    st = lib().fp8_upproj_fwd(
        _ptr(x_q, M * K, "x_q"), _ptr(wt_q, N * K, "wt_q"), _ptr(scale_x, 4, "scale_x"), _ptr(scale_w, 4, "scale_w"),
        act, _ptr(scale_h, 4, "scale_h"), _ptr(h_out, 2 * M * N, "h_out"), _ptr(act_out, 2 * M * N, "act_out"),
        _ptr(h_q, M * N, "h_q"), _ptr(amax_out, 4, "amax_out"), _ptr(sat_count, 8, "sat_count"), M, N, K, flags,
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_upproj_fwd", st)


def fp8_downproj_workspace_bytes(M: int) -> int:
    return int(lib().fp8_downproj_workspace_bytes(M))


def fp8_downproj_fwd(h: torch.Tensor, wt_q: torch.Tensor, scale_x: torch.Tensor, scale_w: torch.Tensor,
                     x_q: torch.Tensor, y: torch.Tensor, workspace: torch.Tensor, *, act: int = ACT_RELU2,
                     act_out=None, amax_out=None, sat_count=None, status=None, stream=None) -> None:
    """Fused quantize of H [M,K] + forward GEMM with W_q^T [N,K] -> y [M,N], one kernel."""
    M, K = h.shape
    N = wt_q.shape[0]
    if wt_q.shape[1] != K:
        raise ValueError("h [M,K] and wt_q [N,K] disagree on K")
    ws = fp8_downproj_workspace_bytes(M)
    st = lib().fp8_downproj_fwd(
        _ptr(h, 2 * M * K, "h"), _ptr(wt_q, N * K, "wt_q"), M, N, K, act, _ptr(scale_x, 4, "scale_x"),
        _ptr(scale_w, 4, "scale_w"), _ptr(act_out, 2 * M * K, "act_out"), _ptr(x_q, M * K, "x_q"),
        _ptr(amax_out, 4, "amax_out"), _ptr(sat_count, 8, "sat_count"), _ptr(y, 2 * M * N, "y"),
        _ptr(workspace, ws, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_downproj_fwd", st)


class HistoryArgs(ctypes.Structure):
    """fp8q_history_args: one delayed-scale update run inside fp8_downproj_fwd_ex."""
    _fields_ = [("history", ctypes.c_void_p), ("L", ctypes.c_int), ("head", ctypes.c_void_p),
                ("margin", ctypes.c_float), ("fmt", ctypes.c_int), ("scale_prev", ctypes.c_void_p),
                ("scale_out", ctypes.c_void_p), ("status", ctypes.c_void_p), ("amax_clear", ctypes.c_void_p),
                ("sat_clear", ctypes.c_void_p)]


def history_args(history: torch.Tensor, head: torch.Tensor, margin: float, fmt: int, scale_out: torch.Tensor, *,
                 scale_prev=None, status=None, amax_clear=None, sat_clear=None) -> HistoryArgs:
    """The arguments of amax_history_update_ex (amax_new is the kernel's own amax)."""
    v = lambda t, nb, name: (lambda p: None if p is None else p.value)(_ptr(t, nb, name))
    L = history.numel()
    a = HistoryArgs(v(history, 4 * L, "history"), L, v(head, 4, "head"), float(margin), fmt,
                    v(scale_prev, 4, "scale_prev"), v(scale_out, 4, "scale_out"), v(status, 4, "status"),
                    v(amax_clear, 4, "amax_clear"), v(sat_clear, 8, "sat_clear"))
    a._tensors = (history, head, scale_out, scale_prev, status, amax_clear, sat_clear)
    return a


def fp8_downproj_fwd_ex(h: torch.Tensor, wt_q: torch.Tensor, scale_x: torch.Tensor, scale_w: torch.Tensor,
                        x_q: torch.Tensor, y: torch.Tensor, workspace: torch.Tensor, *, w=None, w_q=None,
                        amax_w=None, sat_w=None, act: int = ACT_RELU2, act_out=None, amax_out=None, sat_count=None,
                        hist_x=None, hist_w=None, flags: int = 0, status=None, stream=None) -> None:
    """fp8_downproj_fwd with the weight cast (w [K,N] -> wt_q, w_q, amax_w, sat_w) in the same kernel;
    hist_x / hist_w (HistoryArgs): the delayed-scale updates, run by the kernel's last CTA;
    flags=ACCUMULATE: nothing is zeroed first (the workspace must be zero)."""
    M, K = h.shape
    N = wt_q.shape[0]
    if wt_q.shape[1] != K or (w is not None and tuple(w.shape) != (K, N)):
        raise ValueError("h [M,K], wt_q [N,K] and w [K,N] disagree")
    ws = fp8_downproj_workspace_bytes(M)
    st = lib().fp8_downproj_fwd_ex(
        _ptr(h, 2 * M * K, "h"), _ptr(w, 2 * K * N, "w"), _ptr(wt_q, N * K, "wt_q"), M, N, K, act,
        _ptr(scale_x, 4, "scale_x"), _ptr(scale_w, 4, "scale_w"), _ptr(act_out, 2 * M * K, "act_out"),
        _ptr(x_q, M * K, "x_q"), _ptr(amax_out, 4, "amax_out"), _ptr(sat_count, 8, "sat_count"),
        _ptr(w_q, K * N, "w_q"), _ptr(amax_w, 4, "amax_w"), _ptr(sat_w, 8, "sat_w"), _ptr(y, 2 * M * N, "y"),
        _ptr(workspace, ws, "workspace"), workspace.numel() * workspace.element_size(),
        None if hist_x is None else ctypes.byref(hist_x), None if hist_w is None else ctypes.byref(hist_w), flags,
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_downproj_fwd_ex", st)


def fp8_downproj_fwd_noalloc(h: torch.Tensor, wt_q: torch.Tensor, scale_x: torch.Tensor, scale_w: torch.Tensor,
                             x_q: torch.Tensor, y: torch.Tensor, *, act: int = ACT_RELU2, act_out=None,
                             amax_out=None, sat_count=None, status=None, stream=None) -> None:
    """fp8_downproj_fwd with the library's own static scratch (M <= NOALLOC_MAX_M); allocates nothing."""
    M, K = h.shape
    N = wt_q.shape[0]
    if wt_q.shape[1] != K:
        raise ValueError("h [M,K] and wt_q [N,K] disagree on K")
    st = lib().fp8_downproj_fwd_noalloc(
        _ptr(h, 2 * M * K, "h"), _ptr(wt_q, N * K, "wt_q"), M, N, K, act, _ptr(scale_x, 4, "scale_x"),
        _ptr(scale_w, 4, "scale_w"), _ptr(act_out, 2 * M * K, "act_out"), _ptr(x_q, M * K, "x_q"),
        _ptr(amax_out, 4, "amax_out"), _ptr(sat_count, 8, "sat_count"), _ptr(y, 2 * M * N, "y"),
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_downproj_fwd_noalloc", st)


def fp8_mx_scale_bytes(rows: int, K: int) -> int:
    """Bytes of the tiled scale layout of a [rows, K/32] MX block grid (K % 32 == 0)."""
    n = lib().fp8_mx_scale_bytes(int(rows), int(K))
    if n < 0:
        raise ValueError(f"no MX scale layout for rows={rows}, K={K}")
    return n


def fp8_quant_mx(h: torch.Tensor, act: int, fmt: int, *, act_out=None, q_out=None, sf_out=None, q_t_out=None,
                 sf_t_out=None, amax_out=None, sat_count=None, stream=None) -> None:
    """MXFP8 quantize of h [M,K]: one power-of-two scale byte per 32 values, along the rows
    (q_out [M,K], sf_out: the tiled layout of the [M, K/32] grid) or down the columns, transposed
    (q_t_out [K,M], sf_t_out: the tiled layout of the [K, M/32] grid)."""
    M, K = h.shape
    n = M * K
    sf_n = fp8_mx_scale_bytes(M, K) if sf_out is not None else None
    sf_t_n = fp8_mx_scale_bytes(K, M) if sf_t_out is not None else None
    st = lib().fp8_quant_mx(
        _ptr(h, 2 * n, "h"), M, K, act, fmt, _ptr(act_out, 2 * n, "act_out"), _ptr(q_out, n, "q_out"),
        _ptr(sf_out, sf_n, "sf_out"), _ptr(q_t_out, n, "q_t_out"), _ptr(sf_t_out, sf_t_n, "sf_t_out"),
        _ptr(amax_out, 4, "amax_out"), _ptr(sat_count, 8, "sat_count"), _stream(stream))
    _check("fp8_quant_mx", st)


def fp8_gemm_mx(x_q: torch.Tensor, sf_x: torch.Tensor, wt_q: torch.Tensor, sf_w: torch.Tensor, y: torch.Tensor, *,
                fmt_x: int = E4M3, fmt_w: int = E4M3, status=None, stream=None) -> None:
    """y[M,N] = BF16(sum_k x_q 2^(sf_x - 127) wt_q 2^(sf_w - 127)) on the block-scaled tensor cores
    (sf_x, sf_w: the tiled scale layouts of fp8_quant_mx's outputs)."""
    M, K = x_q.shape
    N = wt_q.shape[0]
    if wt_q.shape[1] != K:
        raise ValueError("x_q [M,K] and wt_q [N,K] disagree on K")
    st = lib().fp8_gemm_mx(
        _ptr(x_q, M * K, "x_q"), _ptr(sf_x, fp8_mx_scale_bytes(M, K), "sf_x"), _ptr(wt_q, N * K, "wt_q"),
        _ptr(sf_w, fp8_mx_scale_bytes(N, K), "sf_w"), _ptr(y, 2 * M * N, "y"), M, N, K, fmt_x, fmt_w,
        _ptr(status, 4, "status"), _stream(stream))
    _check("fp8_gemm_mx", st)


def amax_history_update(history: torch.Tensor, head: torch.Tensor, amax_new: torch.Tensor, margin: float,
                        fmt: int, scale_out: torch.Tensor, *, status=None, stream=None) -> None:
    """Push amax_new into the device ring; scale_out = fmt_max / (margin * max(history))."""
    L = history.numel()
    st = lib().amax_history_update(
        _ptr(history, 4 * L, "history"), L, _ptr(head, 4, "head"), _ptr(amax_new, 4, "amax_new"),
        float(margin), fmt, _ptr(scale_out, 4, "scale_out"), _ptr(status, 4, "status"), _stream(stream))
    _check("amax_history_update", st)


def amax_history_update_ex(history: torch.Tensor, head: torch.Tensor, amax_new: torch.Tensor, margin: float,
                           fmt: int, scale_out: torch.Tensor, *, scale_prev=None, status=None, amax_clear=None,
                           sat_clear=None, stream=None) -> None:
    """amax_history_update; a bad amax copies scale_prev into scale_out; zeroes amax_clear / sat_clear."""
    L = history.numel()
    st = lib().amax_history_update_ex(
        _ptr(history, 4 * L, "history"), L, _ptr(head, 4, "head"), _ptr(amax_new, 4, "amax_new"),
        float(margin), fmt, _ptr(scale_prev, 4, "scale_prev"), _ptr(scale_out, 4, "scale_out"),
        _ptr(status, 4, "status"), _ptr(amax_clear, 4, "amax_clear"), _ptr(sat_clear, 8, "sat_clear"),
        _stream(stream))
    _check("amax_history_update_ex", st)


# -- the unfused three-pass comparator (include/fp8q_naive.h, libfp8q_naive.so) --
def fp8q_naive_act(h, act: int, act_out, *, stream=None) -> None:
    M, K = h.shape
    _check("fp8q_naive_act", naive_lib().fp8q_naive_act(
        _ptr(h, 2 * M * K, "h"), M, K, act, _ptr(act_out, 2 * M * K, "act_out"), _stream(stream)))


def fp8q_naive_amax(x, amax_out, *, stream=None) -> None:
    n = x.numel()
    _check("fp8q_naive_amax", naive_lib().fp8q_naive_amax(
        _ptr(x, 2 * n, "x"), n, _ptr(amax_out, 4, "amax_out"), _stream(stream)))


def fp8q_naive_cast(x, fmt: int, amax, margin: float, q_out, *, scale_out=None, stream=None) -> None:
    n = x.numel()
    _check("fp8q_naive_cast", naive_lib().fp8q_naive_cast(
        _ptr(x, 2 * n, "x"), n, fmt, _ptr(amax, 4, "amax"), float(margin),
        _ptr(scale_out, 4, "scale_out"), _ptr(q_out, n, "q_out"), _stream(stream)))


# -- test and tuning hooks (include/fp8q_testing.h): process-wide, not for use in programs --
def fp8q_gemm_set_tile(pair: int, bn: int = 0) -> None:
    """Pin the GEMM tile shape (pair -1 = automatic, 0 = 1-CTA, 1 = 2-SM pair)."""
    _check("fp8q_gemm_set_tile", lib().fp8q_gemm_set_tile(pair, bn))


def fp8q_gemm_test_hold_loads(on: bool) -> None:
    """Failure-path test hook: later GEMMs issue no loads and report FP8Q_DEV_TIMEOUT."""
    lib().fp8q_gemm_test_hold_loads(1 if on else 0)


def fp8q_mx_set_tile(pair: int, bn: int = 0) -> None:
    """Pin fp8_gemm_mx's tile: pair 0/1, width 128 or 256; (0, 0) = automatic."""
    _check("fp8q_mx_set_tile", lib().fp8q_mx_set_tile(int(pair), int(bn)))


def fp8q_test_set_fused_grid(ctas: int) -> None:
    """Launch the one-launch step kernels with this many CTAs (0 = one per SM)."""
    _check("fp8q_test_set_fused_grid", lib().fp8q_test_set_fused_grid(int(ctas)))


def fp8q_test_set_fused_layout(layout: int) -> None:
    """Pin the one-launch step's quantize layout (1 quantize-first, 2 GEMM-first, 0 = by N)."""
    _check("fp8q_test_set_fused_layout", lib().fp8q_test_set_fused_layout(int(layout)))


def fp8q_test_gemm_tile(M: int, N: int, fused: bool) -> tuple:
    """(pair, bn): the tile the one-launch step (fused) or fp8_gemm_fwd takes at M x N."""
    pair, bn = ctypes.c_int(0), ctypes.c_int(0)
    _check("fp8q_test_gemm_tile", lib().fp8q_test_gemm_tile(int(M), int(N), 1 if fused else 0, ctypes.byref(pair),
                                                           ctypes.byref(bn)))
    return pair.value, bn.value


def fp8q_test_noalloc_fill(byte: int, stream=None) -> None:
    """Fill the no-allocation entry's static counter array with a byte value."""
    _check("fp8q_test_noalloc_fill", lib().fp8q_test_noalloc_fill(int(byte), _stream(stream)))


def version() -> int:
    return lib().fp8q_version()
