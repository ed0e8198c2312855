"""quantize_fp8_gemm_gb300 -- the forward FP8 MLP down-projection on one GB300.

The compute lives in libfp8q.so (hand-written sm_103a CUDA behind the C ABI of
include/fp8q.h).  This package is its Python face:

* ``binding``   -- ctypes wrappers with the C names (fp8_quant_fused,
                   fp8_gemm_fwd, fp8_gemm_dgrad, amax_history_update), taking
                   torch CUDA tensors for device memory and the current stream.
* ``downproj``  -- the call order and buffers of one training step with
                   delayed per-tensor (or 1x128 / 128x128 group) scales.
* ``workloads`` -- seeded synthetic inputs of the benchmark workloads.
* ``build``     -- nvcc build of libfp8q.so, in-tree.

Importing the package does not load the library; the first call does, and
raises if it has not been built.
"""
from .binding import (ACT_IDENTITY, ACT_RELU, ACT_RELU2, DEV_BAD_AMAX, DEV_TIMEOUT, E4M3, E5M2,
                      GROUP, Fp8qError, amax_history_update, fp8_gemm_dgrad, fp8_gemm_fwd,
                      fp8_quant_fused, fp8q_naive_act, fp8q_naive_amax, fp8q_naive_cast)
from .downproj import DelayedScale, Fp8DownProj

__all__ = [
    "ACT_IDENTITY", "ACT_RELU", "ACT_RELU2", "DEV_BAD_AMAX", "DEV_TIMEOUT", "E4M3", "E5M2", "GROUP",
    "Fp8qError", "amax_history_update", "fp8_gemm_dgrad", "fp8_gemm_fwd", "fp8_quant_fused",
    "fp8q_naive_act", "fp8q_naive_amax", "fp8q_naive_cast", "DelayedScale", "Fp8DownProj",
]
