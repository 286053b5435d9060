"""mixed_precision_dense_gb300: C = alpha*A*B + beta*C with FP16 A and B and
FP32 accumulation and C, on the tensor cores of one GB300 (sm_103a).

The computation lives in the CUDA library ``libmpgemm.so`` (C ABI in
``include/mpgemm.h``); this package builds it (``build``) and binds it with
ctypes (``binding``). PyTorch is only used for device memory and streams.
"""
from .binding import (BLayout, Handle, MpgemmError, Option, Plan, Status, default_handle, gemm,
                      header_functions, load, plan, probe_mma_rate, run_noalloc, solve,
                      status_string, NOALLOC_SCRATCH_BYTES, PROBE_FLOP_PER_MMA)
from .build import LIB_PATH, build

__all__ = ["BLayout", "Handle", "MpgemmError", "Option", "Plan", "Status", "default_handle", "gemm",
           "header_functions", "load", "plan", "probe_mma_rate", "run_noalloc", "solve", "status_string",
           "NOALLOC_SCRATCH_BYTES", "PROBE_FLOP_PER_MMA", "LIB_PATH", "build"]
