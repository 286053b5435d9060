"""ctypes binding for libmpgemm (include/mpgemm.h). Argument marshalling only:
every step of the GEMM runs in the library's CUDA kernels.

The library must have been built (``mixed_precision_dense_gb300.build``);
loading fails loudly otherwise. There is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import enum
import os
import re
import threading

from .build import LIB_PATH, ROOT


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_VALUE = 1
    ERR_UNSUPPORTED_DEVICE = 2
    ERR_ALLOC = 3
    ERR_LAUNCH = 4
    ERR_DEVICE_TIMEOUT = 5
    ERR_CUDA = 6
    ERR_SCRATCH_LIMIT = 7


class Option(enum.IntEnum):
    TILE_N = 1
    MAX_CTAS = 2
    FORCE_STAGING = 3
    WAIT_LIMIT_US = 4
    RASTER_GROUP = 5
    TEST_STALL = 6
    TILE_M = 7
    L2_KEEP = 8
    SPLIT_K = 9
    C_STORE = 10
    ACCUMULATOR = 11
    REPRODUCIBLE = 12
    STREAM_K = 13
    SPLIT_REDUCE = 14


class BLayout(enum.IntEnum):
    ROW_MAJOR = 0   # (k, j) at B[k*ldb + j]
    COL_MAJOR = 1   # (k, j) at B[j*ldb + k]


class MpgemmError(RuntimeError):
    def __init__(self, status, where):
        self.status = Status(status)
        super().__init__(f"{where}: {self.status.name} ({status_string(status)})")


class Plan(ctypes.Structure):
    _fields_ = [("quick", ctypes.c_int32), ("stage_a", ctypes.c_int32), ("stage_b", ctypes.c_int32),
                ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("m_tiles", ctypes.c_int32), ("n_tiles", ctypes.c_int32),
                ("k_blocks", ctypes.c_int32), ("tiles", ctypes.c_int64), ("grid", ctypes.c_int32),
                ("raster_group", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("last_k_valid", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
                ("split_tiles", ctypes.c_int32), ("items", ctypes.c_int64),
                ("k_splits", ctypes.c_int32), ("a_classes", ctypes.c_int32), ("sk_ranges", ctypes.c_int32),
                ("split_reduce", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None
_lock = threading.Lock()


def header_functions():
    """Names of the functions include/mpgemm.h declares."""
    text = open(os.path.join(ROOT, "include", "mpgemm.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\*?\s+\**(mpgemm_[a-z_]+)\s*\(", text, re.M)))


def load(path: str = LIB_PATH):
    """Load libmpgemm.so and declare its signatures (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libmpgemm is not built ({path} missing); run "
                               "mixed_precision_dense_gb300.build.build() first")
        lib = ctypes.CDLL(path)
        i32, i64, f32, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        lib.mpgemm_create.argtypes = [ctypes.POINTER(p)]
        lib.mpgemm_destroy.argtypes = [p]
        gemm_args = [p, i64, i64, i64, f32, p, i64, p, i64, f32, p, i64, p]
        lib.mpgemm_run.argtypes = gemm_args
        lib.mpgemm_run_ex.argtypes = [p, ctypes.c_int] + gemm_args[1:]
        lib.mpgemm_solve.argtypes = [p, p, p, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t, p]
        lib.mpgemm_run_host.argtypes = gemm_args
        lib.mpgemm_run_noalloc.argtypes = gemm_args[1:]
        lib.mpgemm_sync_status.argtypes = [p, p, ctypes.POINTER(i32)]
        lib.mpgemm_set_option.argtypes = [p, ctypes.c_int, i64]
        lib.mpgemm_plan.argtypes = [i64, i64, i64, f32, p, i64, p, i64, f32, p, i64,
                                    i32, i32, i32, i32, i32, i32, ctypes.POINTER(Plan)]
        lib.mpgemm_plan_call.argtypes = [p, ctypes.c_int, i64, i64, i64, f32, p, i64, p, i64, f32, p, i64,
                                         ctypes.POINTER(Plan)]
        lib.mpgemm_probe_mma_rate.argtypes = [i32, i32, p, p]
        lib.mpgemm_status_string.restype = ctypes.c_char_p
        lib.mpgemm_status_string.argtypes = [ctypes.c_int]
        for name in ("mpgemm_create", "mpgemm_destroy", "mpgemm_run", "mpgemm_run_ex", "mpgemm_solve",
                     "mpgemm_run_host", "mpgemm_run_noalloc",
                     "mpgemm_sync_status", "mpgemm_set_option", "mpgemm_plan", "mpgemm_plan_call",
                     "mpgemm_probe_mma_rate"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status) -> str:
    return load().mpgemm_status_string(int(status)).decode()


def _check(status, where):
    if status != Status.OK:
        raise MpgemmError(status, where)


def plan(M, N, K, alpha=1.0, A=0, lda=None, B=0, ldb=None, beta=0.0, C=0, ldc=None, *,
         num_sms=152, tile_m=0, tile_n=0, max_ctas=0, force_staging=False,
         b_col_major=False) -> dict:
    """Host-only description of what mpgemm_run(_ex) would do (addresses as ints)."""
    lda = max(K, 1) if lda is None else lda
    ldb = max(K if b_col_major else N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    out = Plan()
    st = load().mpgemm_plan(M, N, K, alpha, A or None, lda, B or None, ldb, beta, C or None, ldc,
                            num_sms, tile_m, tile_n, max_ctas, int(bool(force_staging)),
                            int(bool(b_col_major)), ctypes.byref(out))
    _check(st, "mpgemm_plan")
    return out.as_dict()


def run_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> Status:
    """mpgemm_run_noalloc on device addresses (ints): the GEMM without a handle
    and without any allocation, for callers that cannot allocate; staging
    copies go to the library's fixed 16 MiB device scratch area. Returns the
    status instead of raising (ERR_SCRATCH_LIMIT when that area is too small)."""
    return Status(load().mpgemm_run_noalloc(M, N, K, alpha, A or None, lda, B or None, ldb, beta,
                                            C or None, ldc, stream or None))


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

PROBE_FLOP_PER_MMA = 2 * 128 * 256 * 16


def probe_mma_rate(ctas, mmas, out, stream=0):
    """mpgemm_probe_mma_rate: `out` is the device address (int) of 2 * ctas
    uint64 values; see the header for their meaning."""
    _check(load().mpgemm_probe_mma_rate(ctas, mmas, out or None, stream or None), "mpgemm_probe_mma_rate")


def solve(a, b, c, m, n, k, stream=0):
    """mpgemm_solve: the capstone gate's interface, C = A * B with A row-major,
    B column-major, C row-major, densely packed (device addresses as ints)."""
    _check(load().mpgemm_solve(a or None, b or None, c or None, m, n, k, stream or None),
           "mpgemm_solve")


class Handle:
    """An mpgemm handle bound to the current CUDA device."""

    def __init__(self):
        self._lib = load()
        self._h = ctypes.c_void_p()
        _check(self._lib.mpgemm_create(ctypes.byref(self._h)), "mpgemm_create")

    def close(self):
        if self._h:
            self._lib.mpgemm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, option: Option, value: int):
        _check(self._lib.mpgemm_set_option(self._h, int(option), int(value)), "mpgemm_set_option")

    def plan(self, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, b_layout=0) -> dict:
        """mpgemm_plan_call: what run_ex would do with this handle's options."""
        out = Plan()
        st = self._lib.mpgemm_plan_call(self._h, int(b_layout), M, N, K, alpha, A or None, lda, B or None,
                                        ldb, beta, C or None, ldc, ctypes.byref(out))
        _check(st, "mpgemm_plan_call")
        return out.as_dict()

    def run(self, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
        """mpgemm_run on device addresses (ints); raises MpgemmError on a bad status."""
        st = self._lib.mpgemm_run(self._h, M, N, K, alpha, A or None, lda, B or None, ldb, beta,
                                  C or None, ldc, stream or None)
        _check(st, "mpgemm_run")

    def run_ex(self, b_layout, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
        """mpgemm_run_ex: b_layout is BLayout.ROW_MAJOR or BLayout.COL_MAJOR."""
        st = self._lib.mpgemm_run_ex(self._h, int(b_layout), M, N, K, alpha, A or None, lda,
                                     B or None, ldb, beta, C or None, ldc, stream or None)
        _check(st, "mpgemm_run_ex")

    def run_status(self, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> Status:
        """mpgemm_run returning the status instead of raising."""
        return Status(self._lib.mpgemm_run(self._h, M, N, K, alpha, A or None, lda, B or None, ldb,
                                           beta, C or None, ldc, stream or None))

    def run_host(self, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
        """mpgemm_run_host on host addresses (ints)."""
        st = self._lib.mpgemm_run_host(self._h, M, N, K, alpha, A or None, lda, B or None, ldb,
                                       beta, C or None, ldc, stream or None)
        _check(st, "mpgemm_run_host")

    def sync_status(self, stream=0):
        """Synchronise `stream`; returns (Status, [code, role, block, detail])."""
        info = (ctypes.c_int32 * 4)()
        st = self._lib.mpgemm_sync_status(self._h, stream or None, info)
        return Status(st), list(info)


_default = threading.local()


def default_handle() -> Handle:
    h = getattr(_default, "handle", None)
    if h is None:
        h = Handle()
        _default.handle = h
    return h


def _torch_stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def gemm(A, B, C, alpha=1.0, beta=0.0, *, handle=None, stream=None):
    """C = alpha*A@B + beta*C in place on CUDA tensors.

    A: [M, K] float16, B: [K, N] float16, C: [M, N] float32, each with unit
    stride along its last dimension (any row pitch). Runs on the current
    torch stream unless `stream` (a torch.cuda.Stream) is given.
    """
    import torch
    if A.dtype != torch.float16 or B.dtype != torch.float16 or C.dtype != torch.float32:
        raise TypeError("A and B must be float16 and C float32")
    if A.dim() != 2 or B.dim() != 2 or C.dim() != 2:
        raise ValueError("A, B and C must be 2-D")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.numel() and (t.stride(1) != 1 or not t.is_cuda):
            raise ValueError(f"{name} must be a CUDA tensor with unit stride along dim 1")
    h = handle or default_handle()
    h.run(M, N, K, float(alpha), A.data_ptr(), max(A.stride(0), K, 1), B.data_ptr(),
          max(B.stride(0), N, 1), float(beta), C.data_ptr(), max(C.stride(0), N, 1),
          _torch_stream(stream))
    return C
