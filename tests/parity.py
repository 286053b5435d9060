"""Parity helpers: run the CUDA library through its C ABI on seeded operands
and compare element by element with the CPU oracle.

Acceptance per element (the project's stated bound):
    |C_gpu - C_ref| <= 1e-3 * S + 1e-5,   S = sum_k |A_ik * B_kj|
plus: no NaN in the checked output, padding columns of C beyond N untouched,
and guard rows above and below C untouched (canaries).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

CANARY = 12345.0  # float32 guard value, exact


def device_operands(ops: workloads.Operands, *, a_offset=0, b_offset=0, c_offset=0, guard_rows=2,
                    poison=True):
    """Copy host operands to the GPU inside larger buffers.

    Each operand sits `guard_rows` rows below the start of its buffer and
    `offset` elements past a row boundary, so the kernel sees a base address
    that is not 16-byte aligned when offset != 0. C's guard rows and its own
    storage start as CANARY / NaN (beta == 0) or the seeded C (beta != 0).
    """
    dev = torch.device("cuda")
    M, N, K = ops.M, ops.N, ops.K

    def place(t, rows, ld, offset, fill):
        total = (rows + 2 * guard_rows) * ld + 2 * offset + 8
        buf = torch.full((total,), fill, dtype=t.dtype, device=dev)
        start = guard_rows * ld + offset
        if rows * ld:
            buf[start:start + rows * ld] = t.reshape(-1).to(dev)
        return buf, start

    a_buf, a_start = place(ops.A, M, ops.lda, a_offset, 0.0)
    b_buf, b_start = place(ops.B, N if ops.b_col_major else K, ops.ldb, b_offset, 0.0)
    c_src = ops.C
    if ops.beta == 0 and poison:
        c_src = torch.full_like(ops.C, float("nan"))
    c_buf, c_start = place(c_src, M, ops.ldc, c_offset, CANARY)
    return dict(a_buf=a_buf, a_ptr=a_buf.data_ptr() + 2 * a_start,
                b_buf=b_buf, b_ptr=b_buf.data_ptr() + 2 * b_start,
                c_buf=c_buf, c_ptr=c_buf.data_ptr() + 4 * c_start, c_start=c_start,
                c_src=c_src)


def run_gpu(handle, ops, *, a_offset=0, b_offset=0, c_offset=0, stream=None):
    d = device_operands(ops, a_offset=a_offset, b_offset=b_offset, c_offset=c_offset)
    s = torch.cuda.current_stream() if stream is None else stream
    with torch.cuda.stream(s):
        if ops.b_col_major:
            from mixed_precision_dense_gb300 import BLayout
            handle.run_ex(BLayout.COL_MAJOR, ops.M, ops.N, ops.K, ops.alpha, d["a_ptr"], ops.lda,
                          d["b_ptr"], ops.ldb, ops.beta, d["c_ptr"], ops.ldc, s.cuda_stream)
        else:
            handle.run(ops.M, ops.N, ops.K, ops.alpha, d["a_ptr"], ops.lda, d["b_ptr"], ops.ldb,
                       ops.beta, d["c_ptr"], ops.ldc, s.cuda_stream)
    s.synchronize()
    st, info = handle.sync_status(s.cuda_stream)
    assert st == 0, f"device reported {st} {info}"
    return d


def c_result(d, ops):
    """(C as [M, N] float64 numpy, the whole C buffer as float32 numpy)."""
    buf = d["c_buf"].cpu().numpy()
    start = d["c_start"]
    full = buf[start:start + ops.M * ops.ldc].reshape(ops.M, ops.ldc) if ops.M else np.zeros((0, ops.ldc), np.float32)
    return full[:, :ops.N].astype(np.float64), buf, full


def check_guards(d, ops, buf, full):
    start = d["c_start"]
    assert np.all(buf[:start] == CANARY), "write before C"
    assert np.all(buf[start + ops.M * ops.ldc:] == CANARY), "write after C"
    if ops.ldc > ops.N and ops.M:
        pad = full[:, ops.N:]
        if ops.beta == 0:
            assert np.all(np.isnan(pad)), "write into the padding of C"
        else:
            src = d["c_src"].cpu().numpy()[:, ops.N:]
            assert np.array_equal(np.isnan(pad), np.isnan(src)), "write into the padding of C"


def reference(ops, I=None, J=None):
    A, B, C = ops.bits("A"), ops.bits("B"), ops.bits("C")
    if I is None:
        return oracle.gemm(ops.M, ops.N, ops.K, ops.alpha, A, ops.lda, B, ops.ldb, ops.beta, C, ops.ldc,
                           b_col_major=ops.b_col_major)
    return oracle.elements(ops.M, ops.N, ops.K, ops.alpha, A, ops.lda, B, ops.ldb, ops.beta, C,
                           ops.ldc, I, J, b_col_major=ops.b_col_major)


def assert_close(got, ref, S, what=""):
    err = np.abs(got - ref)
    tol = oracle.tolerance(S)
    bad = ~(err <= tol)   # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first "
                             f"{[(tuple(int(x) for x in i), float(got[tuple(i)]), float(ref[tuple(i)])) for i in idx]}")
    return float(np.max(err / tol)) if err.size else 0.0


def check_full(handle, ops, *, exact=False, **kw):
    d = run_gpu(handle, ops, **kw)
    got, buf, full = c_result(d, ops)
    check_guards(d, ops, buf, full)
    ref, S = reference(ops)
    if exact:
        assert np.array_equal(got, ref), "integer case must match bit for bit"
        return 0.0
    return assert_close(got, ref, S, f"{ops.M}x{ops.N}x{ops.K}")


def check_sampled(handle, ops, I, J, **kw):
    d = run_gpu(handle, ops, **kw)
    got_all, buf, full = c_result(d, ops)
    check_guards(d, ops, buf, full)
    assert not np.isnan(got_all).any(), "NaN in C"
    ref, S = reference(ops, I, J)
    return assert_close(got_all[I, J], ref, S, f"{ops.M}x{ops.N}x{ops.K} sampled")
