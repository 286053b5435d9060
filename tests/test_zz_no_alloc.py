"""mpgemm_run_noalloc: the GEMM for callers that cannot allocate.

Some callers may not allocate device memory when they call the GEMM (code
running inside another component's fixed memory budget, or on a path that
runs when device memory is already exhausted) and cannot own a handle. For them the
library exports one entry point that allocates nothing: operands that need
an aligned staging copy are staged into a fixed 16 MiB device array owned
by the library. These tests call it through the C ABI and check its output
against mpgemm_run's on the same inputs, within the parity tolerance
|err| <= 1e-3 * sum_k |A_ik B_kj| + 1e-5, on calls made one after another
(the shared scratch keeps the previous call's contents).

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import device_operands, reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    import mixed_precision_dense_gb300 as m
    m.build()
    m.load()
    return m


def _both(mp, ops):
    """(C from mpgemm_run, C from mpgemm_run_noalloc) as [M, N] float64 arrays."""
    s = torch.cuda.current_stream()
    d1 = device_operands(ops)
    d2 = device_operands(ops)
    with mp.Handle() as h:
        h.run(ops.M, ops.N, ops.K, ops.alpha, d1["a_ptr"], ops.lda, d1["b_ptr"], ops.ldb, ops.beta,
              d1["c_ptr"], ops.ldc, s.cuda_stream)
        st = mp.run_noalloc(ops.M, ops.N, ops.K, ops.alpha, d2["a_ptr"], ops.lda, d2["b_ptr"],
                            ops.ldb, ops.beta, d2["c_ptr"], ops.ldc, s.cuda_stream)
        assert st == mp.Status.OK
        s.synchronize()
        assert h.sync_status(s.cuda_stream)[0] == mp.Status.OK

    def view(d):
        buf = d["c_buf"].cpu().numpy()
        start = d["c_start"]
        return buf[start:start + ops.M * ops.ldc].reshape(ops.M, ops.ldc)[:, :ops.N].astype(np.float64)

    return view(d1), view(d2)


def test_noalloc_matches_run_on_consecutive_calls(mp):
    cases = [
        # lda = 617 halves: A is read in row classes, no scratch needed
        workloads.workload_operands(0),
        # ldb = 259 halves: B goes through the scratch area; beta != 0, another shape
        workloads.make_operands(321, 257, 617, lda=620, ldb=259, ldc=260, alpha=1.5, beta=0.5,
                                c_dist="normal", seed=123),
        # aligned operands: no scratch at all
        workloads.make_operands(256, 512, 320, seed=124),
        # N = 300 over 122 row blocks, odd lda: one 320-wide tile column, A in row classes
        workloads.make_operands(15616, 300, 1000, lda=1001, ldc=303, alpha=1.25, beta=0.5,
                                c_dist="normal", seed=125),
    ]
    assert mp.plan(15616, 300, 1000, 1.25, 1 << 20, 1001, 1 << 30, 300, 0.5, 1 << 34, 303)["tile_n"] == 320
    for ops in cases:
        via_run, via_noalloc = _both(mp, ops)
        _, S = reference(ops)
        tol = oracle.tolerance(S)
        assert np.all(np.abs(via_noalloc - via_run) <= tol), f"{ops.M}x{ops.N}x{ops.K}"
        assert not np.isnan(via_noalloc).any()


def test_noalloc_rejects_staging_beyond_its_scratch(mp):
    # B needs staging (ldb = 2049 halves) and its aligned copy would take
    # 4200 * 2056 * 2 bytes > 16 MiB: rejected, nothing enqueued, C untouched.
    M, N, K = 64, 2049, 4200
    assert K * ((N + 7) // 8 * 8) * 2 > mp.NOALLOC_SCRATCH_BYTES
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    st = mp.run_noalloc(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N,
                        s.cuda_stream)
    assert st == mp.Status.ERR_SCRATCH_LIMIT
    s.synchronize()
    assert bool((C == 7.0).all())
