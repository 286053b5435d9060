"""mpgemm_run_noalloc: the GEMM for callers that cannot allocate.

Some callers may not allocate device memory when they call the GEMM (code
running inside another component's fixed memory budget, or on a path that
runs when device memory is already exhausted) and cannot own a handle. For
them the library exports one entry point that allocates nothing: a B whose
rows break the 16-byte rule is staged into a fixed 16 MiB device array owned
by the library (an unaligned A never needs a copy there: it is read in row
classes). These tests call it through the C ABI and check its output
against the CPU oracle, within the parity tolerance
|err| <= 1e-3 * sum_k |A_ik B_kj| + 1e-5 (bit for bit for exact small
integers), each case twice in a row: the shared scratch keeps the previous
call's contents, and the status words at its start must be cleared.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import c_result, check_guards, device_operands, reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    import mixed_precision_dense_gb300 as m
    m.build()
    m.load()
    return m


def _noalloc(mp, ops):
    """C from mpgemm_run_noalloc (NaN-poisoned C when beta == 0) as an
    [M, N] float64 array; C's guard rows and padding are checked too."""
    s = torch.cuda.current_stream()
    d = device_operands(ops)
    st = mp.run_noalloc(ops.M, ops.N, ops.K, ops.alpha, d["a_ptr"], ops.lda, d["b_ptr"], ops.ldb, ops.beta,
                        d["c_ptr"], ops.ldc, s.cuda_stream)
    assert st == mp.Status.OK
    s.synchronize()
    got, buf, full = c_result(d, ops)
    check_guards(d, ops, buf, full)
    return got


CASES = [
    # (operands, exact): lda = 617 halves, A in row classes, split K: no scratch
    (lambda: workloads.workload_operands(0), False),
    # ldb = 259 halves: B goes through the scratch area; beta != 0
    (lambda: workloads.make_operands(321, 257, 617, lda=620, ldb=259, ldc=260, alpha=1.5, beta=0.5,
                                     c_dist="normal", seed=123), False),
    # aligned operands, 8 tiles of 16 k-blocks: split K with TMA reduce-adds
    (lambda: workloads.make_operands(500, 256, 1024, seed=124), False),
    # exact integers, staged B (ldb = 1030), A in 4 row classes
    (lambda: workloads.make_operands(700, 1023, 900, lda=906, ldb=1030, dist="int3", dist_b="int2",
                                     seed=126), True),
    # 2560 x 2048 x 700 with lda = 703: 256 x 256 CTA pairs reading A in row classes
    (lambda: workloads.make_operands(2560, 2048, 700, lda=703, alpha=-0.75, beta=0.25, c_dist="normal",
                                     seed=127), False),
    # N = 300 over 122 row blocks, odd lda: one 320-wide tile column, A in row classes
    (lambda: workloads.make_operands(15616, 300, 1000, lda=1001, ldc=303, alpha=1.25, beta=0.5,
                                     c_dist="normal", seed=125), False),
]


def test_noalloc_paths_planned_as_described(mp):
    plan = lambda ops: mp.plan(ops.M, ops.N, ops.K, ops.alpha, 256, ops.lda, 256, ops.ldb, ops.beta, 256, ops.ldc)
    p = [plan(make()) for make, _ in CASES]
    assert p[0]["a_classes"] == 8 and p[0]["k_splits"] > 1 and p[0]["workspace_bytes"] == 0
    assert p[1]["stage_b"] == 1 and p[1]["workspace_bytes"] > 0
    assert p[2]["a_classes"] == 0 and p[2]["k_splits"] > 1 and p[2]["workspace_bytes"] == 0
    assert p[3]["stage_b"] == 1 and p[3]["a_classes"] == 4
    assert (p[4]["tile_m"], p[4]["tile_n"]) == (256, 256) and p[4]["a_classes"] == 8
    assert p[5]["tile_n"] == 320
    assert all(x["stage_a"] == 0 for x in p)


@pytest.mark.parametrize("index", range(len(CASES)))
def test_noalloc_matches_oracle_on_consecutive_calls(mp, index):
    make, exact = CASES[index]
    ops = make()
    ref, S = reference(ops)
    for _ in range(2):
        got = _noalloc(mp, ops)
        if exact:
            assert np.array_equal(got, ref)
        else:
            assert np.all(np.abs(got - ref) <= oracle.tolerance(S)), f"{ops.M}x{ops.N}x{ops.K}"


def test_noalloc_scratch_limit_boundary(mp):
    # B needs staging (ldb = 1021 halves): K = 8192 rows of 1024 halves fill
    # the 16 MiB scratch exactly and run; one more row of K is rejected with
    # nothing enqueued and C untouched
    M, N = 64, 1021
    assert 8192 * 1024 * 2 == mp.NOALLOC_SCRATCH_BYTES
    ops = workloads.make_operands(M, N, 8192, dist="int3", dist_b="int2", seed=128)
    assert mp.plan(M, N, 8192, 1.0, 256, 8192, 256, N, 0.0, 256, N)["workspace_bytes"] == mp.NOALLOC_SCRATCH_BYTES
    ref, _ = reference(ops)
    assert np.array_equal(_noalloc(mp, ops), ref)
    K = 8193
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    st = mp.run_noalloc(M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N, s.cuda_stream)
    assert st == mp.Status.ERR_SCRATCH_LIMIT
    s.synchronize()
    assert bool((C == 7.0).all())
    # and the next call still runs
    assert np.array_equal(_noalloc(mp, ops), ref)
