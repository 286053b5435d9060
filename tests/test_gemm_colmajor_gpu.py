"""Column-major B ("Day 80, Capstone 4: a tensor-core GEMM", "Independent
gate": solve() takes A row-major, B column-major, C row-major): the gate's
cases through mpgemm_solve, and mpgemm_run_ex with a column-major B over
ragged shapes, strides, alpha/beta and every tile shape, each compared with
the CPU oracle element by element (bitwise for exact small integers)."""
import random

import numpy as np
import pytest
import torch

import workloads
from parity import assert_close, check_full, check_sampled, reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    import mixed_precision_dense_gb300 as m
    m.build()
    m.load()
    return m


GATE = [  # name, m, n, k, inputs, check
    ("unit", 16, 16, 16, "int", "bitwise"),
    ("onefrag", 16, 8, 16, "int", "bitwise"),
    ("small", 128, 128, 128, "uniform", "tolerance"),
    ("odd", 611, 613, 617, "uniform", "tolerance"),
    ("skinny", 4096, 16, 4096, "uniform", "tolerance"),
    ("square", 1024, 1024, 1024, "normal", "tolerance"),
    ("adversarial", 256, 256, 256, "edge", "tolerance"),
    ("perf", 4096, 4096, 4096, "uniform", "sampled"),
]


def gate_operands(m, n, k, inputs, seed):
    if inputs == "int":
        return workloads.make_operands(m, n, k, dist="int3", dist_b="int2", seed=seed, b_col_major=True)
    return workloads.make_operands(m, n, k, dist=inputs, seed=seed, b_col_major=True)


@pytest.mark.parametrize("name,m,n,k,inputs,check", GATE, ids=[g[0] for g in GATE])
def test_gate_through_solve(mp, name, m, n, k, inputs, check):
    ops = gate_operands(m, n, k, inputs, seed=300 + m + n + k)
    dev = torch.device("cuda")
    A = ops.A.to(dev)
    B = ops.B.to(dev)                       # n rows of k: column-major B
    C = torch.full((m, n), float("nan"), dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream()
    mp.solve(A.data_ptr(), B.data_ptr(), C.data_ptr(), m, n, k, s.cuda_stream)
    s.synchronize()
    got = C.cpu().double().numpy()
    if check == "sampled":
        I, J = workloads.sample_indices(m, n, 20000, seed=301)
        ref, S = reference(ops, I, J)
        assert not np.isnan(got).any()
        assert_close(got[I, J], ref, S, name)
        return
    ref, S = reference(ops)
    if check == "bitwise":
        assert np.array_equal(got, ref), f"{name}: integer case must match bit for bit"
    else:
        assert_close(got, ref, S, name)


CM_SHAPES = [(1, 1, 1), (17, 15, 65), (129, 257, 63), (200, 136, 617), (1000, 800, 1200),
             (513, 1025, 300)]


@pytest.mark.parametrize("tile_m,tile_n", [(0, 0), (128, 128), (128, 256), (128, 320), (256, 0), (256, 512)])
@pytest.mark.parametrize("M,N,K", CM_SHAPES)
def test_run_ex_column_major(mp, tile_m, tile_n, M, N, K):
    ops = workloads.make_operands(M, N, K, alpha=1.5, beta=0.5, c_dist="normal", seed=M * 7 + N + K,
                                  b_col_major=True)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, tile_m)
        h.set_option(mp.Option.TILE_N, tile_n)
        check_full(h, ops)


@pytest.mark.parametrize("delta", [0, 1, 3, 8])
def test_column_major_ldb_sweep_and_misalignment(mp, delta):
    # ldb = K + delta halves: unaligned pitches go through the staging copy
    ops = workloads.make_operands(300, 200, 150, ldb=150 + delta, beta=0.25, c_dist="normal",
                                  seed=310 + delta, b_col_major=True)
    with mp.Handle() as h:
        check_full(h, ops)
        check_full(h, ops, b_offset=1)      # base 2 bytes past a 16-byte boundary


def test_column_major_integer_bitwise_pair_and_persistence(mp):
    ops = workloads.make_operands(700, 900, 1024, dist="int3", dist_b="int2", seed=320, b_col_major=True)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.MAX_CTAS, 4)
        check_full(h, ops, exact=True)


def test_column_major_large_sampled(mp):
    ops = workloads.make_operands(4096, 4096, 2048, dist="normal_0.5", seed=321, b_col_major=True)
    I, J = workloads.sample_indices(4096, 4096, 20000, seed=322)
    with mp.Handle() as h:
        check_sampled(h, ops, I, J)


def test_column_major_matches_row_major_bitwise(mp):
    # same values of B in both layouts, same tile shape, A read the same way
    # (K = 512: aligned rows, one plain tensor map): identical sums
    rm = workloads.make_operands(384, 320, 512, seed=330)
    cm = workloads.make_operands(384, 320, 512, seed=330, b_col_major=True)
    from parity import run_gpu, c_result
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, 128)
        h.set_option(mp.Option.SPLIT_K, 1)      # no atomics: a fixed summation order
        g1, _, _ = c_result(run_gpu(h, rm), rm)
        g2, _, _ = c_result(run_gpu(h, cm), cm)
    assert np.array_equal(g1, g2)


def test_solve_from_several_host_threads(mp):
    # mpgemm_solve shares one handle per device; host threads may call it at
    # the same time (the library serialises them while it enqueues). Eight
    # threads, three calls each, different shapes (some with a ragged K whose
    # B needs an aligned staging copy), all on one stream; every result is
    # checked against the oracle.
    import threading
    s = torch.cuda.current_stream()
    jobs = []
    for t in range(8):
        for c in range(3):
            m, n, k = 64 + 37 * t, 48 + 29 * c, 96 + 61 * (t + c) + (t % 2)
            ops = gate_operands(m, n, k, "int", seed=500 + 10 * t + c)
            A = ops.A.cuda()
            B = ops.B.cuda()
            C = torch.full((m, n), float("nan"), device="cuda")
            jobs.append((t, ops, A, B, C))
    errors = []

    def worker(t):
        try:
            for (tt, ops, A, B, C) in jobs:
                if tt == t:
                    mp.solve(A.data_ptr(), B.data_ptr(), C.data_ptr(), ops.M, ops.N, ops.K, s.cuda_stream)
        except Exception as e:   # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(8)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    s.synchronize()
    for (_, ops, A, B, C) in jobs:
        ref, _ = reference(ops)
        assert np.array_equal(C.cpu().double().numpy(), ref)
