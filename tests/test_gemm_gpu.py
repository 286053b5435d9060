"""Parity of the CUDA library (called through its C ABI) with the CPU oracle.

Every case draws seeded operands (workloads.py), runs mpgemm_run on the GPU
with a NaN-poisoned C when beta == 0 (the poison-before-launch convention of
the "02_mixed_precision_gemm" README, "Verification"), and compares with the
oracle element by element within |err| <= 1e-3 * sum_k|A_ik B_kj| + 1e-5.
Exact small-integer inputs ("Day 72: Tensor cores with WMMA", "Why this
program calls cuBLAS twice") must match bit for bit.
"""
import random

import numpy as np
import pytest
import torch

import workloads
from parity import check_full, check_sampled, run_gpu, c_result

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    import mixed_precision_dense_gb300 as m
    m.build()
    m.load()
    return m


@pytest.fixture()
def handle(mp):
    h = mp.Handle()
    yield h
    h.close()


# --------------------------------------------------------------------------- configs

@pytest.mark.parametrize("index", [0, 1, 2])
def test_workload_every_element(handle, index):
    check_full(handle, workloads.workload_operands(index))


@pytest.mark.parametrize("index", [3, 4])
def test_workload_sampled_and_edges(handle, index):
    ops = workloads.workload_operands(index)
    I, J = workloads.workload_sample(index)
    check_sampled(handle, ops, I, J)


# --------------------------------------------------------------------------- the capstone gate shapes

GATE = [  # "Day 80, Capstone 4: a tensor-core GEMM", "Independent gate" (B row-major here)
    ("unit", 16, 16, 16, "int"), ("onefrag", 16, 8, 16, "int"),
    ("small", 128, 128, 128, "uniform"), ("odd", 611, 613, 617, "uniform"),
    ("skinny", 4096, 16, 4096, "uniform"), ("square", 1024, 1024, 1024, "normal"),
    ("adversarial", 256, 256, 256, "edge"),
]


@pytest.mark.parametrize("name,M,N,K,dist", GATE, ids=[g[0] for g in GATE])
def test_gate_cases(handle, name, M, N, K, dist):
    if dist == "int":
        ops = workloads.make_operands(M, N, K, dist="int3", dist_b="int2", seed=31)
        check_full(handle, ops, exact=True)
    else:
        ops = workloads.make_operands(M, N, K, dist=dist, seed=32)
        check_full(handle, ops)


def test_gate_perf_shape_sampled(handle):
    ops = workloads.make_operands(4096, 4096, 4096, dist="uniform", seed=33)
    I, J = workloads.sample_indices(4096, 4096, 20000, seed=34)
    check_sampled(handle, ops, I, J)


# --------------------------------------------------------------------------- ragged sizes

EDGE_SIZES = [1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 617]


@pytest.mark.parametrize("size", EDGE_SIZES)
def test_ragged_M(handle, size):
    check_full(handle, workloads.make_operands(size, 129, 65, seed=40 + size))


@pytest.mark.parametrize("size", EDGE_SIZES)
def test_ragged_N(handle, size):
    check_full(handle, workloads.make_operands(131, size, 65, seed=41 + size))


@pytest.mark.parametrize("size", EDGE_SIZES)
def test_ragged_K(handle, size):
    check_full(handle, workloads.make_operands(131, 129, size, seed=42 + size))


def test_random_ragged_triples(handle):
    rng = random.Random(2024)
    for _ in range(40):
        M, N, K = (rng.choice(EDGE_SIZES) for _ in range(3))
        check_full(handle, workloads.make_operands(M, N, K, seed=rng.randint(0, 10 ** 6)))


def test_integer_inputs_bitwise_large_k(handle):
    # partial sums are integers of magnitude <= 6 * 2048 = 12,288: exact in FP32
    ops = workloads.make_operands(300, 520, 2048, dist="int3", dist_b="int2", seed=7)
    check_full(handle, ops, exact=True)


# --------------------------------------------------------------------------- strides and alignment

@pytest.mark.parametrize("delta", range(0, 9))
def test_leading_dimension_sweep(handle, delta):
    M, N, K = 150, 200, 300
    ops = workloads.make_operands(M, N, K, lda=K + delta, ldb=N + delta, ldc=N + delta,
                                  beta=0.5, c_dist="normal", seed=50 + delta)
    check_full(handle, ops)


@pytest.mark.parametrize("which", ["a", "b", "c", "abc"])
def test_misaligned_base_pointers(handle, which):
    ops = workloads.make_operands(200, 136, 256, beta=1.0, c_dist="normal", seed=60)
    kw = {}
    if "a" in which:
        kw["a_offset"] = 1   # 2 bytes past a 16-byte boundary
    if "b" in which:
        kw["b_offset"] = 3
    if "c" in which:
        kw["c_offset"] = 1   # 4 bytes
    check_full(handle, ops, **kw)


# --------------------------------------------------------------------------- alpha, beta and quick returns

def test_beta_zero_never_reads_nan_c(handle):
    ops = workloads.make_operands(333, 444, 555, alpha=2.0, beta=0.0, seed=70)
    check_full(handle, ops)  # C is NaN-poisoned before the launch


@pytest.mark.parametrize("alpha,beta", [(1.0, 1.0), (1.5, -0.5), (-2.0, 0.25), (0.0, 0.5),
                                        (0.0, 0.0), (3.0, 1.0)])
def test_alpha_beta(handle, alpha, beta):
    ops = workloads.make_operands(257, 129, 200, alpha=alpha, beta=beta, c_dist="normal", seed=71)
    check_full(handle, ops)


def test_k_zero_scales_c(handle):
    ops = workloads.make_operands(100, 60, 0, alpha=1.0, beta=0.5, c_dist="normal", seed=72)
    check_full(handle, ops)


def test_empty_m_and_n(handle):
    for (M, N) in [(0, 10), (10, 0)]:
        ops = workloads.make_operands(M, N, 32, beta=0.0, seed=73)
        d = run_gpu(handle, ops)
        got, buf, full = c_result(d, ops)
        assert got.size == 0


# --------------------------------------------------------------------------- kernel configurations

@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("max_ctas", [0, 1, 3])
def test_tile_width_and_persistence(mp, tile_n, max_ctas):
    # few CTAs walk many tiles: both accumulator buffers and every ring phase wrap
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, tile_n)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        check_full(h, workloads.make_operands(700, 600, 450, beta=1.0, c_dist="normal", seed=80))


WIDE_ONE_CTA = [  # (M, N, K, lda, ldb, ldc, beta, max_ctas): 128 x 320 tiles (parts of 256 and 64 columns)
    (640, 257, 333, 335, 264, 257, 0.0, 0),     # odd lda (row classes), a one-column second part
    (1000, 300, 700, 700, 300, 301, 0.5, 2),    # two CTAs walk 8 tiles: the one accumulator and the ring wrap
    (1000, 641, 129, 129, 648, 641, 1.0, 0),    # three tile columns, the last one a single column
    (129, 320, 65, 72, 320, 320, -0.5, 3),      # the full 256 + 64 columns, ragged rows, two k-blocks
    (700, 1000, 450, 450, 1000, 1000, 0.0, 5),  # 320-wide tiles across a wide N
]


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,beta,max_ctas", WIDE_ONE_CTA)
def test_one_cta_320_wide_tiles(mp, M, N, K, lda, ldb, ldc, beta, max_ctas):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, 320)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        ops = workloads.make_operands(M, N, K, lda=lda, ldb=ldb, ldc=ldc, alpha=1.25, beta=beta,
                                      c_dist="normal" if beta else "zeros", seed=M + 3 * N + K)
        check_full(h, ops)


@pytest.mark.parametrize("split_k", [1, 3])
def test_one_cta_320_integer_bitwise(mp, split_k):
    # the planner's own choice at N = 300 (one wave of 320-wide tiles), and forced split-K
    ops = workloads.make_operands(19456, 300, 1000, dist="int3", dist_b="int2", seed=86 + split_k)
    with mp.Handle() as h:
        h.set_option(mp.Option.SPLIT_K, split_k)
        assert mp.plan(19456, 300, 1000, A=1 << 20, B=1 << 30, C=1 << 34)["tile_n"] == 320
        check_full(h, ops, exact=True)


PAIR_SHAPES = [  # (M, N, K): one pair tile, ragged in every dimension, many tiles
    (256, 256, 64), (256, 256, 192), (200, 136, 617), (300, 500, 700), (511, 257, 129),
    (1024, 768, 1000), (257, 1025, 65), (1000, 800, 1200),
]


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
def test_cta_pair_tiles(mp, M, N, K):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        check_full(h, workloads.make_operands(M, N, K, beta=0.75, c_dist="normal", seed=M + N + K))


def test_cta_pair_integer_bitwise(mp):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        ops = workloads.make_operands(512, 512, 1024, dist="int3", dist_b="int2", seed=83)
        check_full(h, ops, exact=True)


@pytest.mark.parametrize("max_ctas", [2, 6])
def test_cta_pair_persistence_and_staging(mp, max_ctas):
    # few pairs walk many tiles; unaligned lda, ldb and ldc go through staging
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        ops = workloads.make_operands(1300, 1100, 333, lda=335, ldb=1103, ldc=1101, alpha=-1.5,
                                      beta=0.5, c_dist="normal", seed=84)
        check_full(h, ops)


@pytest.mark.parametrize("tile_n", [256, 512])
def test_cta_pair_stall_reports_timeout(mp, tile_n):
    ops = workloads.make_operands(512, 512, 128, seed=85)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, tile_n)
        h.set_option(mp.Option.WAIT_LIMIT_US, 20000)
        h.set_option(mp.Option.TEST_STALL, 1)
        from parity import device_operands
        d = device_operands(ops)
        s = torch.cuda.current_stream()
        h.run(ops.M, ops.N, ops.K, 1.0, d["a_ptr"], ops.lda, d["b_ptr"], ops.ldb, 0.0, d["c_ptr"],
              ops.ldc, s.cuda_stream)
        st, info = h.sync_status(s.cuda_stream)
        assert st == mp.Status.ERR_DEVICE_TIMEOUT
        h.set_option(mp.Option.TEST_STALL, 0)
        check_full(h, ops)


WIDE_SHAPES = [  # (M, N, K): 256 x 512 pair tiles; one tile, ragged edges, many tiles
    (256, 512, 64), (256, 512, 192), (200, 136, 617), (300, 700, 700), (511, 513, 129),
    (1024, 1536, 1000), (257, 1025, 65), (1000, 800, 1200),
]


@pytest.mark.parametrize("M,N,K", WIDE_SHAPES)
def test_wide_pair_tiles(mp, M, N, K):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, 512)
        check_full(h, workloads.make_operands(M, N, K, beta=0.75, c_dist="normal", seed=M + N + K + 1))


def test_wide_pair_integer_bitwise(mp):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, 512)
        ops = workloads.make_operands(512, 1024, 1024, dist="int3", dist_b="int2", seed=86)
        check_full(h, ops, exact=True)


@pytest.mark.parametrize("max_ctas", [2, 6])
def test_wide_pair_persistence_and_staging(mp, max_ctas):
    # few pairs walk many tiles through the single accumulator buffer (both
    # of its halves wrap many phases); unaligned lda, ldb and ldc are staged
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, 512)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        ops = workloads.make_operands(1300, 1100, 333, lda=335, ldb=1103, ldc=1101, alpha=-1.5,
                                      beta=0.5, c_dist="normal", seed=87)
        check_full(h, ops)


def test_wide_pair_large_sampled(mp):
    # the workload's own recipe (N(0, 0.5^2) inputs) at 4096 x 6144 x 4096 in
    # 256 x 512 tiles, sampled
    ops = workloads.make_operands(4096, 6144, 4096, dist="normal_0.5", seed=88)
    I, J = workloads.sample_indices(4096, 6144, 20000, seed=89)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, 512)
        check_sampled(h, ops, I, J)


SPLIT_CASES = [  # (tile_m, tile_n, max_ctas, M, N, K): the last partial wave is split in halves
    (128, 256, 5, 1000, 800, 200),     # half tiles wholly past column 800 are skipped
    (128, 128, 7, 700, 600, 336),
    (256, 256, 8, 1300, 1100, 152),
    (256, 256, 10, 768, 1024, 320),
    (256, 512, 8, 1300, 1100, 152),    # 256-wide halves; the half past column 1100 is skipped
]


@pytest.mark.parametrize("tile_m,tile_n,max_ctas,M,N,K", SPLIT_CASES)
def test_split_tail_tiles(mp, tile_m, tile_n, max_ctas, M, N, K):
    set_n = tile_m == 128 or tile_n == 512
    plan = mp.plan(M, N, K, 1.0, 256, K, 256, N, 0.5, 256, N, tile_m=tile_m,
                   tile_n=tile_n if set_n else 0, max_ctas=max_ctas)
    assert plan["split_tiles"] > 0 and plan["items"] == plan["tiles"] + plan["split_tiles"]
    assert (plan["tile_m"], plan["tile_n"]) == (tile_m, tile_n)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, tile_m)
        if set_n:
            h.set_option(mp.Option.TILE_N, tile_n)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        check_full(h, workloads.make_operands(M, N, K, beta=0.5, c_dist="normal", seed=M + K))


SPLITK_CASES = [  # (M, N, K, alpha, beta, splits)
    (4096, 16, 4096, 1.0, 0.0, 0),      # the gate's skinny case: automatic split
    (1000, 800, 1200, 1.5, 1.0, 2),     # beta = 1: no pre-pass, slices add onto C
    (300, 200, 1000, -0.5, 0.25, 3),
    (129, 65, 617, 2.0, 0.0, 7),        # ragged K tail in the last slice
    (256, 300, 513, 1.0, -1.0, 5),
]


@pytest.mark.parametrize("reduce", [1, 2])
@pytest.mark.parametrize("M,N,K,alpha,beta,splits", SPLITK_CASES)
def test_split_k(mp, M, N, K, alpha, beta, splits, reduce):
    # both ways of summing the slices: into C (reduce 1, the default) and in
    # clusters through distributed shared memory (reduce 2)
    plan = mp.plan(M, N, K, alpha, 256, K, 256, N, beta, 256, N)
    if splits == 0:
        assert plan["k_splits"] > 1 and plan["split_reduce"] == 0
    with mp.Handle() as h:
        h.set_option(mp.Option.SPLIT_K, splits)
        h.set_option(mp.Option.SPLIT_REDUCE, reduce)
        hp = h.plan(M, N, K, alpha, 256, K, 256, N, beta, 256, N)
        assert hp["k_splits"] > 1 and hp["split_reduce"] == (reduce == 2)
        check_full(h, workloads.make_operands(M, N, K, alpha=alpha, beta=beta, c_dist="normal",
                                              seed=M + N + K))


@pytest.mark.parametrize("reduce", [1, 2])
def test_split_k_integer_bitwise_and_column_major(mp, reduce):
    with mp.Handle() as h:
        h.set_option(mp.Option.SPLIT_K, 4)
        h.set_option(mp.Option.SPLIT_REDUCE, reduce)
        check_full(h, workloads.make_operands(200, 300, 2048, dist="int3", dist_b="int2", seed=86),
                   exact=True)
        check_full(h, workloads.make_operands(200, 300, 2048, dist="int3", dist_b="int2", seed=87,
                                              b_col_major=True), exact=True)


CLUSTER_SPLIT_CASES = [  # (M, N, K, lda, beta, splits): slices summed in clusters
    (200, 136, 617, 617, 0.0, 0),       # the small workload: 16 tiles x 5 slices, A in 8 row classes
    (1000, 800, 1200, 1200, 1.0, 0),    # beta = 1: two slices
    (129, 65, 617, 617, 0.5, 8),        # the largest cluster, ragged rows, columns and K
    (300, 200, 1000, 1003, -0.75, 3),   # 3 slices share 128 rows (43, 43, 42), A in row classes
    (64, 1000, 4096, 4096, 0.0, 6),     # 8 tiles x 6 slices of 11 k-blocks (the last 9)
]


@pytest.mark.parametrize("M,N,K,lda,beta,splits", CLUSTER_SPLIT_CASES)
def test_cluster_split_k_identical_bits(mp, M, N, K, lda, beta, splits):
    # Against the oracle (C NaN-poisoned when beta == 0), then three calls
    # give identical bits, and exact integers match bit for bit.
    from parity import device_operands
    s = torch.cuda.current_stream()
    with mp.Handle() as h:
        h.set_option(mp.Option.SPLIT_K, splits)
        h.set_option(mp.Option.SPLIT_REDUCE, 2)
        hp = h.plan(M, N, K, 1.25, 256, lda, 256, N, beta, 256, N)
        assert hp["k_splits"] > 1 and hp["split_reduce"] == 1
        ops = workloads.make_operands(M, N, K, lda=lda, alpha=1.25, beta=beta,
                                      c_dist="normal" if beta else "zeros", seed=M + N + K + lda)
        check_full(h, ops)
        outs = []
        for _ in range(3):
            d = device_operands(ops)
            h.run(ops.M, ops.N, ops.K, ops.alpha, d["a_ptr"], ops.lda, d["b_ptr"], ops.ldb, ops.beta,
                  d["c_ptr"], ops.ldc, s.cuda_stream)
            s.synchronize()
            outs.append(d["c_buf"].cpu().numpy().view(np.uint32))
        assert all(np.array_equal(outs[0], o) for o in outs[1:])
        ints = workloads.make_operands(M, N, K, lda=lda, beta=beta, dist="int3", dist_b="int2",
                                       c_dist="int3" if beta else "zeros", seed=M + N + K + lda + 1)
        check_full(h, ints, exact=True)


def test_cluster_split_k_plan(mp):
    # Clusters are the default for reproducible calls, which split K only
    # that way (cutting more than 8 slices to 8); otherwise the slices add
    # into C. One tile of 128 k-blocks: 16 slices by the automatic rule.
    args = (128, 128, 8192, 1.0, 256, 8192, 256, 128, 0.5, 256, 128)
    assert mp.plan(*args)["k_splits"] == 16 and mp.plan(*args)["split_reduce"] == 0
    ops = workloads.make_operands(128, 128, 8192, beta=0.5, c_dist="normal", seed=77)
    with mp.Handle() as h:
        h.set_option(mp.Option.REPRODUCIBLE, 1)
        hp = h.plan(*args)
        assert (hp["k_splits"], hp["split_reduce"], hp["grid"]) == (8, 1, 8)
        check_full(h, ops)
        h.set_option(mp.Option.SPLIT_REDUCE, 1)   # reproducible without clusters: no split
        assert h.plan(*args)["k_splits"] == 1
    with mp.Handle() as h:
        h.set_option(mp.Option.SPLIT_K, 16)
        h.set_option(mp.Option.SPLIT_REDUCE, 2)   # clusters: 16 slices cut to 8
        assert (h.plan(*args)["k_splits"], h.plan(*args)["split_reduce"]) == (8, 1)
        check_full(h, ops)
        h.set_option(mp.Option.SPLIT_REDUCE, 1)   # 16 slices added into C, within the tolerance
        assert (h.plan(*args)["k_splits"], h.plan(*args)["split_reduce"]) == (16, 0)
        check_full(h, ops)


CLASS_CASES = [  # (M, N, K, lda, a_offset, tile_n, split_k): A read in row classes
    (200, 136, 617, 617, 0, 0, 0),      # 8 classes of 25 rows
    (1000, 300, 500, 503, 0, 128, 0),   # NaN padding between rows: leading columns zeroed
    (700, 257, 1000, 1002, 0, 256, 0),  # 4 classes
    (513, 200, 333, 340, 0, 0, 0),      # 2 classes
    (300, 200, 256, 256, 1, 0, 0),      # aligned pitch, base 2 bytes off: 1 class, shift 1
    (3, 50, 70, 71, 0, 0, 0),           # fewer rows than classes
    (640, 128, 2049, 2049, 3, 128, 4),  # classes with split-K
    (300, 200, 100, 109, 0, 0, 0),      # 9 NaN padding elements: every shift 1..7 lands in NaN
    (1100, 64, 300, 311, 0, 128, 0),    # 137-138 rows per class: second tiles of 9-10 rows
    # aligned pitch (a multiple of 128 bytes), base off a 16-byte boundary: one
    # class read from the 128-byte line below, shifted 40 or 63 elements (the
    # first two or three 16-wide K slices of k-block 0 not issued, 8 or 15
    # columns zeroed)
    (300, 200, 256, 256, 40 + 1, 0, 0),
    (300, 200, 256, 256, 63, 256, 0),
]


@pytest.mark.parametrize("M,N,K,lda,a_offset,tile_n,split_k", CLASS_CASES)
def test_a_row_classes(mp, M, N, K, lda, a_offset, tile_n, split_k):
    plan = mp.plan(M, N, K, 1.0, 256 + 2 * a_offset, lda, 256, N, 0.5, 256, N, tile_n=tile_n)
    assert plan["a_classes"] >= 1 and plan["stage_a"] == 0
    if lda == 256:
        assert plan["a_classes"] == 1 and plan["k_blocks"] == -(-(K + (2 * a_offset + 256) % 128 // 2) // 64)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, tile_n)
        h.set_option(mp.Option.SPLIT_K, split_k)
        ops = workloads.make_operands(M, N, K, lda=lda, alpha=1.25, beta=0.5, c_dist="normal",
                                      seed=M + lda)
        check_full(h, ops, a_offset=a_offset)
        # the same problem through the staging copy gives the same result within tolerance
        h.set_option(mp.Option.FORCE_STAGING, 1)
        check_full(h, ops, a_offset=a_offset)


def test_a_row_classes_integer_bitwise(mp):
    ops = workloads.make_operands(777, 260, 1021, lda=1021, dist="int3", dist_b="int2", seed=88)
    with mp.Handle() as h:
        check_full(h, ops, exact=True)


PAIR_CLASS_CASES = [  # (M, N, K, lda, a_offset, tile_n): A read in row classes by CTA pairs
    (600, 300, 500, 503, 0, 256),    # NaN padding between rows: both CTAs' leading columns zeroed
    (1100, 520, 333, 340, 0, 256),   # 2 classes
    (700, 257, 1000, 1002, 0, 384),  # 4 classes, 256 x 384 tiles
    (513, 700, 129, 131, 0, 512),    # 8 classes, 256 x 512 tiles, the odd CTA with few rows
    (300, 200, 256, 256, 1, 256),    # aligned pitch, base 2 bytes off: 1 class, shift 1
    (40, 300, 70, 71, 0, 256),       # 5 rows per class: the odd CTA of every pair has none
]


@pytest.mark.parametrize("M,N,K,lda,a_offset,tile_n", PAIR_CLASS_CASES)
def test_a_row_classes_cta_pairs(mp, M, N, K, lda, a_offset, tile_n):
    plan = mp.plan(M, N, K, 1.0, 256 + 2 * a_offset, lda, 256, N, 0.5, 256, N, tile_m=256,
                   tile_n=0 if tile_n == 256 else tile_n)
    assert plan["tile_m"] == 256 and plan["tile_n"] == tile_n
    assert plan["a_classes"] >= 1 and plan["stage_a"] == 0
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, 0 if tile_n == 256 else tile_n)
        ops = workloads.make_operands(M, N, K, lda=lda, alpha=1.25, beta=0.5, c_dist="normal",
                                      seed=M + lda + tile_n)
        check_full(h, ops, a_offset=a_offset)
        h.set_option(mp.Option.FORCE_STAGING, 1)
        check_full(h, ops, a_offset=a_offset)


@pytest.mark.parametrize("tile_n", [256, 384, 512])
def test_a_row_classes_cta_pairs_integer_bitwise(mp, tile_n):
    ops = workloads.make_operands(777, 520, 1021, lda=1021, dist="int3", dist_b="int2", seed=89 + tile_n)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, 0 if tile_n == 256 else tile_n)
        check_full(h, ops, exact=True)


PAIR384_SHAPES = [  # (M, N, K, lda, ldb, ldc, beta, max_ctas): 256 x 384 CTA-pair tiles
    (256, 384, 64, 64, 384, 384, 0.0, 0),       # one full tile
    (256, 257, 617, 617, 257, 257, 0.5, 0),     # one column past 256: the 128-column part
    (1000, 300, 700, 700, 300, 301, 1.0, 4),    # two pairs walk 4 tiles through the one accumulator
    (511, 600, 129, 129, 600, 600, -0.5, 0),    # second tile column 216 wide: trimmed to 256
    (1300, 1100, 333, 335, 1103, 1101, 0.75, 6),  # unaligned A (row classes), B and C staged / per lane
]


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,beta,max_ctas", PAIR384_SHAPES)
def test_cta_pair_384_wide_tiles(mp, M, N, K, lda, ldb, ldc, beta, max_ctas):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_N, 384)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        ops = workloads.make_operands(M, N, K, lda=lda, ldb=ldb, ldc=ldc, alpha=1.5, beta=beta,
                                      c_dist="normal" if beta else "zeros", seed=M + 5 * N + K)
        check_full(h, ops)
        ops = workloads.make_operands(M, N, K, lda=lda, ldb=K + 3, ldc=ldc, alpha=1.5, beta=beta,
                                      c_dist="normal" if beta else "zeros", seed=M + 5 * N + K + 1,
                                      b_col_major=True)
        check_full(h, ops)


PAIR320_SHAPES = [  # (M, N, K, lda, ldb, ldc, beta, max_ctas): 256 x 320 pair tiles, narrow last part
    (256, 320, 64, 64, 320, 320, 0.0, 0),       # one full tile
    (256, 257, 617, 617, 257, 257, 0.5, 0),     # one column past 256: the 64-column part
    (1000, 300, 700, 700, 300, 301, 1.0, 4),    # two pairs walk 4 tiles through the one accumulator
    (511, 700, 129, 129, 700, 700, -0.5, 0),    # three tile columns, the last 60 wide (one 128 unit)
    (1300, 1100, 333, 335, 1103, 1101, 0.75, 6),  # A in row classes, B staged, C per lane
    (700, 290, 1000, 1002, 290, 290, 0.0, 0),   # 4 row classes, columns 256..289 in the narrow part
]


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,beta,max_ctas", PAIR320_SHAPES)
def test_cta_pair_320_wide_tiles(mp, M, N, K, lda, ldb, ldc, beta, max_ctas):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, 320)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        ops = workloads.make_operands(M, N, K, lda=lda, ldb=ldb, ldc=ldc, alpha=1.5, beta=beta,
                                      c_dist="normal" if beta else "zeros", seed=M + 7 * N + K)
        check_full(h, ops)


def test_cta_pair_320_integer_bitwise(mp):
    # every column of the narrow part exact: 288 columns, A in 8 row classes
    ops = workloads.make_operands(777, 288, 1021, lda=1021, dist="int3", dist_b="int2", seed=90)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, 320)
        check_full(h, ops, exact=True)


PAIR288_SHAPES = [  # (M, N, K, lda, ldb, ldc, beta, max_ctas): 256 x 288 pair tiles, 32-column last part
    (256, 288, 64, 64, 288, 288, 0.0, 0),       # one full tile (TMA stores of 32 x 16 boxes)
    (700, 288, 1000, 1000, 288, 288, 0.0, 0),   # A aligned: stages of two k-blocks, TMA stores
    (1500, 280, 4096, 4096, 280, 280, 0.5, 6),  # A aligned, beta * C, three pairs walk the tiles
    (256, 257, 617, 617, 257, 257, 0.5, 0),     # one column past 256: the 32-column part, 8 row classes
    (1000, 280, 700, 700, 280, 281, 1.0, 4),    # two pairs walk 4 tiles through the staggered layouts
    (511, 700, 129, 129, 700, 700, -0.5, 0),    # three tile columns, the last 124 wide (one 128 unit)
    (1300, 1100, 333, 335, 1103, 1101, 0.75, 6),  # A in row classes, B staged, C per lane
    (16384, 270, 300, 365, 270, 270, 0.5, 0),   # A in 64 line-aligned row classes; 65 NaN halves
                                                 # between rows: every shift (up to 63) starts in NaN
]


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,beta,max_ctas", PAIR288_SHAPES)
def test_cta_pair_288_wide_tiles(mp, M, N, K, lda, ldb, ldc, beta, max_ctas):
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, 288)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        ops = workloads.make_operands(M, N, K, lda=lda, ldb=ldb, ldc=ldc, alpha=1.5, beta=beta,
                                      c_dist="normal" if beta else "zeros", seed=M + 11 * N + K)
        check_full(h, ops)


@pytest.mark.parametrize("M,N,K,lda,classes", [(777, 288, 1021, 1021, 8), (16384, 272, 515, 515, 64)])
def test_cta_pair_288_integer_bitwise(mp, M, N, K, lda, classes):
    # every column of the 32-column part exact; A in 16-byte or line-aligned row classes
    plan = mp.plan(M, N, K, 1.0, 256, lda, 256, N, 0.0, 256, N, tile_m=256, tile_n=288)
    assert plan["a_classes"] == classes
    ops = workloads.make_operands(M, N, K, lda=lda, dist="int3", dist_b="int2", seed=91 + classes)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, 288)
        check_full(h, ops, exact=True)


def test_line_aligned_classes_in_320_pairs(mp):
    # 64 row classes in 256 x 320 pairs, NaN between rows, beta * C
    plan = mp.plan(16384, 300, 300, 1.0, 256, 365, 256, 300, 0.5, 256, 300, tile_m=256, tile_n=320)
    assert plan["a_classes"] == 64
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, 320)
        check_full(h, workloads.make_operands(16384, 300, 300, lda=365, alpha=0.75, beta=0.5, c_dist="normal",
                                              seed=92))
        check_full(h, workloads.make_operands(16384, 300, 300, lda=365, dist="int3", dist_b="int2", seed=93),
                   exact=True)


@pytest.mark.parametrize("M,N,K", [(600, 100, 300), (600, 640, 300), (700, 129, 129)])
def test_cta_pair_tiles_trimmed_to_valid_columns(mp, M, N, K):
    # a pair tile's columns are cut to the 128-column units below N (N = 128
    # instructions for a 256-wide tile with at most 128 valid columns)
    for tile_n in (0, 512):
        with mp.Handle() as h:
            h.set_option(mp.Option.TILE_M, 256)
            h.set_option(mp.Option.TILE_N, tile_n)
            check_full(h, workloads.make_operands(M, N, K, beta=0.5, c_dist="normal", seed=M + N + tile_n))
            check_full(h, workloads.make_operands(M, N, K, dist="int3", dist_b="int2", seed=M + N + tile_n + 1),
                       exact=True)


@pytest.mark.parametrize("tile_n", [288, 320, 384])
def test_tall_skinny_workload_in_pairs(mp, tile_n):
    ops = workloads.workload_operands(4)
    I, J = workloads.workload_sample(4)
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, 256)
        h.set_option(mp.Option.TILE_N, tile_n)
        check_sampled(h, ops, I, J)


def test_forced_staging_matches(mp):
    with mp.Handle() as h:
        h.set_option(mp.Option.FORCE_STAGING, 1)
        check_full(h, workloads.make_operands(300, 300, 300, seed=81))


@pytest.mark.parametrize("group", [1, 2, 5, 64])
def test_raster_groups(mp, group):
    with mp.Handle() as h:
        h.set_option(mp.Option.RASTER_GROUP, group)
        h.set_option(mp.Option.MAX_CTAS, 7)
        check_full(h, workloads.make_operands(1100, 900, 130, seed=82))


def test_side_stream_and_back_to_back_shapes(handle):
    s = torch.cuda.Stream()
    for (M, N, K, seed) in [(64, 64, 64, 1), (900, 1000, 700, 2), (65, 17, 3000, 3), (64, 64, 64, 4)]:
        ops = workloads.make_operands(M, N, K, seed=90 + seed)
        d = run_gpu(handle, ops, stream=s)
        got, _, _ = c_result(d, ops)
        from parity import reference, assert_close
        ref, S = reference(ops)
        assert_close(got, ref, S)


@pytest.mark.parametrize("first,second", [((2048, 2048, 2048), (2048, 2048, 64)),
                                          ((2048, 2048, 64), (2048, 2048, 2048)),
                                          ((512, 640, 3000), (512, 640, 17))])
def test_back_to_back_dependent_calls(mp, handle, first, second):
    # The GEMM is launched with programmatic dependent launch: its CTAs may be
    # scheduled while the previous kernel still runs, and must not touch
    # memory before it has completed. C = A1 B1, then at once C = A2 B2 + C on
    # the same stream (the second call reads what the first writes), then
    # C = A3 B3 - C: integer inputs make every sum exact.
    M, N = first[0], first[1]
    s = torch.cuda.current_stream()
    ks = [first[2], second[2], first[2] // 2 + 1]
    gen = torch.Generator().manual_seed(sum(ks))
    As = [torch.randint(-3, 4, (M, k), generator=gen).half() for k in ks]
    Bs = [torch.randint(-2, 3, (k, N), generator=gen).half() for k in ks]
    dA = [a.cuda() for a in As]
    dB = [b.cuda() for b in Bs]
    C = torch.full((M, N), float("nan"), device="cuda")
    for i, beta in enumerate([0.0, 1.0, -1.0]):
        handle.run(M, N, ks[i], 1.0, dA[i].data_ptr(), ks[i], dB[i].data_ptr(), N, beta, C.data_ptr(), N,
                   s.cuda_stream)
    s.synchronize()
    assert handle.sync_status(s.cuda_stream)[0] == mp.Status.OK
    # (float64 products of these integers are exact)
    prods = [a.double().numpy() @ b.double().numpy() for a, b in zip(As, Bs)]
    ref = prods[2] - (prods[0] + prods[1])
    assert np.array_equal(C.cpu().double().numpy(), ref)


def test_offsets_beyond_32_bits(mp):
    # Maximum-size addressing: A at a pitch of 32800 halves and C at a pitch
    # of 32772 floats over 65539 rows, so their last rows start past element
    # 2^31 (4.3 GB and 8.6 GB buffers). Sampled rows at both ends and in
    # between are checked against the oracle, and C's padding columns of
    # those rows must still hold the NaN poison.
    import oracle
    M, N, K, lda, ldc = 65539, 40, 200, 32800, 32772
    assert M * lda > 2 ** 31 and M * ldc > 2 ** 31
    gen = torch.Generator().manual_seed(97)
    A = (torch.rand(M, K, generator=gen) * 2 - 1).half()
    B = (torch.rand(K, N, generator=gen) * 2 - 1).half()
    dA = torch.empty((M, lda), dtype=torch.float16, device="cuda")
    dA[:, :K] = A.cuda()
    dB = B.cuda()
    dC = torch.empty((M, ldc), device="cuda")
    s = torch.cuda.current_stream()
    rows = np.array([0, 1, 127, 128, M // 2, 65409, 65535, M - 2, M - 1], dtype=np.int64)
    I = np.repeat(rows, N)
    J = np.tile(np.arange(N, dtype=np.int64), len(rows))
    ref, S = oracle.elements(M, N, K, 1.0, A.reshape(-1).view(torch.int16).numpy().view(np.uint16), K,
                             B.reshape(-1).view(torch.int16).numpy().view(np.uint16), N, 0.0, None, N, I, J)
    for c_store in (0, 1):   # TMA stores of C, then per-lane stores
        dC.fill_(float("nan"))
        with mp.Handle() as h:
            h.set_option(mp.Option.C_STORE, c_store)
            h.run(M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), N, 0.0, dC.data_ptr(), ldc, s.cuda_stream)
            s.synchronize()
            assert h.sync_status(s.cuda_stream)[0] == mp.Status.OK
        got = dC[torch.from_numpy(rows).cuda()].cpu().numpy()
        err = np.abs(got[:, :N].astype(np.float64).reshape(-1) - ref)
        assert np.all(err <= oracle.tolerance(S)), c_store
        assert np.isnan(got[:, N:]).all(), c_store
    del dA, dC
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- tensor-core rate probe

def test_mma_rate_probe_pins_the_per_sm_rate(mp):
    # One probe CTA per SM issues back-to-back M = 128, N = 256, K = 16
    # kind::f16 MMAs: the per-SM dense FP16 rate is 1,048,576 FLOP over the
    # cycles each takes. Every CTA must finish, and the rate must be one
    # value for all SMs (the factor of the "02_mixed_precision_gemm" README's
    # peak = MACs/SM/clk x SMs x 2 x clock, measured rather than assumed).
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mmas = 1 << 14
    out = torch.zeros(2 * sms, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream()
    mp.probe_mma_rate(sms, mmas, out.data_ptr(), s.cuda_stream)
    s.synchronize()
    res = out.cpu().numpy().reshape(sms, 2)
    assert np.all(res[:, 1] == 1)
    flop_per_clk = mp.PROBE_FLOP_PER_MMA * mmas / res[:, 0]
    # (a data-sheet figure would be 8192; allow the issue overhead of the
    # first and last instruction, and nothing above the cycle count of one
    # 128 x 256 x 16 MMA per 128 cycles)
    assert 7000 < float(np.median(flop_per_clk)) <= 8192 * 1.001
    assert float(flop_per_clk.max() / flop_per_clk.min()) < 1.05


# --------------------------------------------------------------------------- host-buffer entry point

def test_run_host_matches_oracle(handle):
    ops = workloads.make_operands(321, 257, 617, lda=620, ldb=259, ldc=260, alpha=1.5, beta=0.5,
                                  c_dist="normal", seed=95)
    C = ops.C.clone()
    s = torch.cuda.current_stream()
    handle.run_host(ops.M, ops.N, ops.K, ops.alpha, ops.A.data_ptr(), ops.lda, ops.B.data_ptr(),
                    ops.ldb, ops.beta, C.data_ptr(), ops.ldc, s.cuda_stream)
    s.synchronize()
    from parity import reference, assert_close
    ref, S = reference(ops)
    assert_close(C[:, :ops.N].double().numpy(), ref, S)
    assert torch.isnan(C[:, ops.N:]).all()  # padding untouched


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_run_host_keeps_host_padding(handle, beta):
    # padding columns of the host C hold a marker that must survive the call
    ops = workloads.make_operands(97, 130, 71, lda=75, ldb=130, ldc=133, beta=beta,
                                  c_dist="normal", seed=96)
    C = ops.C.clone()
    C[:, ops.N:] = 7.25
    s = torch.cuda.current_stream()
    handle.run_host(ops.M, ops.N, ops.K, ops.alpha, ops.A.data_ptr(), ops.lda, ops.B.data_ptr(),
                    ops.ldb, ops.beta, C.data_ptr(), ops.ldc, s.cuda_stream)
    s.synchronize()
    from parity import reference, assert_close
    ref, S = reference(ops)
    assert_close(C[:, :ops.N].double().numpy(), ref, S)
    assert bool((C[:, ops.N:] == 7.25).all())


# --------------------------------------------------------------------------- bounded waits

def test_stalled_pipeline_reports_timeout_and_context_survives(mp):
    # The load warp issues nothing, so the MMA warp's bounded wait expires; the
    # kernel records the timeout and exits, and the next call works normally.
    ops = workloads.make_operands(256, 256, 128, seed=99)
    with mp.Handle() as h:
        h.set_option(mp.Option.WAIT_LIMIT_US, 20000)
        h.set_option(mp.Option.TEST_STALL, 1)
        from parity import device_operands
        d = device_operands(ops)
        s = torch.cuda.current_stream()
        h.run(ops.M, ops.N, ops.K, 1.0, d["a_ptr"], ops.lda, d["b_ptr"], ops.ldb, 0.0, d["c_ptr"],
              ops.ldc, s.cuda_stream)
        st, info = h.sync_status(s.cuda_stream)
        assert st == mp.Status.ERR_DEVICE_TIMEOUT
        assert info[0] == 1 and info[1] in (2, 3)
        st, info = h.sync_status(s.cuda_stream)   # the report is collected once
        assert st == mp.Status.OK
        h.set_option(mp.Option.TEST_STALL, 0)
        check_full(h, ops)


C_STORE_CASES = [  # (M, N, K, ldc, tile_m, tile_n): beta == 0, C rows 16-byte aligned
    (300, 260, 200, 260, 0, 0),          # ragged rows: the TMA store clips past row 300
    (257, 129, 65, 132, 128, 256),       # ragged columns: clipped past column 129, padding untouched
    (1000, 800, 1200, 804, 128, 128),
    (511, 700, 300, 704, 256, 0),        # CTA pairs, 256 x 256
    (513, 1025, 129, 1028, 256, 512),    # N % 4 != 0: per-lane stores (a TMA store would write
                                         # the rest of the last 16-byte group, into the padding)
    (513, 1028, 128, 1032, 256, 512),    # CTA pairs, 256 x 512, eight epilogue warps, partial last chunk
    (513, 1028, 128, 1032, 256, 0),
    (64, 4096, 700, 4096, 128, 256),
]


@pytest.mark.parametrize("M,N,K,ldc,tile_m,tile_n", C_STORE_CASES)
def test_tma_store_of_c_matches_per_lane_stores(mp, M, N, K, ldc, tile_m, tile_n):
    # C written by tiled TMA stores (the automatic choice here) against the
    # oracle, and bit for bit against the per-lane stores of the same sums
    # (integer inputs: the sums are exact whatever order a path adds in)
    ops = workloads.make_operands(M, N, K, ldc=ldc, alpha=1.25, dist="int3", dist_b="int2",
                                  seed=M + N + K + 5)
    outs = []
    for c_store in (0, 1):
        with mp.Handle() as h:
            h.set_option(mp.Option.TILE_M, tile_m)
            h.set_option(mp.Option.TILE_N, tile_n)
            h.set_option(mp.Option.C_STORE, c_store)
            check_full(h, ops)
            got, _, _ = c_result(run_gpu(h, ops), ops)
            outs.append(got)
    assert np.array_equal(outs[0], outs[1])


SPLIT_REDUCE_CASES = [  # (M, N, K, lda, ldc, beta, splits): split-K slices added into C
    (129, 68, 617, 624, 68, 0.0, 4),          # ragged rows and K: the reduce-add clips past row 129
    (1000, 800, 1200, 1200, 804, 1.0, 2),     # beta = 1: slices add onto C as it is
    (300, 200, 1000, 1000, 200, -0.5, 3),     # C = beta * C first, then the slices
    (4096, 16, 4096, 4096, 16, 0.0, 0),       # the gate's skinny case (automatic split)
    (1000, 128, 640, 640, 128, 0.5, 0),       # 8 tiles of 10 k-blocks: five automatic slices
    (500, 256, 1024, 1024, 256, 0.0, 0),      # 8 tiles of 16 k-blocks: four automatic slices
]


@pytest.mark.parametrize("M,N,K,lda,ldc,beta,splits", SPLIT_REDUCE_CASES)
def test_split_k_tma_reduce_matches_atomics(mp, M, N, K, lda, ldc, beta, splits):
    # split-K slices added into C by tiled TMA reduce-adds (automatic for an
    # aligned C) and by per-lane atomic adds: both against the oracle, and
    # bit for bit with integer inputs, whose partial sums are exact
    assert mp.plan(M, N, K, 1.0, 256, lda, 256, N, beta, 256, ldc)["a_classes"] == 0
    ops = workloads.make_operands(M, N, K, lda=lda, ldc=ldc, alpha=1.5, beta=beta, c_dist="normal",
                                  seed=M + K + 3)
    ints = workloads.make_operands(M, N, K, lda=lda, ldc=ldc, beta=beta, dist="int3", dist_b="int2",
                                   c_dist="int3", seed=M + K + 4)
    outs = []
    for c_store in (0, 1):
        with mp.Handle() as h:
            h.set_option(mp.Option.SPLIT_K, splits)
            h.set_option(mp.Option.C_STORE, c_store)
            check_full(h, ops)
            check_full(h, ints, exact=True)
            got, _, _ = c_result(run_gpu(h, ints), ints)
            outs.append(got)
    assert np.array_equal(outs[0], outs[1])


def test_cta_pair_256_repeats_bits_and_reproducible_option(mp):
    # The two MMA threads of a 256 x 256 CTA-pair tile take alternate
    # k-blocks and hand each one over before the other thread issues the
    # next, so the accumulator receives the k-blocks in one fixed order:
    # identical calls give identical bits. REPRODUCIBLE = 1 additionally
    # rules out split-K whose slices add into C in arrival order (slices
    # summed in clusters stay).
    from parity import device_operands
    s = torch.cuda.current_stream()

    def repeat(h, ops, n=3):
        outs = []
        for _ in range(n):
            d = device_operands(ops)
            h.run(ops.M, ops.N, ops.K, ops.alpha, d["a_ptr"], ops.lda, d["b_ptr"], ops.ldb, ops.beta,
                  d["c_ptr"], ops.ldc, s.cuda_stream)
            s.synchronize()
            outs.append(d["c_buf"].cpu().numpy().view(np.uint32))
        return all(np.array_equal(outs[0], o) for o in outs[1:])

    ops = workloads.make_operands(2560, 2048, 700, dist="normal", seed=98)
    plan = mp.plan(ops.M, ops.N, ops.K, 1.0, 256, ops.lda, 256, ops.ldb, 0.0, 256, ops.ldc)
    assert (plan["tile_m"], plan["tile_n"]) == (256, 256)
    with mp.Handle() as h:
        check_full(h, ops)
        assert repeat(h, ops)
    ops = workloads.make_operands(4096, 16, 4096, dist="normal", seed=99)
    assert mp.plan(ops.M, ops.N, ops.K, 1.0, 256, ops.lda, 256, ops.ldb, 0.0, 256, ops.ldc)["k_splits"] > 1
    for reduce in (0, 1):
        with mp.Handle() as h:
            h.set_option(mp.Option.REPRODUCIBLE, 1)
            h.set_option(mp.Option.SPLIT_REDUCE, reduce)
            check_full(h, ops)
            assert repeat(h, ops)


def test_cta_pair_256_long_k_integer_stress(mp):
    # The planner's own 256 x 256 CTA-pair choice at a long K, called 30
    # times back to back on exact small-integer inputs ("Day 72: Tensor cores
    # with WMMA", "Why this program calls cuBLAS twice": every partial sum is
    # an integer below 2^24, so any lost or doubled MMA shows as a mismatch):
    # every call's C must equal the oracle's bit for bit.
    from parity import device_operands, reference
    M, N, K = 2560, 2048, 4096
    ops = workloads.make_operands(M, N, K, dist="int3", dist_b="int2", seed=4242)
    plan = mp.plan(M, N, K, 1.0, 256, K, 256, N, 0.0, 256, N)
    assert (plan["tile_m"], plan["tile_n"]) == (256, 256)
    ref, _ = reference(ops)
    d = device_operands(ops)
    s = torch.cuda.current_stream()
    outs = []
    with mp.Handle() as h:
        for _ in range(30):
            c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
            h.run(M, N, K, 1.0, d["a_ptr"], K, d["b_ptr"], N, 0.0, c.data_ptr(), N, s.cuda_stream)
            outs.append(c)
        s.synchronize()
        assert h.sync_status(s.cuda_stream)[0] == mp.Status.OK
    for i, c in enumerate(outs):
        got = c.cpu().double().numpy()
        assert np.array_equal(got, ref), f"call {i}: {int((got != ref).sum())} elements differ"


def test_tma_store_falls_back_for_unaligned_c(mp):
    # a C base 4 bytes past a 16-byte boundary cannot be a TMA target: the
    # per-lane path writes it, guard rows and padding stay untouched
    ops = workloads.make_operands(300, 260, 200, ldc=264, seed=91)
    with mp.Handle() as h:
        check_full(h, ops, c_offset=1)
        check_full(h, ops, c_offset=2)


def test_tensor_map_cache_across_buffers_and_shapes(mp):
    # one handle, 20 different operand sets (more tensor maps than the
    # handle's 16-entry cache holds) in two rounds: every result is checked,
    # so a map reused for the wrong buffer or shape would show
    sets = [workloads.make_operands(64 + 32 * (i % 5), 96 + 16 * (i % 4), 64 * (1 + i % 3), seed=600 + i)
            for i in range(20)]
    with mp.Handle() as h:
        for _ in range(2):
            for ops in sets:
                check_full(h, ops)


# --------------------------------------------------------------------------- stream-K walk

STREAM_K_CASES = [  # (tile_m, tile_n, max_ctas, M, N, K, lda, ldb, ldc, beta, b_col_major)
    # 256 x 256 pairs, 10 tiles on 3 pairs: TMA stores for whole tiles, per-lane for cut ones
    (256, 256, 6, 1280, 512, 1000, 1000, 512, 512, 0.0, False),
    # 256 x 320 pairs, A in row classes, beta * C on the later k-blocks
    (256, 320, 6, 1900, 300, 617, 617, 300, 300, 0.5, False),
    # 256 x 288 pairs, A in row classes (16-byte), beta * C on the later k-blocks
    (256, 288, 6, 1900, 257, 617, 617, 257, 257, 0.5, False),
    # 256 x 288 pairs, A in 64 line-aligned classes (the walk crosses classes)
    (256, 288, 20, 16384, 260, 300, 301, 260, 260, 0.5, False),
    # 256 x 288 pairs, A aligned (stages of two k-blocks, 16-column chunks):
    # whole tiles through TMA stores of 32 x 16 boxes, cut ones per lane
    (256, 288, 20, 16384, 260, 512, 512, 260, 260, 0.0, False),
    (256, 288, 12, 4096, 288, 1024, 1024, 288, 288, 0.75, False),
    # 256 x 384 pairs, beta == 1, unaligned A and C, 6 tiles on 5 pairs
    (256, 384, 10, 1300, 380, 333, 335, 380, 383, 1.0, False),
    # 256 x 384 pairs with a column-major B, 4 tiles on 2 pairs (one range = two tiles)
    (256, 384, 4, 1024, 300, 500, 500, 503, 300, -0.5, True),
    # ranges of 1.3 tiles: every pair cuts two tiles
    (256, 256, 14, 2304, 256, 1536, 1536, 256, 256, 0.25, False),
]


@pytest.mark.parametrize("tile_m,tile_n,max_ctas,M,N,K,lda,ldb,ldc,beta,b_col", STREAM_K_CASES)
def test_stream_k_walk(mp, tile_m, tile_n, max_ctas, M, N, K, lda, ldb, ldc, beta, b_col):
    # Every pair walks one contiguous range of k-blocks; a tile cut between
    # two ranges is written by the later k-blocks (with beta * C) and then
    # added to by the earlier ones. Against the oracle, element by element,
    # NaN-poisoned C when beta == 0; then on exact integers bit for bit.
    with mp.Handle() as h:
        h.set_option(mp.Option.TILE_M, tile_m)
        h.set_option(mp.Option.TILE_N, tile_n)
        h.set_option(mp.Option.MAX_CTAS, max_ctas)
        h.set_option(mp.Option.STREAM_K, 2)
        ops = workloads.make_operands(M, N, K, lda=lda, ldb=ldb, ldc=ldc, alpha=1.25, beta=beta,
                                      c_dist="normal" if beta else "zeros", seed=M + 3 * N + K,
                                      b_col_major=b_col)
        check_full(h, ops)
        ints = workloads.make_operands(M, N, K, lda=lda, ldb=ldb, ldc=ldc, beta=beta, dist="int3",
                                       dist_b="int2", c_dist="int3" if beta else "zeros",
                                       seed=M + 3 * N + K + 1, b_col_major=b_col)
        check_full(h, ints, exact=True)


def test_stream_k_plan_reaches_the_kernel(mp):
    # the planner's ranges for the cases above (the kernel reads them the same way)
    for tile_m, tile_n, max_ctas, M, N, K, lda, ldb, ldc, beta, b_col in STREAM_K_CASES:
        del tile_m, beta
        p = mp.plan(M, N, K, 1.0, 256, lda, 256, ldb, 0.0, 256, ldc, tile_m=256, tile_n=tile_n,
                    max_ctas=max_ctas, b_col_major=b_col)
        assert p["tiles"] >= max_ctas // 2


def test_stream_k_identical_bits_on_repeat_and_against_the_whole_tile_walk(mp):
    # The tall-skinny shape the planner walks in stream-K ranges by itself
    # (256 tiles of 256 x 288 on 76 pairs): identical calls give identical
    # bits, and the whole-tile walk (STREAM_K = 1) agrees within the
    # tolerance; on integers both equal the oracle.
    from parity import device_operands, reference, assert_close
    s = torch.cuda.current_stream()
    M, N, K = 65536, 257, 1021
    plan = mp.plan(M, N, K, 1.0, 256, K, 256, N, 0.5, 256, N)
    if plan["grid"] != 152:
        pytest.skip("written for 76 CTA pairs")
    assert plan["tile_n"] == 288 and plan["sk_ranges"] == 76

    def run(h, ops, n):
        outs = []
        for _ in range(n):
            d = device_operands(ops)
            h.run(ops.M, ops.N, ops.K, ops.alpha, d["a_ptr"], ops.lda, d["b_ptr"], ops.ldb, ops.beta,
                  d["c_ptr"], ops.ldc, s.cuda_stream)
            s.synchronize()
            assert h.sync_status(s.cuda_stream)[0] == mp.Status.OK
            outs.append(c_result(d, ops)[0])
        return outs

    ops = workloads.make_operands(M, N, K, alpha=0.75, beta=0.5, c_dist="normal", seed=77)
    rows = np.arange(0, M, 97)
    I, J = np.repeat(rows, N), np.tile(np.arange(N), rows.size)

    def sampled(ops):
        ref, S = reference(ops, I, J)
        return ref.reshape(rows.size, N), S.reshape(rows.size, N)

    ref, S = sampled(ops)
    with mp.Handle() as h:
        outs = run(h, ops, 3)
    assert all(np.array_equal(outs[0].view(np.uint64), o.view(np.uint64)) for o in outs[1:])
    assert_close(outs[0][rows], ref, S, "stream-K")
    with mp.Handle() as h:
        h.set_option(mp.Option.STREAM_K, 1)
        whole = run(h, ops, 1)[0]
    assert_close(whole[rows], ref, S, "whole tiles")
    ints = workloads.make_operands(M, N, K, beta=0.5, dist="int3", dist_b="int2", c_dist="int3", seed=78)
    ref, _ = sampled(ints)
    with mp.Handle() as h:
        got = run(h, ints, 2)
    for g in got:
        assert np.array_equal(g[rows], ref)
