"""Pins for the CPU oracle: each test ties it to something other than itself.

* its binary16 decoder, exhaustively, to numpy's float16 conversion and to the
  format facts the pages print;
* its accumulation and indexing to exact rational arithmetic (brute force),
  to exact integer matmul and to numpy's float64 matmul;
* closed forms (all-ones, identity, permutation), linearity in alpha and beta,
  and the BLAS alpha/beta reading (beta = 0 never reads C, alpha = 0 never
  reads A or B).

A wrong sign, a dropped term, a wrong or transposed index fails at least one
of these; ``test_planted_mistakes_are_caught`` proves it on mutated builds.
"""
import math
import os
import random
import shutil
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads


def _f16(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


# ---------------------------------------------------------------------------
# decoder
# ---------------------------------------------------------------------------

def test_decoder_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle.half_to_double(0x8000)) == -1.0


def test_decoder_through_gemm_table():
    # 1x1x1 products with B = 1.0 expose the decode table the GEMM uses.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(want)
    A = bits[finite]
    B = _f16([1.0])
    n = A.size
    # one GEMM of shape (n x 1 x 1): A is a column with lda = 1
    out, S = oracle.gemm(n, 1, 1, 1.0, A, 1, B, 1, 0.0)
    assert np.array_equal(out[:, 0], want[finite])
    assert np.array_equal(S[:, 0], np.abs(want[finite]))


def test_fp16_facts_from_pages(golden_facts):
    g = golden_facts
    max_bits = int(g["fp16_max_finite_bits"], 16)
    assert oracle.half_to_double(max_bits) == float(g["fp16_max_finite"])
    assert math.isinf(oracle.half_to_double(max_bits + 1))
    all_vals = np.array([oracle.half_to_double(b) for b in range(0x7C00)])  # +0 .. max finite
    ints = set(v for v in all_vals if v == int(v) and v > 0)
    top = int(g["fp16_consecutive_integers_to"])
    assert all(v in ints for v in range(1, top + 1))
    assert (top + 1) not in ints
    even_to, four_to = int(g["fp16_even_integers_to"]), int(g["fp16_multiple_of_four_to"])
    assert sorted(v for v in ints if top <= v <= even_to) == list(range(top, even_to + 1, 2))
    assert sorted(v for v in ints if even_to <= v <= four_to) == list(range(even_to, four_to + 1, 4))
    # 10 fraction bits: the spacing just above 1.0 is 2^-10
    assert oracle.half_to_double(0x3C01) - 1.0 == 2.0 ** -int(g["fp16_fraction_bits"])


# ---------------------------------------------------------------------------
# brute force against exact rational arithmetic
# ---------------------------------------------------------------------------

def _exact(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc):
    dec = lambda b: Fraction(float(np.uint16(b).view(np.float16)))
    out = np.empty((M, N), dtype=object)
    S = np.empty((M, N), dtype=object)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            sabs = Fraction(0)
            for k in range(K):
                p = dec(A[i * lda + k]) * dec(B[k * ldb + j])
                acc += p
                sabs += abs(p)
            v = Fraction(alpha) * acc
            if beta != 0:
                v += Fraction(beta) * Fraction(float(C[i * ldc + j]))
            out[i, j] = v
            S[i, j] = sabs
    return out, S


def _random_case(rng, integer=False):
    M, N, K = rng.randint(1, 7), rng.randint(1, 7), rng.randint(1, 9)
    lda, ldb, ldc = K + rng.randint(0, 3), N + rng.randint(0, 3), N + rng.randint(0, 3)
    if integer:
        A = _f16([rng.randint(-3, 3) for _ in range(M * lda)])
        B = _f16([rng.randint(-2, 2) for _ in range(K * ldb)])
        C = np.array([rng.randint(-5, 5) for _ in range(M * ldc)], dtype=np.float32)
        alpha, beta = rng.choice([1.0, 2.0, -1.0, 0.5]), rng.choice([0.0, 1.0, -2.0, 0.25])
    else:
        A = _f16([rng.uniform(-1, 1) * 2.0 ** rng.randint(-14, 4) for _ in range(M * lda)])
        B = _f16([rng.uniform(-1, 1) * 2.0 ** rng.randint(-14, 4) for _ in range(K * ldb)])
        C = np.array([rng.gauss(0, 1) for _ in range(M * ldc)], dtype=np.float32)
        alpha, beta = rng.choice([1.0, 1.5, -0.75, 3.0]), rng.choice([0.0, 1.0, 0.5, -1.25])
    return M, N, K, alpha, A, lda, B, ldb, beta, C, ldc


def _check_against_exact(case, lib=None):
    M, N, K, alpha, A, lda, B, ldb, beta, C, ldc = case
    out, S = oracle.gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, lib=lib)
    ex, exS = _exact(*case)
    for i in range(M):
        for j in range(N):
            scale = abs(alpha) * float(exS[i, j]) + abs(beta * float(C[i * ldc + j]))
            bound = 4 * (K + 2) * 2.0 ** -53 * scale
            if abs(out[i, j] - float(ex[i, j])) > bound:
                return False
            if S[i, j] != float(exS[i, j]):  # S of <= 9 exact products: exact here
                return False
    return True


def test_brute_force_exact_rational():
    rng = random.Random(12345)
    for _ in range(120):
        assert _check_against_exact(_random_case(rng))


def test_brute_force_exact_integers_bitwise():
    rng = random.Random(777)
    for _ in range(60):
        case = _random_case(rng, integer=True)
        M, N, K, alpha, A, lda, B, ldb, beta, C, ldc = case
        out, _ = oracle.gemm(*case)
        ex, _ = _exact(*case)
        assert np.array_equal(out, ex.astype(np.float64))


# ---------------------------------------------------------------------------
# exact library routines and closed forms
# ---------------------------------------------------------------------------

def test_small_integers_match_exact_int_matmul(golden_facts):
    # A in [-3, 3], B in [-2, 2] as on "Day 72", K = 2048: every partial sum is
    # an integer of magnitude <= 12,288, so the result is exact.
    g = golden_facts
    M, N, K = 48, 40, 2048
    ops = workloads.make_operands(M, N, K, dist="int3", dist_b="int2", seed=4)
    a = ops.A.to(torch.int64).numpy()
    b = ops.B.to(torch.int64).numpy()
    assert np.abs(a).max() <= int(g["int_a_max_abs"]) and np.abs(b).max() <= int(g["int_b_max_abs"])
    assert int(g["int_a_max_abs"]) * int(g["int_b_max_abs"]) == int(g["int_max_product"])
    assert int(g["int_max_product"]) * 2048 == int(g["int_max_dot_at_2048"])
    assert int(g["int_max_dot_at_2048"]) < 2 ** int(g["int_exact_float_limit_log2"])
    out, S = oracle.gemm(M, N, K, 1.0, ops.bits("A"), K, ops.bits("B"), N, 0.0)
    want = a @ b
    assert np.array_equal(out, want.astype(np.float64))
    assert np.array_equal(S, (np.abs(a) @ np.abs(b)).astype(np.float64))


@pytest.mark.parametrize("index", [0, 2])
def test_agrees_with_numpy_float64(index):
    ops = workloads.workload_operands(index)
    w = workloads.WORKLOADS[index]
    out, S = oracle.gemm(w.M, w.N, w.K, w.alpha, ops.bits("A"), w.lda, ops.bits("B"), w.ldb,
                         w.beta, ops.bits("C"), w.ldc)
    a = ops.A[:, :w.K].double().numpy()
    b = ops.B[:, :w.N].double().numpy()
    c = ops.C[:, :w.N].double().numpy()
    want = w.alpha * (a @ b) + (w.beta * c if w.beta != 0 else 0.0)
    assert np.all(np.abs(out - want) <= 1e-12 * (abs(w.alpha) * S + np.abs(w.beta * c)) + 1e-300)
    assert np.allclose(S, np.abs(a) @ np.abs(b), rtol=1e-12, atol=0)


def test_all_ones_closed_form():
    # C_ij = alpha * K + beta * C_in
    for (M, N, K) in [(5, 7, 617), (3, 2, 4093), (1, 1, 1)]:
        ops = workloads.make_operands(M, N, K, dist="ones", c_dist="normal", seed=9)
        out, _ = oracle.gemm(M, N, K, 1.0, ops.bits("A"), K, ops.bits("B"), N, 0.0)
        assert np.all(out == K)
        out, _ = oracle.gemm(M, N, K, 1.5, ops.bits("A"), K, ops.bits("B"), N, 0.5, ops.bits("C"), N)
        c = ops.C.double().numpy()
        assert np.array_equal(out, 1.5 * K + 0.5 * c)


def test_identity_and_permutation():
    K, N = 37, 53
    ops = workloads.make_operands(K, N, K, dist="uniform", seed=21)
    b = ops.B.double().numpy()
    eye = _f16(np.eye(K))
    out, _ = oracle.gemm(K, N, K, 1.0, eye, K, ops.bits("B"), N, 0.0)
    assert np.array_equal(out, b)
    perm = np.random.default_rng(5).permutation(K)
    P = np.zeros((K, K)); P[np.arange(K), perm] = 1.0
    out, _ = oracle.gemm(K, N, K, 1.0, _f16(P), K, ops.bits("B"), N, 0.0)
    assert np.array_equal(out, b[perm])
    # permutation on the right: A * P^T picks columns of A
    M = 29
    opa = workloads.make_operands(M, K, K, dist="uniform", seed=22)
    a = opa.A.double().numpy()
    out, _ = oracle.gemm(M, K, K, 1.0, opa.bits("A"), K, _f16(P.T), K, 0.0)
    assert np.array_equal(out, a[:, perm])


def test_linearity_in_alpha_and_beta():
    M, N, K = 23, 19, 131
    ops = workloads.make_operands(M, N, K, dist="int3", dist_b="int2", c_dist="int3", seed=3)
    A, B, C = ops.bits("A"), ops.bits("B"), ops.bits("C")
    ab1, _ = oracle.gemm(M, N, K, 1.0, A, K, B, N, 0.0)
    for alpha in (2.0, -3.0, 0.5):
        for beta in (1.0, -2.0, 0.25):
            out, _ = oracle.gemm(M, N, K, alpha, A, K, B, N, beta, C, N)
            cb, _ = oracle.gemm(M, N, K, 0.0, A, K, B, N, beta, C, N)
            assert np.array_equal(out, alpha * ab1 + cb)
            assert np.array_equal(cb, beta * C.reshape(M, N).astype(np.float64))
    a2, _ = oracle.gemm(M, N, K, 2.0 + 3.0, A, K, B, N, 0.0)
    a_2, _ = oracle.gemm(M, N, K, 2.0, A, K, B, N, 0.0)
    a_3, _ = oracle.gemm(M, N, K, 3.0, A, K, B, N, 0.0)
    assert np.array_equal(a2, a_2 + a_3)


def test_blas_reading_of_alpha_and_beta():
    M, N, K = 6, 5, 9
    ops = workloads.make_operands(M, N, K, lda=K + 3, ldb=N + 2, ldc=N + 1, seed=11)
    A, B = ops.bits("A"), ops.bits("B")
    nanC = np.full(M * (N + 1), np.nan, dtype=np.float32)
    out, _ = oracle.gemm(M, N, K, 1.0, A, K + 3, B, N + 2, 0.0, nanC, N + 1)
    assert np.all(np.isfinite(out))              # beta = 0: C not read
    nanA = np.full(M * (K + 3), 0x7E00, dtype=np.uint16)
    C = np.arange(M * (N + 1), dtype=np.float32)
    out, _ = oracle.gemm(M, N, K, 0.0, nanA, K + 3, nanA, N + 2, 2.0, C, N + 1)
    assert np.array_equal(out, 2.0 * C.reshape(M, N + 1)[:, :N])  # alpha = 0: A, B not read
    out, _ = oracle.gemm(M, N, 0, 1.0, None, 1, None, N, 0.5, C, N + 1)
    assert np.array_equal(out, 0.5 * C.reshape(M, N + 1)[:, :N])  # K = 0
    # padding columns hold NaN; a result free of NaN shows they were never read
    out, _ = oracle.gemm(M, N, K, 1.0, A, K + 3, B, N + 2, 0.0)
    assert np.all(np.isfinite(out))


def test_kahan_and_plain_agree():
    ops = workloads.workload_operands(0)
    w = workloads.WORKLOADS[0]
    args = (w.M, w.N, w.K, w.alpha, ops.bits("A"), w.lda, ops.bits("B"), w.ldb, w.beta)
    plain, S = oracle.gemm(*args)
    kah, _ = oracle.gemm(*args, kahan=True)
    assert np.all(np.abs(plain - kah) <= 1e-14 * S)


def test_elements_match_gemm_bitwise_and_threads_do_not_matter():
    ops = workloads.workload_operands(2)
    w = workloads.WORKLOADS[2]
    args = (w.M, w.N, w.K, w.alpha, ops.bits("A"), w.lda, ops.bits("B"), w.ldb, w.beta,
            ops.bits("C"), w.ldc)
    full, S = oracle.gemm(*args, threads=3)
    full1, _ = oracle.gemm(*args, threads=1)
    assert np.array_equal(full, full1)
    I, J = workloads.sample_indices(w.M, w.N, 500, seed=1)
    got, gS = oracle.elements(*args, I, J, threads=2)
    assert np.array_equal(got, full[I, J])
    assert np.array_equal(gS, S[I, J])


def test_rejects_bad_arguments():
    A = np.zeros(16, dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm(2, 2, 4, 1.0, A, 3, A, 2, 0.0)     # lda < K
    with pytest.raises(ValueError):
        oracle.elements(2, 2, 2, 1.0, A, 2, A, 2, 0.0, None, 2, [2], [0])  # row out of range


def test_edge_values_need_fp32_range(golden_facts):
    # "adversarial" gate case: magnitudes near the top of FP16; products exceed
    # FP16's range but the sums stay finite in FP32 (and double).
    M = N = K = 64
    ops = workloads.make_operands(M, N, K, dist="edge", seed=8)
    a = ops.A.double().numpy(); b = ops.B.double().numpy()
    assert np.abs(a).max() <= float(golden_facts["fp16_max_finite"])
    out, S = oracle.gemm(M, N, K, 1.0, ops.bits("A"), K, ops.bits("B"), N, 0.0)
    assert S.max() > 65504.0 ** 2 and S.max() < np.finfo(np.float32).max
    assert np.allclose(out, a @ b, rtol=0, atol=1e-12 * S.max())


# ---------------------------------------------------------------------------
# column-major B (the gate's layout)
# ---------------------------------------------------------------------------

def test_column_major_b_equals_row_major_of_the_transpose():
    # B stored column-major with ldb >= K; numpy builds the row-major copy
    M, N, K = 37, 29, 53
    ldb_c = K + 3
    rng = np.random.default_rng(17)
    bt = rng.uniform(-1, 1, size=(N, ldb_c)).astype(np.float16)   # row j holds column j of B
    b_rm = np.ascontiguousarray(bt[:, :K].T)                        # K x N row-major
    ops = workloads.make_operands(M, N, K, beta=0.5, c_dist="normal", seed=18)
    A, C = ops.bits("A"), ops.bits("C")
    col, Sc = oracle.gemm(M, N, K, 1.5, A, K, bt.view(np.uint16), ldb_c, 0.5, C, N, b_col_major=True)
    row, Sr = oracle.gemm(M, N, K, 1.5, A, K, b_rm.view(np.uint16), N, 0.5, C, N)
    assert np.array_equal(col, row) and np.array_equal(Sc, Sr)
    I, J = workloads.sample_indices(M, N, 200, seed=19)
    got, gS = oracle.elements(M, N, K, 1.5, A, K, bt.view(np.uint16), ldb_c, 0.5, C, N, I, J,
                              b_col_major=True)
    assert np.array_equal(got, row[I, J]) and np.array_equal(gS, Sr[I, J])


def test_column_major_b_brute_force_exact():
    rng = random.Random(99)
    for _ in range(40):
        M, N, K = rng.randint(1, 6), rng.randint(1, 6), rng.randint(1, 8)
        lda, ldb, ldc = K + rng.randint(0, 2), K + rng.randint(0, 2), N + rng.randint(0, 2)
        A = _f16([rng.randint(-3, 3) for _ in range(M * lda)])
        B = _f16([rng.randint(-2, 2) for _ in range(N * ldb)])
        out, _ = oracle.gemm(M, N, K, 1.0, A, lda, B, ldb, 0.0, b_col_major=True)
        for i in range(M):
            for j in range(N):
                want = sum(Fraction(float(np.uint16(A[i * lda + k]).view(np.float16))) *
                           Fraction(float(np.uint16(B[j * ldb + k]).view(np.float16))) for k in range(K))
                assert out[i, j] == float(want)


def test_column_major_b_checks_ldb_against_k():
    A = np.zeros(64, dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm(2, 8, 4, 1.0, A, 4, A, 3, 0.0, b_col_major=True)   # ldb < K
    oracle.gemm(2, 8, 4, 1.0, A, 4, A, 4, 0.0, b_col_major=True)       # ldb = K < N is fine


# ---------------------------------------------------------------------------
# mutation check: plausible mistakes planted in a copy of the oracle (CPU only)
# ---------------------------------------------------------------------------

MUTANTS = {
    "sign": ("sum += prod;", "sum -= prod;"),
    "dropped_beta": ("if (p->beta != 0.0) v += p->beta", "if (0) v += p->beta"),
    "transposed_b": ("b_col_major ? 1 : ldb, b_col_major ? ldb : 1",
                     "b_col_major ? ldb : 1, b_col_major ? 1 : ldb"),
    "lda_ignored": ("p->A + i * p->lda", "p->A + i * p->K"),
    "k_off_by_one": ("for (int64_t k = 0; k < p->K; ++k) {\n        const double a",
                     "for (int64_t k = 1; k < p->K; ++k) {\n        const double a"),
    "subnormal_scale": ("ldexp((double)fraction, -24)", "ldexp((double)fraction, -25)"),
    "exponent_bias": ("exponent - 25", "exponent - 24"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.bind(oracle.compile_source(str(mutated), str(tmp_path / f"lib_{name}.so")))
    rng = random.Random(12345)
    caught = False
    for _ in range(40):
        case = _random_case(rng)
        if not _check_against_exact(case, lib=lib):
            caught = True
            break
    if not caught:  # the decoder mutants must show up in the exhaustive pin
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        want = bits.view(np.float16).astype(np.float64)
        got = np.array([oracle.half_to_double(int(b), lib=lib) for b in bits])
        ok = np.isnan(want)
        caught = not np.array_equal(got[~ok], want[~ok])
    assert caught, f"planted mistake {name!r} went unnoticed"
