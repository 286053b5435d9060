"""Edge values through every tile shape: FP16 subnormal operands, and
infinities and NaN in A and B ("Day 80, Capstone 4: a tensor-core GEMM",
"Common failures": edge values and overflow).

Subnormal A (integers up to 1023 times 2^-24) against B of small integers
times 2^13 gives products that are exact multiples of 2^-11, so every sum
is exact in FP32: C must equal the oracle bit for bit, which pins the
tensor cores' reading of subnormal FP16 to the oracle's decoder. With Inf
and NaN placed in A and B, the oracle's double arithmetic fixes which
elements are NaN, which are +-Inf and which are finite: the GPU result must
agree on every element's class, equal the infinities, and be within the
tolerance elsewhere.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import c_result, check_guards, reference, run_gpu

pytestmark = pytest.mark.gpu

# the tile shapes of the library, forced through the handle's options
SHAPES = {
    "128x128": {"TILE_M": 128, "TILE_N": 128, "SPLIT_K": 1},
    "128x256": {"TILE_M": 128, "TILE_N": 256, "SPLIT_K": 1},
    "128x320": {"TILE_M": 128, "TILE_N": 320, "SPLIT_K": 1},
    "128x128_split3": {"TILE_M": 128, "TILE_N": 128, "SPLIT_K": 3},
    "pair256x256": {"TILE_M": 256, "TILE_N": 0},
    "pair256x320": {"TILE_M": 256, "TILE_N": 320},
    "pair256x384": {"TILE_M": 256, "TILE_N": 384},
    "pair256x512": {"TILE_M": 256, "TILE_N": 512},
}


@pytest.fixture(scope="module")
def mp():
    import mixed_precision_dense_gb300 as m
    m.build()
    m.load()
    return m


def _handle(mp, opts):
    h = mp.Handle()
    for k, v in opts.items():
        h.set_option(getattr(mp.Option, k), v)
    return h


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("subnormal_side", ["A", "B"])
def test_subnormal_operands_bitwise(mp, shape, subnormal_side):
    da, db = ("subnormal", "int3_x8192") if subnormal_side == "A" else ("int3_x8192", "subnormal")
    ops = workloads.make_operands(520, 600, 1000, lda=1003, dist=da, dist_b=db, seed=300 + len(shape))
    a = ops.A[:, :ops.K].float()
    assert (a[(a != 0)].abs() < 2.0 ** -14).all() if subnormal_side == "A" else True
    with _handle(mp, SHAPES[shape]) as h:
        d = run_gpu(h, ops)
    got, buf, full = c_result(d, ops)
    check_guards(d, ops, buf, full)
    ref, _ = reference(ops)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_inf_and_nan_propagate_as_in_the_oracle(mp, shape):
    M, N, K = 520, 600, 1000
    ops = workloads.make_operands(M, N, K, lda=1003, seed=400 + len(shape))
    inf, nan = float("inf"), float("nan")
    # +Inf in A (row 3, k = 17), NaN in A (row 300, k = 500), -Inf in B (k = 900,
    # column 555), +Inf in B (k = 10, column 7): whole rows and columns become
    # infinite, NaN where infinities of both signs meet and in row 300
    ops.A[3, 17] = inf
    ops.A[300, 500] = nan
    ops.B[900, 555] = -inf
    ops.B[10, 7] = inf
    # no exact zeros next to the infinities (Inf * 0 would be NaN)
    for t, idx in ((ops.A, (slice(None), 900)), (ops.A, (slice(None), 10)), (ops.B, (17, slice(None)))):
        v = t[idx]
        v[v == 0] = 0.5
    with _handle(mp, SHAPES[shape]) as h:
        d = run_gpu(h, ops)
    got, buf, full = c_result(d, ops)
    check_guards(d, ops, buf, full)
    ref, S = reference(ops)
    nan_ref, inf_ref = np.isnan(ref), np.isinf(ref)
    assert nan_ref[300].all() and inf_ref[:, 555].sum() > M // 2 and inf_ref[3].sum() > N // 2
    assert np.array_equal(np.isnan(got), nan_ref)
    assert np.array_equal(got[inf_ref], ref[inf_ref])
    fin = ~(nan_ref | inf_ref)
    assert np.all(np.abs(got[fin] - ref[fin]) <= oracle.tolerance(S[fin]))
