"""FP16-accumulator study variant (MPGEMM_OPT_ACCUMULATOR = 16).

"Day 72: Tensor cores with WMMA" (Exercise) rebuilds its kernel with
AccT = __half and finds that no case fails on its small-integer inputs;
"Day 80, Capstone 4: a tensor-core GEMM" ("Common failures") warns that a
4096-term sum can overflow 65,504 and that smaller sums lose low bits long
before that. The tensor cores here accumulate kind::f16 products into an
FP16 D, one rounding per K = 16 instruction. These tests pin what the pages
and FP16 arithmetic fix, independently of how the hardware orders the
additions inside one instruction:
  * the pages' integer inputs at their sizes: every partial sum is an
    integer far below 2048, so the FP16 result equals the exact sum;
  * 4096 products of 4 x 4: the sum 65,536 is past FP16's largest finite
    value, so every element overflows to +infinity (FP32: exactly 65,536);
  * sums that grow by 15 per K = 16 step past 2048 cannot all be held, so
    the result differs from the exact one, by at most half an FP16 spacing
    per step; the FP32 path stays exact.
"""
import numpy as np
import pytest
import torch

import workloads
from parity import c_result, reference, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    import mixed_precision_dense_gb300 as m
    m.build()
    m.load()
    return m


def operands_from(A, B):
    M, K = A.shape
    N = B.shape[1]
    return workloads.Operands(M, N, K, K, N, N, 1.0, 0.0, A.half().contiguous(), B.half().contiguous(),
                              torch.zeros(M, N, dtype=torch.float32))


def run(mp, ops, acc, **opts):
    with mp.Handle() as h:
        h.set_option(mp.Option.ACCUMULATOR, acc)
        for k, v in opts.items():
            h.set_option(getattr(mp.Option, k), v)
        got, _, _ = c_result(run_gpu(h, ops), ops)
    return got


@pytest.mark.parametrize("size", [256, 1024, 2048])
def test_acc16_pages_integer_sizes_exact(mp, size):
    ops = workloads.make_operands(size, size, size, dist="int3", dist_b="int2", seed=700 + size)
    ref, _ = reference(ops)
    assert np.array_equal(run(mp, ops, 16), ref)


@pytest.mark.parametrize("tile_m,tile_n", [(128, 128), (128, 256), (128, 320), (256, 256), (256, 512)])
def test_acc16_overflows_past_65504(mp, tile_m, tile_n):
    M = N = 256
    K = 4096
    ops = operands_from(torch.full((M, K), 4.0), torch.full((K, N), 4.0))
    got16 = run(mp, ops, 16, TILE_M=tile_m, TILE_N=tile_n)
    got32 = run(mp, ops, 32, TILE_M=tile_m, TILE_N=tile_n)
    assert np.all(got32 == 65536.0)
    assert np.all(np.isposinf(got16))


def test_acc16_loses_low_bits_past_2048(mp):
    M = N = 128
    steps = 512                    # K = 16 * steps
    K = 16 * steps
    A = torch.ones(M, K)
    B = torch.ones(K, N)
    B[15::16, :] = 0.0             # each K = 16 step adds exactly 15
    ops = operands_from(A, B)
    exact = 15.0 * steps
    got32 = run(mp, ops, 32)
    got16 = run(mp, ops, 16)
    assert np.all(got32 == exact)
    # past 2048 the FP16 spacing is 2 (then 4 past 4096): odd partial sums
    # cannot be held, so the result moves off the exact value, by at most
    # half a spacing (<= 2 below 8192) per step
    assert np.all(got16 != exact)
    assert np.all(np.abs(got16 - exact) <= 2.0 * steps)
    # every element saw the same sums in the same order
    assert np.all(got16 == got16[0, 0])
