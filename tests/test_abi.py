"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every function include/mpgemm.h declares, and its
host planning (validation, quick returns, alignment classification, tiling)
behaves as documented."""
import ctypes
import subprocess

import pytest

import mixed_precision_dense_gb300 as mp
from mixed_precision_dense_gb300 import Status


@pytest.fixture(scope="module")
def lib():
    mp.build()
    return mp.load()


def test_exports_every_declared_function(lib):
    names = mp.header_functions()
    assert {"mpgemm_create", "mpgemm_run", "mpgemm_destroy", "mpgemm_status_string",
            "mpgemm_plan", "mpgemm_run_host", "mpgemm_sync_status", "mpgemm_set_option"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", mp.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, f"{n} declared but not exported"
        assert hasattr(lib, n)


def test_built_for_sm103a_only():
    text = open(mp.LIB_PATH.replace("libmpgemm.so", "ptxas.txt")).read()
    assert "arch=compute_103a,code=sm_103a" in text
    assert "spill stores" in text and " 0 bytes spill stores" in text


def test_status_strings(lib):
    for s in Status:
        assert mp.status_string(s)
    assert mp.status_string(99) == "unknown status"


def test_null_handle_is_rejected(lib):
    assert lib.mpgemm_run(None, 1, 1, 1, 1.0, 16, 1, 16, 1, 0.0, 16, 1, None) == Status.ERR_INVALID_VALUE
    assert lib.mpgemm_destroy(None) == Status.OK
    assert lib.mpgemm_set_option(None, 1, 0) == Status.ERR_INVALID_VALUE
    assert lib.mpgemm_create(None) == Status.ERR_INVALID_VALUE


@pytest.mark.parametrize("ctas,mmas,out", [(0, 64, 256), (65536, 64, 256), (1, 3, 256), (1, 1 << 23, 256),
                                           (1, 64, 0), (1, 64, 260)])
def test_probe_rejects_bad_arguments(lib, ctas, mmas, out):
    # checked before any CUDA call, so this runs without a GPU
    assert lib.mpgemm_probe_mma_rate(ctas, mmas, out or None, None) == Status.ERR_INVALID_VALUE


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(1)
    st = lib.mpgemm_create(ctypes.byref(h))
    assert st in (Status.ERR_UNSUPPORTED_DEVICE, Status.ERR_CUDA)
    assert not h.value


def _plan(**kw):
    base = dict(M=200, N=136, K=617, alpha=1.0, A=256, lda=617, B=256, ldb=136, beta=0.0,
                C=256, ldc=136)
    base.update(kw)
    return mp.plan(**base)


@pytest.mark.parametrize("kw", [dict(M=-1), dict(N=-1), dict(K=-1), dict(lda=616), dict(ldb=135),
                                dict(ldc=135), dict(A=0), dict(B=0), dict(C=0), dict(C=258),
                                dict(A=257), dict(B=255), dict(M=2 ** 31), dict(lda=2 ** 31)])
def test_invalid_arguments(kw):
    with pytest.raises(mp.MpgemmError) as e:
        _plan(**kw)
    assert e.value.status == Status.ERR_INVALID_VALUE


def test_column_major_b_validation():
    # column-major B: ldb counts K (rows of B are columns of the product)
    p = _plan(M=64, N=300, K=40, lda=40, ldb=40, ldc=300, b_col_major=True)
    assert p["quick"] == 0 and p["stage_b"] == 0
    with pytest.raises(mp.MpgemmError):
        _plan(M=64, N=300, K=40, lda=40, ldb=39, ldc=300, b_col_major=True)
    with pytest.raises(mp.MpgemmError):          # the same ldb is too small for row-major B
        _plan(M=64, N=300, K=40, lda=40, ldb=40, ldc=300)
    p = _plan(M=64, N=300, K=617, lda=617, ldb=617, ldc=300, b_col_major=True)
    r256 = lambda x: (x + 255) // 256 * 256
    assert p["stage_b"] == 1 and p["workspace_bytes"] == r256(64 * 624 * 2) + r256(300 * 624 * 2)


def test_quick_returns():
    assert _plan(M=0, A=0, B=0, C=0)["quick"] == 1
    assert _plan(N=0, ldb=1, ldc=1, A=0, B=0, C=0)["quick"] == 1
    assert _plan(K=0, lda=1, A=0, B=0)["quick"] == 2     # C = beta*C, A and B never read
    assert _plan(alpha=0.0, A=0, B=0)["quick"] == 2
    assert _plan()["quick"] == 0


def test_alignment_classification():
    # lda = 617 halves = 1234 bytes: rows start at 8 different offsets modulo
    # 16, so A is read directly in 8 row classes (one-CTA tiles, row-major B)
    p = _plan()
    assert (p["stage_a"], p["stage_b"], p["a_classes"]) == (0, 0, 8)
    assert p["workspace_bytes"] == 0
    # the same A staged when asked, or under a column-major B
    p = _plan(force_staging=True)
    assert p["stage_a"] == 1 and p["a_classes"] == 0
    p = _plan(ldb=617, b_col_major=True)
    assert p["stage_a"] == 1 and p["a_classes"] == 0
    assert p["workspace_bytes"] == 200 * 624 * 2 + 136 * 624 * 2
    p = _plan(M=2048, N=2048, K=2048, lda=2048, ldb=2048, ldc=2048)
    assert (p["stage_a"], p["stage_b"]) == (0, 0) and p["workspace_bytes"] == 0
    # the tall-skinny pairs take classes of rows that start at the same offset
    # in a 128-byte line: 8186-byte rows start at 64 offsets
    p = _plan(M=65536, N=257, K=4093, lda=4093, ldb=257, ldc=257, beta=0.5)
    assert (p["stage_a"], p["stage_b"], p["a_classes"]) == (0, 1, 64)
    # lda = 4094: rows start at four offsets; lda = 4100: two
    assert _plan(M=4096, N=257, K=4093, lda=4094, ldb=257, ldc=257)["a_classes"] == 4
    assert _plan(M=4096, N=257, K=4093, lda=4100, ldb=257, ldc=257)["a_classes"] == 2
    # a base address 2 bytes past a 16-byte boundary with an aligned pitch: one
    # class, read with a shift of one element
    p = _plan(M=128, N=128, K=128, lda=128, ldb=128, ldc=128, A=256 + 2)
    assert (p["stage_a"], p["stage_b"], p["a_classes"]) == (0, 0, 1)
    assert p["k_blocks"] == 3                      # K + 1 view columns
    # CTA pairs read an unaligned A in row classes too, with 256-row class
    # tiles: ceil(1024 / 256) tiles in each of the 8 classes
    p = _plan(M=8192, N=8192, K=8192, lda=8193, ldb=8192, ldc=8192)
    assert p["tile_m"] == 256 and p["stage_a"] == 0 and p["a_classes"] == 8
    assert p["m_tiles"] == 8 * 4
    # 256 x 384 pair tiles (room for 8 row classes): pairs only, never split
    # into half-width items
    p = _plan(M=65536, N=257, K=4093, lda=4093, ldb=257, ldc=257, tile_n=384)
    assert (p["tile_m"], p["tile_n"], p["a_classes"], p["split_tiles"]) == (256, 384, 8, 0)
    with pytest.raises(mp.MpgemmError):
        _plan(M=65536, N=257, K=4093, lda=4093, ldb=257, ldc=257, tile_m=128, tile_n=384)
    p = _plan(M=128, N=128, K=128, lda=128, ldb=128, ldc=128, force_staging=True)
    assert (p["stage_a"], p["stage_b"]) == (1, 1)


def test_tiling_of_the_ragged_k_tail(golden_facts):
    # The page's K loop steps by 16 and its last step starts at 608 with 9 valid
    # values; this library steps by 64, and the same K = 617 ends with 41 valid.
    g = golden_facts
    K, step = int(g["tail_k"]), int(g["tail_step"])
    assert (K // step) * step == int(g["tail_last_start"])
    assert K - int(g["tail_last_start"]) == int(g["tail_valid"])
    assert step - int(g["tail_valid"]) == int(g["tail_invalid"])
    p = _plan()
    assert p["tile_k"] == 64 and p["k_blocks"] == 10 and p["last_k_valid"] == 41
    assert (p["k_blocks"] - 1) * p["tile_k"] + p["last_k_valid"] == K


def test_tile_selection_and_grid():
    # large square, long K: CTA pairs on 256 x 512 tiles, one pair per two SMs
    p = _plan(M=8192, N=8192, K=8192, lda=8192, ldb=8192, ldc=8192)
    assert (p["tile_m"], p["tile_n"]) == (256, 512) and p["tiles"] == 32 * 16 and p["grid"] == 152
    assert p["smem_bytes"] <= 232448 and p["stages"] == 4
    # (512 tiles on 76 pairs: a last wave of 56 tiles, more than half full, not split)
    assert p["split_tiles"] == 0 and p["items"] == 512
    # the same square with a short K keeps 256 x 256 pair tiles
    p = _plan(M=8192, N=8192, K=1024, lda=1024, ldb=8192, ldc=8192)
    assert (p["tile_m"], p["tile_n"]) == (256, 256) and p["stages"] == 3 and p["tile_k"] == 128   # two 64-wide k-blocks per stage
    # 512-wide tiles on request, also for small or ragged shapes; never with one CTA per tile
    p = _plan(M=300, N=700, K=200, lda=200, ldb=700, ldc=700, tile_n=512)
    assert (p["tile_m"], p["tile_n"]) == (256, 512) and p["tiles"] == 2 * 2 and p["grid"] == 8
    p = _plan(M=300, N=700, K=200, lda=200, ldb=700, ldc=700, tile_m=256, tile_n=512)
    assert (p["tile_m"], p["tile_n"]) == (256, 512)
    with pytest.raises(mp.MpgemmError):
        _plan(tile_m=128, tile_n=512)
    # N = 257 would waste half of the last column band: one tile column of
    # 256 x 288 CTA pairs (A read once per row block; A in 64 row classes of
    # 4 pair tiles each, five 34 KB stages)
    p = _plan(M=65536, N=257, K=4093, lda=4093, ldb=257, ldc=257, beta=0.5)
    assert (p["tile_m"], p["tile_n"]) == (256, 288) and p["tiles"] == 256 and p["stages"] == 5
    assert p["tile_k"] == 64 and p["a_classes"] == 64 and p["split_tiles"] == 0
    assert 200 * 1024 < p["smem_bytes"] <= 232448
    # A aligned: three 68 KB stages of two k-blocks
    p = _plan(M=58368, N=257, K=4096, lda=4096, ldb=264, ldc=257, beta=0.5)
    assert (p["tile_m"], p["tile_n"]) == (256, 288) and p["tiles"] == 228
    assert (p["stages"], p["tile_k"], p["a_classes"]) == (3, 128, 0) and p["smem_bytes"] <= 232448
    # N from 289 to 320: 256 x 320 pairs (five 36 KB stages)
    p = _plan(M=58368, N=300, K=4096, lda=4096, ldb=304, ldc=300, beta=0.5)
    assert (p["tile_m"], p["tile_n"], p["stages"], p["tile_k"]) == (256, 320, 5, 64) and p["tiles"] == 228
    # fewer rows than one full wave of pair tiles: one-CTA tiles; with A
    # aligned, a wave of 320-wide tiles (1.9 waves of 256-wide ones) costs
    # more than one wave of 256-wide tiles, and less than two
    p = _plan(M=9600, N=257, K=4096, lda=4096, ldb=264, ldc=257, beta=0.5)
    assert (p["tile_m"], p["tile_n"]) == (128, 256) and p["a_classes"] == 0
    p = _plan(M=19200, N=257, K=4096, lda=4096, ldb=264, ldc=257, beta=0.5)
    assert (p["tile_m"], p["tile_n"], p["stages"]) == (128, 320, 3) and p["tiles"] == 150
    # N = 321: one tile column of 256 x 384 pairs; too few row blocks: not 320
    p = _plan(M=65536, N=321, K=4093, lda=4093, ldb=321, ldc=321)
    assert (p["tile_m"], p["tile_n"]) == (256, 384)
    p = _plan(M=1000, N=300, K=1000, lda=1000, ldb=300, ldc=300)
    assert p["tile_n"] == 128
    # 320 wide on request (one CTA per tile, or a pair with tile_m 256), never
    # split in half-width items
    p = _plan(M=5000, N=1000, K=700, lda=700, ldb=1000, ldc=1000, tile_n=320)
    assert (p["tile_m"], p["tile_n"]) == (128, 320) and p["tiles"] == 40 * 4 and p["split_tiles"] == 0
    p = _plan(M=5000, N=1000, K=700, lda=700, ldb=1000, ldc=1000, tile_m=256, tile_n=320)
    assert (p["tile_m"], p["tile_n"], p["stages"]) == (256, 320, 5) and p["tiles"] == 20 * 4
    assert p["split_tiles"] == 0
    # the 256 x 320 and 256 x 288 pairs read B in narrow row-major boxes: not
    # for a column-major B; 288 wide: pairs only
    with pytest.raises(mp.MpgemmError):
        _plan(tile_m=256, tile_n=320, ldb=617, b_col_major=True)
    with pytest.raises(mp.MpgemmError):
        _plan(tile_n=288, ldb=617, b_col_major=True)
    with pytest.raises(mp.MpgemmError):
        _plan(tile_m=128, tile_n=288)
    p = _plan(M=5000, N=1000, K=700, lda=700, ldb=1000, ldc=1000, tile_n=288)
    # (lda 700: 1400-byte rows, read in row classes: five stages of one k-block)
    assert (p["tile_m"], p["tile_n"], p["stages"], p["tile_k"]) == (256, 288, 5, 64) and p["tiles"] == 20 * 4
    assert p["split_tiles"] == 0
    # forced pairs with a CTA cap: the grid stays even
    p = _plan(M=1000, N=800, K=64, lda=64, ldb=800, ldc=800, tile_m=256, max_ctas=5)
    assert p["tile_m"] == 256 and p["grid"] == 4 and p["tiles"] == 4 * 4
    p = _plan(M=300, N=300, K=64, lda=64, ldb=300, ldc=300, tile_m=256, max_ctas=1)
    assert p["grid"] == 2
    p = _plan(M=8192, N=8192, K=8192, lda=8192, ldb=8192, ldc=8192, tile_m=128)
    assert (p["tile_m"], p["tile_n"]) == (128, 256) and p["tiles"] == 64 * 32
    # 2048^3: 128 tiles of 128 x 256 keep 84 % of the SMs busy: wide tiles
    p = _plan(M=2048, N=2048, K=2048, lda=2048, ldb=2048, ldc=2048)
    assert p["tile_m"] == 128 and p["tile_n"] == 256 and p["tiles"] == 16 * 8 and p["grid"] == 128
    # with K = 4096 the same square takes 64 CTA-pair tiles (84 % of the pairs)
    p = _plan(M=2048, N=2048, K=4096, lda=4096, ldb=2048, ldc=2048)
    assert (p["tile_m"], p["tile_n"]) == (256, 256) and p["tiles"] == 64 and p["grid"] == 128
    # 1000 x 800: 32 wide tiles would leave most SMs idle: 128 x 128
    p = _plan(M=1000, N=800, K=1200, lda=1200, ldb=800, ldc=800)
    assert p["tile_n"] == 128 and p["tiles"] == 8 * 7
    # 8192^3 in 256 x 256 pair tiles: 1024 tiles on 76 pairs leave a last wave
    # of 36 tiles, split in halves
    p = _plan(M=8192, N=8192, K=8192, lda=8192, ldb=8192, ldc=8192, tile_m=256)
    assert p["tile_n"] == 256 and p["split_tiles"] == 1024 % 76 and p["items"] == 1024 + 36
    # too few tiles to occupy the GPU: K is cut into slices (no empty slice)
    p = _plan(M=4096, N=16, K=4096, lda=4096, ldb=16, ldc=16)
    assert p["k_splits"] == 4 and p["items"] == 32 * 4 and p["split_tiles"] == 0
    p = _plan(M=4096, N=16, K=4096, lda=4096, ldb=16, ldc=16, tile_m=256)
    assert p["k_splits"] == 1                       # pairs never split K
    for K in (520, 576, 9 * 64):
        p = _plan(M=256, N=128, K=K, lda=K, ldb=128, ldc=128)
        per = -(-p["k_blocks"] // p["k_splits"])
        assert (p["k_splits"] - 1) * per < p["k_blocks"]
    # a last wave more than half full is not split in halves; the 288-wide
    # pairs of this tall-skinny problem walk stream-K ranges instead
    p = _plan(M=65536, N=257, K=4093, lda=4093, ldb=257, ldc=257)
    assert p["split_tiles"] == 0 and p["sk_ranges"] == 76
    p = _plan()
    assert p["a_classes"] == 8 and p["tiles"] == 8 * 2                      # 8 classes of 25 rows
    # 16 tiles of 10 k-blocks (at most an eighth of the SMs): five K slices,
    # added into C (clusters only on request or for reproducible calls)
    assert p["k_splits"] == 5 and p["items"] == 16 * 5 and p["grid"] == 80 and p["split_reduce"] == 0
    p = _plan(M=128, N=128, K=8192, lda=8192, ldb=128, ldc=128)   # one tile of 128 k-blocks
    assert p["k_splits"] == 16 and p["split_reduce"] == 0
    p = _plan(M=611, N=613, K=617, lda=617, ldb=613, ldc=613)
    assert p["tiles"] == 40 and p["k_splits"] == 1
    p = _plan(M=8192, N=8192, K=8192, lda=8192, ldb=8192, ldc=8192, tile_n=128, max_ctas=10)
    assert p["tile_n"] == 128 and p["grid"] == 10
    with pytest.raises(mp.MpgemmError):
        _plan(tile_n=192)
    with pytest.raises(mp.MpgemmError):
        _plan(tile_m=64)


def _row_classes(lda, M, tile_m, room):
    """The planner's row classes of an A whose rows are not 16-byte aligned,
    restated: P16 = 16 / gcd(2 lda, 16) classes (rows at the same offset
    modulo 16), or P128 = 128 / gcd(2 lda, 128) (the same offset in a 128-byte
    line) when the kernel has room for them and they cost at most 1/32 more
    M-tiles."""
    from math import gcd
    p16, p128 = 16 // gcd(2 * lda, 16), 128 // gcd(2 * lda, 128)
    tiles = lambda P: sum(-(-((M - r + P - 1) // P) // tile_m) for r in range(min(P, M)))
    return p128 if p128 > p16 and p128 <= room and tiles(p128) * 32 <= tiles(p16) * 33 else p16


@pytest.mark.parametrize("M,N,K,lda,A,expect", [
    (65536, 257, 4093, 4093, 256, 64),    # 8186-byte rows: 64 line offsets, 4 pair tiles per class
    (65536, 257, 4093, 4094, 256, 32),
    (65536, 257, 4092, 4092, 256, 16),
    (65536, 300, 4093, 4093, 256, 64),    # the 320-wide pairs too
    (65536, 384, 4093, 4093, 256, 8),     # the 384-wide ones have room for 8
    (19456, 257, 4093, 4093, 256, 8),     # 64 classes of 304 rows: 128 pair tiles against 80
    (19200, 257, 4093, 4093, 256, 8),     # one-CTA tiles: room for 8 classes
    (8192, 8192, 8192, 8193, 256, 8),     # 256 x 256 pairs: room for 8
    (4096, 4096, 4096, 4096, 258, 1),     # one class (aligned pitch), shifted by (A mod 128) / 2
])
def test_line_aligned_row_classes(M, N, K, lda, A, expect):
    p = _plan(M=M, N=N, K=K, lda=lda, ldb=N, ldc=N, A=A)
    assert p["stage_a"] == 0 and p["a_classes"] == expect
    room = 64 if (p["tile_m"], p["tile_n"]) in ((256, 288), (256, 320)) else 8
    if lda * 2 % 16:
        assert expect == _row_classes(lda, M, p["tile_m"], room)
    P = expect
    unit = 128 if P * 2 * lda % 128 == 0 else 16
    shifts = [((A + r * 2 * lda) % unit) // 2 for r in range(P)]
    rows = [(M - r + P - 1) // P for r in range(P)]
    assert p["m_tiles"] == sum(-(-n // p["tile_m"]) for n in rows)
    assert p["k_blocks"] == -(-(K + max(shifts)) // p["tile_k"])


@pytest.mark.parametrize("M,N,lda,b_col,expect", [
    (65536, 256, 4093, False, (128, 256)),   # one 256-wide column covers N: one-CTA tiles
    (65536, 257, 4093, False, (256, 288)),   # the tall-skinny workload: 256 x 288 pairs
    (58368, 288, 4096, False, (256, 288)),
    (58368, 289, 4096, False, (256, 320)),   # past 288: 256 x 320 pairs
    (58368, 320, 4096, False, (256, 320)),
    (65536, 321, 4096, False, (256, 384)),   # past 320: 256 x 384 pairs
    (65536, 384, 4096, False, (256, 384)),
    (65536, 300, 4096, True, (256, 384)),    # column-major B: the 384-wide pair
    (65536, 385, 4093, False, (128, 256)),   # past 384: two 256-wide columns of one-CTA tiles
    (19456, 257, 4093, False, (256, 288)),   # 76 pair tiles: every pair busy
    (19200, 257, 4093, False, (128, 320)),   # 75: the one-CTA rule (row classes: 1.6 waves of 320 < 2)
    (9600, 257, 4096, False, (128, 256)),    # aligned A: 1.9 waves of 320 against one wave of 256
])
def test_narrow_tile_column_rules(M, N, lda, b_col, expect):
    p = _plan(M=M, N=N, K=4093, lda=lda, ldb=4093 if b_col else N + 8, ldc=N, beta=0.5, b_col_major=b_col)
    assert (p["tile_m"], p["tile_n"]) == expect, (M, N, lda)
    if expect[1] in (288, 320, 384):
        assert p["split_tiles"] == 0 and p["n_tiles"] == 1


@pytest.mark.parametrize("M,K,beta,splits", [
    (19 * 128, 640, 0.0, 5),   # 19 tiles: an eighth of 152 SMs, 10 k-blocks: five slices
    (20 * 128, 640, 0.0, 1),   # 20 tiles: past an eighth
    (128, 7 * 64, 0.0, 1),     # 7 k-blocks: too short
    (128, 8 * 64, 0.0, 4),     # 8 k-blocks: four slices of two
    (19 * 128, 640, 1.0, 5),   # beta == 1: no pass over C first, the same short-K rule
    (19 * 128, 640, 0.5, 5),   # any other beta: C = beta * C first, then the slices
])
def test_short_k_split_rule(M, K, beta, splits):
    p = _plan(M=M, N=128, K=K, lda=K, ldb=128, ldc=128, beta=beta)
    assert p["tile_n"] == 128 and p["k_splits"] == splits
    per = -(-p["k_blocks"] // p["k_splits"])
    assert (p["k_splits"] - 1) * per < p["k_blocks"] and p["items"] == p["tiles"] * p["k_splits"]


def _sk_starts(units, kb, R):
    """The planner's stream-K boundaries, restated: equal ranges, then each
    inner boundary within an eighth of a tile's k-blocks of a tile edge moved
    onto that edge, unless a range would become shorter than one tile."""
    length, rem, snap = units // R, units % R, max(1, kb // 8)
    start = [r * length + min(r, rem) for r in range(R + 1)]
    moved = list(start)
    for r in range(1, R):
        off = moved[r] % kb
        if off and off <= snap:
            moved[r] -= off
        elif off and kb - off <= snap:
            moved[r] += kb - off
    return moved if all(moved[r + 1] - moved[r] >= kb for r in range(R)) else start


def test_stream_k_planning():
    """The stream-K walk: automatic for 288-, 320- and 384-wide CTA-pair tiles
    whose last wave leaves pairs idle; one range of about equal length per
    pair; the items cover the tiles every range touches."""
    p = _plan(M=65536, N=257, K=4093, lda=4093, ldb=257, ldc=257)
    # k-blocks over K plus the largest row-class shift (63)
    assert (p["tile_m"], p["tile_n"], p["tiles"], p["k_blocks"]) == (256, 288, 256, 65)
    ranges, kb = p["sk_ranges"], p["k_blocks"]
    assert ranges == 76 and p["grid"] == 2 * ranges
    units = p["tiles"] * kb
    start = _sk_starts(units, kb, ranges)
    assert start[0] == 0 and start[-1] == units
    lengths = [start[r + 1] - start[r] for r in range(ranges)]
    assert min(lengths) >= kb and sum(lengths) == units
    # no piece of a tile shorter than an eighth of its k-blocks at any boundary
    assert all(s_ % kb == 0 or kb // 8 < s_ % kb < kb - kb // 8 for s_ in start)
    # lengths within two eighths of a tile of each other
    assert max(lengths) - min(lengths) <= 2 * (kb // 8) + 1
    touched = max((start[r + 1] - 1) // kb - start[r] // kb + 1 for r in range(ranges))
    assert p["items"] == ranges * touched
    # 320- and 384-wide pairs (N from 289 and 321 on), and the K-major B variant
    p = _plan(M=65536, N=300, K=4096, lda=4096, ldb=304, ldc=300)
    assert p["tile_n"] == 320 and p["sk_ranges"] == 76
    p = _plan(M=65536, N=384, K=4096, lda=4096, ldb=384, ldc=384)
    assert p["tile_n"] == 384 and p["sk_ranges"] == 76
    p = _plan(M=65536, N=300, K=4096, lda=4096, ldb=4096, ldc=300, b_col_major=True)
    assert p["tile_n"] == 384 and p["sk_ranges"] == 76
    # exactly three waves of tiles: nothing to balance
    p = _plan(M=58368, N=257, K=4096, lda=4096, ldb=257, ldc=257)
    assert p["tiles"] == 3 * 76 and p["sk_ranges"] == 0 and p["items"] == p["tiles"]
    # one column of 256-wide pair tiles (3.37 waves); more columns, single
    # CTAs and fewer tiles than pairs: never automatic
    p = _plan(M=65536, N=256, K=4096, lda=4096, ldb=256, ldc=256, tile_m=256)
    assert (p["tile_n"], p["n_tiles"], p["sk_ranges"], p["split_tiles"]) == (256, 1, 76, 0)
    assert _plan(M=20480, N=1024, K=4096, lda=4096, ldb=1024, ldc=1024, tile_m=256)["sk_ranges"] == 0
    assert _plan(M=8192, N=300, K=4096, lda=4096, ldb=300, ldc=300)["sk_ranges"] == 0
    assert _plan(M=8192, N=8192, K=8192, lda=8192, ldb=8192, ldc=8192)["sk_ranges"] == 0
    # a smaller grid: ranges follow the pairs launched
    p = _plan(M=65536, N=257, K=4093, lda=4093, ldb=257, ldc=257, max_ctas=100)
    assert p["sk_ranges"] == 50 and p["grid"] == 100
