"""Host logic of bench.py (no GPU): the FLOP and byte counters against the
numbers the pages print, the reference arm's JSON line, and the multi-rank
aggregation (max time, summed FLOPs) on two gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_worked_tile_counts(golden_facts):
    # "Day 80", Worked path: a 128x16 A tile plus a 16x128 B tile, FP16
    g = golden_facts
    m, n, k = int(g["worked_tile_m"]), int(g["worked_tile_n"]), int(g["worked_tile_k"])
    values = m * k + k * n
    assert values == int(g["worked_tile_values"])
    assert 2 * values == int(g["worked_tile_bytes"])
    assert bench.gemm_flops(m, n, k) == int(g["worked_tile_flops"])
    assert bench.gemm_flops(m, n, k) / (2 * values) == int(g["worked_flop_per_byte"])


def test_arithmetic_intensity_at_2048(golden_facts):
    # "02_mixed_precision_gemm" README, Experimental Setup: A+B = 16.8 MB,
    # C = 16 MB (MiB), intensity ~682 flop/byte. The 682 counts C at FP16
    # size (2*2048^3 / (3 * 2048^2 * 2 bytes)); this bench counts C at its
    # FP32 size, which gives 512.
    g = golden_facts
    n = 2048
    ab = bench.gemm_bytes(n, n, n, 0.0) - 4 * n * n
    assert round(ab / 1e6, 1) == float(g["ai_2048_ab_megabytes"])
    assert 4 * n * n / 2 ** 20 == float(g["ai_2048_c_megabytes"])
    pages_ai = bench.gemm_flops(n, n, n) / bench.gemm_bytes(n, n, n, 0.0, c_bytes=2)
    assert int(pages_ai) == int(g["ai_2048_flop_per_byte"])
    assert bench.gemm_flops(n, n, n) / bench.gemm_bytes(n, n, n, 0.0) == 512


def test_tflops_formula_reproduces_the_pages_rows(golden_facts):
    g = golden_facts
    n = 2048
    for ms_key, gf_key in [("t4_cublas_2048_ms", "t4_cublas_2048_gflops"),
                           ("t4_staged_2048_ms", "t4_staged_2048_gflops"),
                           ("rtx3050_cp_async_2048_ms", "rtx3050_cp_async_2048_gflops")]:
        gflops = bench.gemm_flops(n, n, n) / (float(g[ms_key]) / 1e3) / 1e9
        # the printed times are rounded to 3-4 significant digits
        assert gflops == pytest.approx(float(g[gf_key]), rel=4e-3)


def test_smem_and_peak_arithmetic(golden_facts):
    g = golden_facts
    assert 2 * (128 * 40 + 32 * 72) * 2 == int(g["cp_async_smem_bytes"])
    assert round(512 * 16 * 2 * 1.5e9 / 1e12, 1) == float(g["rtx3050_hmma_peak_tflops"])


def test_beta_doubles_c_traffic():
    assert bench.gemm_bytes(10, 20, 30, 0.0) == 10 * 30 * 2 + 30 * 20 * 2 + 10 * 20 * 4
    assert bench.gemm_bytes(10, 20, 30, 0.5) == 10 * 30 * 2 + 30 * 20 * 2 + 2 * 10 * 20 * 4


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = [0.5, 0.8][rank]
        flops = [1e12, 2e12][rank]
        t, f = bench.aggregate(seconds, flops)
        out[rank] = (t, f)
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    port = _free_port()
    mgr = tmp.Manager()
    out = mgr.dict()
    tmp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        assert out[r] == (0.8, 3e12)   # slowest rank's time, all ranks' work


def test_aggregate_single_process_is_identity():
    assert bench.aggregate(1.5, 7.0) == (1.5, 7.0)


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "0", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, env=env, timeout=300, check=True).stdout
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "ragged_tiny_200x136x617"


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--workload", "0", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, env=env, timeout=300, check=True).stdout
    assert out.strip() == ""


@pytest.mark.parametrize("index", [3, 4])
def test_traffic_records_match_the_planner(index):
    """The committed ncu traffic records (profiles/) name the tile the planner
    picks for their workload on 152 SMs, read at least the operands once, and
    bench.py reports a record only for its own tile and kernel sources."""
    import mixed_precision_dense_gb300 as mp
    import workloads
    path = bench.traffic_path(index)
    with open(path) as f:
        rec = json.load(f)
    for key in ("kernel", "workload", "tile", "dram_bytes_read_per_launch", "dram_bytes_write_per_launch",
                "dram_bytes_per_launch", "ncu_duration_ns", "source_hash", "command"):
        assert key in rec, key
    w = workloads.WORKLOADS[index]
    assert rec["workload"] == w.name
    assert "--clock-control none" in rec["command"]
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]
    # the same fake, 256-byte aligned addresses record_traffic plans with
    p = mp.plan(w.M, w.N, w.K, w.alpha, 256, w.lda, 256, w.ldb, w.beta, 256, w.ldc, num_sms=152)
    tile = f"{p['tile_m']}x{p['tile_n']}"
    assert rec["tile"] == tile
    assert f"TileConfig<{p['tile_n']}, {p['stages']}, {int(p['tile_m'] == 256)}" in rec["kernel"]
    operands_once = 2 * w.M * w.K + 2 * w.K * w.N
    assert rec["dram_bytes_read_per_launch"] >= 0.95 * operands_once
    if rec["source_hash"] == bench.source_hash():
        assert bench.stored_traffic(index, tile) == rec["dram_bytes_per_launch"]
    else:
        assert bench.stored_traffic(index, tile) is None
    assert bench.stored_traffic(index, "0x0") is None


def test_check_world_rejects_a_mismatch():
    bench.check_world(1, 1)
    bench.check_world(4, 4)
    for gpus, world in [(2, 1), (1, 2), (8, 4), (0, 1)]:
        with pytest.raises(SystemExit):
            bench.check_world(gpus, world)


def test_gpus_flag_without_ranks_exits_nonzero():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "3"],
                          capture_output=True, text=True, env=env, timeout=300)
    assert proc.returncode != 0 and "--gpus 2" in proc.stderr and proc.stdout.strip() == ""


def _world_rank_main(rank, world, port, out):
    # two gloo ranks launched for --gpus 3: every rank refuses before any GPU work
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank))
    try:
        bench.check_world(3, bench.dist_env()[0])
        out[rank] = "ran"
    except SystemExit:
        out[rank] = "refused"


def test_check_world_on_two_gloo_ranks():
    mgr = tmp.Manager()
    out = mgr.dict()
    tmp.spawn(_world_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
    assert dict(out) == {0: "refused", 1: "refused"}


PEAKS = {"tflops": 1927.1, "tflops_sustained": 1710.6, "hbm_gbs": 6775.9, "source": "measured"}


def test_roofline_picks_hbm_for_the_tall_skinny_workload():
    # 65536 x 257 x 4093 with beta != 0: 2MNK / bytes = 204.8 flop/B, below
    # the ridge 1927.1e12 / 6775.9e9 = 284 flop/B -> HBM-bound
    w = __import__("workloads").WORKLOADS[4]
    nbytes = bench.gemm_bytes(w.M, w.N, w.K, w.beta)
    assert nbytes == 2 * w.M * w.K + 2 * w.K * w.N + 2 * 4 * w.M * w.N
    main, alt = bench.roofline_pair(w.M, w.N, w.K, w.beta, 0.2, PEAKS)
    assert main["bound"] == "hbm" and alt["bound"] == "tensor"
    assert main["unit"] == "GB/s" and main["achieved"] == pytest.approx(nbytes / 0.2e-3 / 1e9, rel=1e-3)
    assert main["frac"] == pytest.approx(main["achieved"] / 6775.9, rel=1e-3)


def test_roofline_picks_tensor_for_the_square_workload():
    theory = {"tflops": 2577.6}
    main, alt = bench.roofline_pair(8192, 8192, 8192, 0.0, 0.6, PEAKS, traffic=123, theoretical=theory)
    assert main["bound"] == "tensor" and alt["bound"] == "hbm"
    assert main["achieved"] == pytest.approx(2 * 8192 ** 3 / 0.6e-3 / 1e12, rel=1e-3)
    assert main["frac_of_theoretical"] == pytest.approx(main["achieved"] / 2577.6, rel=1e-3)
    assert main["traffic"] == 123 == alt["traffic"]


def test_clock_samples_parse_and_window():
    text = ("2026/12/02 11:20:01.000, 0, 1500, 2070, 1350.5, 0x4, Not Active, Not Active, Not Active, Active\n"
            "2026/12/02 11:20:01.050, 0, 1600, 2070, 1360.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            "garbage line\n"
            "2026/12/02 11:20:02.000, 0, 2070, 2070, 200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    samples = bench.parse_clock_samples(text)
    assert len(samples) == 3 and samples[0]["reasons"] == ["sw_power_cap"]
    t0 = samples[0]["t"]
    s = bench.ClockSampler.summarize(samples, t0, t0 + 0.1)
    assert s["samples"] == 2 and s["sm_mhz"] == 1550 and s["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler.summarize(samples, t0 + 5, None)["samples"] == 0


def test_both_arms_report_the_same_config():
    w = __import__("workloads").WORKLOADS[3]
    assert bench.workload_config(w, 1) == bench.workload_config(w, 1)
    assert bench.workload_config(w, 2)["parallelism"] == "replicas x2"
