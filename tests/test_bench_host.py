"""Host-side logic of bench.py: whole-job aggregation over ranks (world size
2, gloo, CPU), clock-sample parsing and the roofline arithmetic."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from cross_model_kv_transfer_gb300.workloads import WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist("gloo")
    ms_local = [4.0, 5.0][rank]
    value, ms = bench.aggregate(1000, ms_local)
    bench.barrier()
    out[rank] = (value, ms)
    dist.destroy_process_group()


def test_aggregate_takes_slowest_rank_and_all_tokens():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    for r in range(2):
        value, ms = out[r]
        assert ms == 5.0
        assert value == pytest.approx(2 * 1000 / 5e-3)


def test_single_process_aggregate_is_local():
    value, ms = bench.aggregate(32768, 8.0)
    assert ms == 8.0 and value == pytest.approx(32768 / 8e-3)


def test_clock_summary_flags_throttle_reasons():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.lines = ["1900, 2070, 900.0, Not Active, Not Active, Not Active, Active",
               "2070, 2070, 1000.0, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s["sm_mhz"] == pytest.approx(1985.0) and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def test_roofline_picks_the_tighter_bound():
    wl = WORKLOADS["qwen3_14b_32b"]
    idx = torch.stack([torch.arange(4) + i % 36 for i in range(64)]).to(torch.int32)
    peaks = {"hbm_gbs": 6766.7, "bf16_tflops": 1908.0, "bf16_tflops_sustained": 1679.6}
    r = bench.roofline(wl, idx, 4.398046511104, "tcgen05", peaks, "measured")
    # 4.398 TFLOP in 4.398 ms = 1000 TFLOP/s; tensor time 2.31 ms > HBM time
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1000.0, rel=1e-6)
    assert r["frac"] == pytest.approx(1000.0 / 1908.0, rel=1e-6)
    assert r["algorithmic_flops"] == 2 * 32768 * 512 * 128 * 64 * 8 * 2
    small = wl.with_tokens([512], [0])
    r = bench.roofline(small, idx, 1.0, "tcgen05", peaks, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"


def test_roofline_compares_a_power_capped_run_with_the_sustained_peak():
    # the timed region ran under the power cap: the sustained cuBLAS figure
    # (measured in the same regime) is the denominator; both fractions and
    # the nominal one (SMs x 8192 flops/clk x sampled clock) are reported
    wl = WORKLOADS["qwen3_14b_32b"]
    idx = torch.stack([torch.arange(4) + i % 36 for i in range(64)]).to(torch.int32)
    peaks = {"hbm_gbs": 6766.7, "bf16_tflops": 1908.0, "bf16_tflops_sustained": 1679.6}
    capped = {"sm_mhz": 1740.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    r = bench.roofline(wl, idx, 4.398046511104, "tcgen05", peaks, "measured", clocks=capped)
    assert r["peak"] == 1679.6 and r["frac"] == pytest.approx(1000.0 / 1679.6, rel=1e-6)
    assert "sustained" in r["peak_source"]
    assert r["frac_of_burst"] == pytest.approx(1000.0 / 1908.0, rel=1e-6)
    assert r["nominal_peak"] == pytest.approx(152 * 8192 * 1740e6 / 1e12)
    free = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    r = bench.roofline(wl, idx, 4.398046511104, "tcgen05", peaks, "measured", clocks=free)
    assert r["peak"] == 1908.0 and "burst" in r["peak_source"]


def test_published_context_number_is_the_32k_mapper_latency():
    # the Qwen3 article's 14B -> 32B mapper: 277.6 ms at 32,768 tokens
    assert bench.PUBLISHED_MS["qwen3_14b_32b"] == 277.6
    assert json.dumps(bench.METRIC)


def test_wide_roofline_uses_the_wide_map_accounting():
    # one [8192 x 2048] map per target layer: 70.37 TFLOP per 32K transfer,
    # W counted as stored (fp32, 4.3 GB)
    wl = WORKLOADS["qwen3_14b_32b"]
    idx = torch.stack([torch.arange(4) + i % 36 for i in range(64)]).to(torch.int32)
    assert wl.wide_algorithmic_flops() == 2 * 32768 * 8192 * 2048 * 64
    peaks = {"hbm_gbs": 6766.7, "bf16_tflops": 1908.0, "bf16_tflops_sustained": 1679.6}
    r = bench.roofline(wl, idx, 46.0, "wide", peaks, "measured", wide=True)
    assert r["bound"] == "tensor"
    assert r["frac_of_sustained"] == pytest.approx(r["achieved"] / 1679.6)
    w_bytes = 64 * 8192 * 2048 * 4
    assert r["algorithmic_bytes"] - wl.algorithmic_bytes(idx) == pytest.approx(
        w_bytes - 64 * 8 * 2 * 512 * 128 * 4, rel=0, abs=64 * 2048 * 2)


def test_kernel_source_hash_follows_includes_only():
    # a kernel's hash covers its file, the csrc headers it includes
    # (transitively) and the host launch code, not unrelated headers
    h1 = bench.kernel_source_sha("diag")
    assert h1 == bench.kernel_source_sha("diag") and len(h1) == 16
    assert bench.kernel_source_sha("tcgen05") != h1
    csrc = os.path.join(bench.ROOT, "cross_model_kv_transfer_gb300", "csrc")
    tc = open(os.path.join(csrc, "kvx_tcgen05.cu")).read()
    assert '#include "kvx_async.cuh"' not in tc     # so kvx_async.cuh cannot move its hash


def test_dram_records_name_known_kernels_and_commands():
    rows = json.load(open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")))
    for r in rows:
        assert r["kernel"] in bench.KERNEL_FILES
        assert r["dram_bytes_per_launch"] == r["dram_bytes_read"] + r["dram_bytes_write"]
        assert r["command"].startswith("ncu ") and "--clock-control none" in r["command"]


def test_phase_roofline_picks_the_phase_with_the_largest_ideal_time():
    peaks, _ = bench.load_peaks()
    tf32 = peaks["bf16_tflops"] * bench.TF32_PER_BF16
    # 1 ms of tensor work, 3 ms of fp64 work, 0.5 ms of HBM traffic, 10 ms call
    r = bench.phase_roofline(10.0, tf32 * 1e9, bench.NOMINAL_FP64_TFLOPS * 3e9,
                             peaks["hbm_gbs"] * 0.5e6, "ridge", "none")
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert abs(r["ideal_ms"]["tensor"] - 1.0) < 1e-3 and abs(r["ideal_ms"]["alu"] - 3.0) < 1e-3
    assert abs(r["frac"] - 0.3) < 1e-9 and abs(r["frac_of_ideal_sum"] - 0.45) < 1e-6
    r = bench.phase_roofline(2.0, tf32 * 1e9, 0.0, 0.0, "ridge", "none")
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-9 and r["traffic"] is None


def test_feature_bytes_count_named_source_layers_once_and_both_outputs():
    import torch
    from cross_model_kv_transfer_gb300.workloads import WORKLOADS
    wl = WORKLOADS["qwen3_14b_32b"]
    table = torch.tensor([[0, 1, 2, 3], [3, 2, 1, 0]] * 32, dtype=torch.int32)
    row = 32768 * 8 * 128 * 2 * 2                  # one layer's K and V, bf16
    out = 64 * 8 * 2 * 32768 * (4 * 128 + 128) * 4  # x and y, fp32
    assert bench.feature_bytes(wl, table, 2) == (4 + 64) * row + out
