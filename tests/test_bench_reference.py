"""The benchmark's reference arm (the fp64 oracle on the host cores), run on
the CPU: one JSON line with the GPU arm's metric and workload config for
every op, a cpu_baseline describing the sample, a zero-copy e2e, no GPU
launches; under torchrun only rank 0 prints."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from cross_model_kv_transfer_gb300.workloads import WORKLOADS  # noqa: E402

MODES = {
    "transfer": [],
    "wide": ["--mapper", "wide"],
    "paged_source": ["--src-block-size", "16"],
    "kv_diagnostics": ["--op", "kv_diagnostics"],
    "ridge_fit": ["--op", "ridge_fit"],
    "layer_scores": ["--op", "layer_scores"],
    "ridge_features": ["--op", "ridge_features"],
    "small_override": ["--tokens", "4096", "--tgt-layers", "8"],
}


def _lines(out: str):
    return [json.loads(s) for s in out.splitlines() if s.startswith("{")]


def _run(extra, timeout=300):
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"] + extra, capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    return _lines(p.stdout)


@pytest.mark.parametrize("mode", list(MODES))
def test_reference_line_matches_the_gpu_arm_contract(mode):
    extra = MODES[mode]
    lines = _run(extra)
    assert len(lines) == 1
    d = lines[0]
    args = bench.parse_args(extra)
    if args.op == "ridge_fit":
        wl = WORKLOADS[args.workload]
        metric, unit = bench.RIDGE_METRIC, "fits/s"
        config = bench.ridge_config(wl, args.ridge_batch, args.ridge_n)
    elif args.op == "layer_scores":
        wl = WORKLOADS[args.workload].with_tokens([args.score_tokens], [0])
        metric, unit = bench.SCORE_METRIC, "tokens/s"
        config = bench.score_config(wl, args.score_tokens)
    elif args.op == "ridge_features":
        wl = WORKLOADS[args.workload]
        metric, unit, config = bench.FEATURE_METRIC, "tokens/s", bench.feature_config(wl)
    elif args.op == "kv_diagnostics":
        wl = bench.select_workload(args)
        metric, unit, config = bench.DIAG_METRIC, "tokens/s", bench.diag_config(wl)
    else:
        wl = bench.select_workload(args)
        metric, unit = bench.transfer_metric(wl, args.mapper == "wide"), "tokens/s"
        config = bench.transfer_config(wl, args)
    assert d["impl"] == "reference"
    assert d["metric"] == metric and d["unit"] == unit and d["config"] == config
    assert ("op" in d) == (args.op != "transfer")
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3 and d["vs_baseline"] is None
    assert d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["value"] == d["value"] and cb["unit"] == unit and cb["kind"] == "oracle"
    assert cb["cores"] == 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["gpu_launches"] == 0


def test_override_flags_select_a_smaller_workload():
    args = bench.parse_args(["--tokens", "4096", "--tgt-layers", "8"])
    wl = bench.select_workload(args)
    assert wl.ntok == 4096 and wl.tgt_layers == 8
    assert wl.name == "qwen3_14b_32b@4096/Lt8"
    assert bench.transfer_metric(wl, False).startswith("KV-transfer tokens/s, qwen3_14b_32b@4096")
    base = bench.select_workload(bench.parse_args([]))
    assert base is WORKLOADS["qwen3_14b_32b"] and bench.transfer_metric(base, False) == bench.METRIC


def test_reference_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", "29761",
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _lines(p.stdout)
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
