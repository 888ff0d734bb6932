"""The C-ABI library builds, loads, exports every symbol of include/kvx.h, and
rejects bad descriptors / arguments on the host (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from cross_model_kv_transfer_gb300 import kvx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def _declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[\w\s\*]+?\b(kvx_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    lib = kvx.load()
    declared = _declared_functions()
    assert {"kvx_plan_create", "kvx_transfer", "kvx_plan_destroy"} <= declared
    for name in sorted(declared):
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", kvx.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvx_\w+)", out))
    assert declared <= exported


def test_ctypes_structs_match_the_c_layout(tmp_path):
    # Compile a probe against include/kvx.h that prints sizes and offsets.
    fields = {"kvx_plan_desc": kvx.PlanDesc, "kvx_transfer_args": kvx.TransferArgs,
              "kvx_diag_args": kvx.DiagArgs, "kvx_ridge_args": kvx.RidgeArgs,
              "kvx_score_args": kvx.ScoreArgs, "kvx_feature_args": kvx.FeatureArgs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kvx.h"', "int main(void){"]
    for cname, cls in fields.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(ln.split() for ln in subprocess.run([str(exe)], capture_output=True, text=True,
                                                    check=True).stdout.splitlines())
    for cname, cls in fields.items():
        assert int(got[cname]) == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(cls, f).offset, f"{cname}.{f}"


def _desc(**over):
    base = dict(src_layers=4, tgt_layers=6, src_kv_heads=2, tgt_kv_heads=2, src_head_dim=64,
                tgt_head_dim=64, k=2, rope_theta_src=1e4, rope_theta_tgt=1e4,
                kv_dtype=kvx.KVX_F32, w_dtype=kvx.KVX_F32, b_dtype=kvx.KVX_F32,
                dst_layout=kvx.KVX_CONTIGUOUS, block_size=0, max_position=128,
                kernel=kvx.KVX_KERNEL_AUTO)
    base.update(over)
    return kvx.PlanDesc(**base)


@pytest.mark.parametrize("over,want", [
    (dict(src_layers=0), kvx.KVX_ERR_INVALID_ARG),
    (dict(tgt_layers=-1), kvx.KVX_ERR_INVALID_ARG),
    (dict(k=0), kvx.KVX_ERR_INVALID_ARG),
    (dict(src_head_dim=63, tgt_head_dim=63), kvx.KVX_ERR_INVALID_ARG),
    (dict(src_head_dim=512, tgt_head_dim=512), kvx.KVX_ERR_INVALID_ARG),
    (dict(rope_theta_src=0.0), kvx.KVX_ERR_INVALID_ARG),
    (dict(rope_theta_tgt=float("nan")), kvx.KVX_ERR_INVALID_ARG),
    (dict(kv_dtype=7), kvx.KVX_ERR_INVALID_ARG),
    (dict(dst_layout=2), kvx.KVX_ERR_INVALID_ARG),
    (dict(dst_layout=kvx.KVX_PAGED, block_size=0), kvx.KVX_ERR_INVALID_ARG),
    (dict(max_position=0), kvx.KVX_ERR_INVALID_ARG),
    (dict(kernel=9), kvx.KVX_ERR_INVALID_ARG),
    (dict(mapper=2), kvx.KVX_ERR_INVALID_ARG),
    (dict(max_tokens=-1), kvx.KVX_ERR_INVALID_ARG),
    (dict(src_layout=2), kvx.KVX_ERR_INVALID_ARG),
    (dict(src_layout=kvx.KVX_PAGED, src_block_size=0), kvx.KVX_ERR_INVALID_ARG),
    # "Requirements": same number of KV heads and the same head dimension
    (dict(tgt_kv_heads=4), kvx.KVX_ERR_PAIR_MISMATCH),
    (dict(tgt_head_dim=128), kvx.KVX_ERR_PAIR_MISMATCH),
])
def test_bad_descriptor_is_refused_before_touching_the_device(over, want):
    st, h = kvx.kvx_plan_create(_desc(**over))
    assert st == want and h is None


def test_tensor_core_kernel_refuses_fp32_caches():
    st, h = kvx.kvx_plan_create(_desc(kernel=kvx.KVX_KERNEL_TCGEN05))
    assert st == kvx.KVX_ERR_UNSUPPORTED and h is None


def test_valid_descriptor_without_gpu_reports_unsupported():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = kvx.kvx_plan_create(_desc())
    assert st == kvx.KVX_ERR_UNSUPPORTED and h is None


def test_transfer_and_destroy_reject_null():
    assert kvx.kvx_transfer(None, kvx.TransferArgs(), None) == kvx.KVX_ERR_INVALID_ARG
    assert kvx.load().kvx_transfer(None, None, None) == kvx.KVX_ERR_INVALID_ARG
    assert kvx.kvx_plan_destroy(None) == kvx.KVX_OK
    assert kvx.kvx_plan_kernel(None) == -1
    assert kvx.kvx_plan_launches(None) == -1
    assert kvx.kvx_kv_diagnostics(None, kvx.DiagArgs(), None) == kvx.KVX_ERR_INVALID_ARG
    assert kvx.load().kvx_kv_diagnostics(None, None, None) == kvx.KVX_ERR_INVALID_ARG


def test_status_strings():
    for s in range(7):
        assert kvx.kvx_status_string(s) not in ("", "unknown status")
    assert kvx.kvx_status_string(99) == "unknown status"


def test_ridge_workspace_size_and_host_validation():
    # 8 bytes per column sum, Gram entry and cross product, each block
    # rounded up to 256 bytes, the hi and lo fp32 planes of one chunk of
    # 16,384 observations of every feature and output, the fp64 inverses of
    # the factor's 64 x 64 diagonal blocks, and one fp64 shift per column
    r = lambda x: (x + 255) // 256 * 256
    assert kvx.kvx_ridge_workspace_bytes(3, 10, 4) == \
        r(8 * 3 * 14) + r(8 * 3 * 100) + r(8 * 3 * 40) + r(2 * 4 * 3 * 14 * 16384) + \
        r(3 * 64 * 64 * 8) + 8 * 3 * 14
    assert kvx.kvx_ridge_workspace_bytes(0, 10, 4) == 0
    assert kvx.kvx_ridge_workspace_bytes(1, 5000, 4) == 0
    assert kvx.load().kvx_ridge_fit(None, None) == kvx.KVX_ERR_INVALID_ARG
    a = kvx.RidgeArgs(1, 10, 4, 2, 0.01, kvx.KVX_F32, 16, 16, 16, 16, 16, 0, None)
    assert kvx.kvx_ridge_fit(a, None) == kvx.KVX_ERR_INVALID_ARG      # workspace too small
    a = kvx.RidgeArgs(1, 10, 4, 2, float("inf"), kvx.KVX_F32, 16, 16, 16, 16, 16, 1 << 20, None)
    assert kvx.kvx_ridge_fit(a, None) == kvx.KVX_ERR_INVALID_ARG      # lambda not finite
    # more observations than 65,535 slices of 16,384 is refused before any launch
    a = kvx.RidgeArgs(1, 65535 * 16384 + 1, 4, 2, 0.01, kvx.KVX_F32, 16, 16, 16, 16, 16, 1 << 20,
                      None)
    assert kvx.kvx_ridge_fit(a, None) == kvx.KVX_ERR_INVALID_ARG


def test_ridge_features_rejects_null_before_touching_the_device():
    lib = kvx.load()
    assert lib.kvx_ridge_features(None, None, None) == kvx.KVX_ERR_INVALID_ARG
    a = kvx.FeatureArgs()
    assert kvx.kvx_ridge_features(None, a, None) == kvx.KVX_ERR_INVALID_ARG
