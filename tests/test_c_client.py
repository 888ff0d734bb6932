"""The C ABI from plain C (CPU only): ``tests/c/kvx_c_client.c`` is compiled
as strict C99 against ``include/kvx.h``, linked against ``libkvx.so`` and run;
it checks the answers of every call that needs no GPU (validation, NULL
handles, the ridge scratch size, the status strings)."""
import os
import shutil
import subprocess

import pytest

from cross_model_kv_transfer_gb300 import kvx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_compiles_links_and_gets_the_documented_answers(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib = kvx.load()._name
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "kvx_c_client")
    cc = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
          "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "kvx_c_client.c"),
          "-L", libdir, "-lkvx", f"-Wl,-rpath,{libdir}", "-o", exe]
    subprocess.run(cc, check=True, capture_output=True, text=True)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, f"check {p.returncode} failed: {p.stdout}{p.stderr}"
    lines = p.stdout.strip().splitlines()
    assert lines[-1] == "ok"
    assert lines[0] == "0 ok" and lines[6].startswith("6 RoPE tables exceed")
