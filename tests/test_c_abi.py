"""The boundary is a plain C ABI: a C program compiled against include/moe.h
and linked to libmoe.so runs its host-side checks (no GPU, no Python types)."""
import os
import shutil
import subprocess

import pytest

from sparse_moe_layer_fwd_b300 import moe as M

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_uses_the_abi(tmp_path):
    exe = tmp_path / "abi_host"
    lib_dir = os.path.dirname(M.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-o", str(exe),
                    os.path.join(HERE, "c", "abi_host.c"), "-I", os.path.join(ROOT, "include"),
                    "-L", lib_dir, "-lmoe", f"-Wl,-rpath,{lib_dir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "passed" in r.stdout
