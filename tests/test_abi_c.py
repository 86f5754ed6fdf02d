"""include/moe.h from plain C: a C99 program (tests/abi_check.c) compiles
against the header with warnings as errors, links libmoe.so and calls the
host-only entry points (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

import expert_streaming_ffn_gb300 as moe
from tests.conftest import ROOT


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_compiles_as_c99_and_host_calls_work(tmp_path):
    moe.load()
    build = os.path.dirname(moe.LIB_PATH)
    exe = str(tmp_path / "abi_check")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "abi_check.c"), "-o", exe, f"-L{build}", "-lmoe", f"-Wl,-rpath,{build}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe, str(tmp_path / "no_such_file")], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "abi ok" in r.stdout, r.stdout + r.stderr
