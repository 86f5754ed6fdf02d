"""The CPU oracle and the input generator under AddressSanitizer and UBSan (no
GPU): tests/oracle_sanitize_main.c compiles oracle/oracle.c and synth/gen.c
with -fsanitize=address,undefined (the oracle's own flags otherwise:
-ffp-contract=off) and runs small layers of several shapes through routing,
the sparse layer against its dense brute force, both cache policies and pair
grouping. A memory error or undefined behaviour in the oracle would make its
expected values untrustworthy, so it fails the test."""
import os
import shutil
import subprocess

import pytest

from tests.conftest import ROOT


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_oracle_is_clean_under_address_and_ub_sanitizers(tmp_path):
    probe = tmp_path / "probe.c"
    probe.write_text("int main(void){return 0;}\n")
    if subprocess.run(["gcc", "-fsanitize=address,undefined", str(probe), "-o", str(tmp_path / "p")],
                      capture_output=True).returncode != 0:
        pytest.skip("sanitizer runtimes not available")
    exe = str(tmp_path / "oracle_san")
    cmd = ["gcc", "-std=c11", "-O1", "-g", "-ffp-contract=off", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=undefined", os.path.join(ROOT, "tests", "oracle_sanitize_main.c"), "-o", exe,
           "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1 exitcode=66", UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0 and "oracle ok" in r.stdout, r.stdout + r.stderr[-4000:]
