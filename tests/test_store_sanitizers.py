"""The expert store and the host cache manager under the sanitizers (no GPU):
store.cpp and host_cache.cpp built alone with
g++ -fsanitize=thread (and, separately, -fsanitize=address,undefined) and
driven by tests/store_sanitize_main.cpp from four threads (fetch, release,
readahead) against its own reader threads, with whole-expert reads and with
reads in pieces; the cache manager on random steps of up to 512 ids under
both policies with its invariants checked. A data race, a memory error,
undefined behaviour, a wrong byte, a broken invariant or a lost fetch fails
the test."""
import os
import shutil
import subprocess

import pytest

import expert_streaming_ffn_gb300 as moe
import synth
from tests.conftest import ROOT

SHAPES = synth.Shapes(512, 8, 2, 192, 512, synth.GELU_TANH)


def _sanitizer_works(tmp_path, flag) -> bool:
    src = tmp_path / "probe.cpp"
    src.write_text("#include <thread>\nint main(){std::thread t([]{});t.join();}\n")
    exe = str(tmp_path / "probe")
    r = subprocess.run(["g++", flag, str(src), "-o", exe], capture_output=True)
    return r.returncode == 0 and subprocess.run([exe]).returncode == 0


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
@pytest.mark.parametrize("sanitizer,options", [
    ("thread", {"TSAN_OPTIONS": "halt_on_error=1 exitcode=66"}),
    ("address,undefined", {"ASAN_OPTIONS": "detect_leaks=1 exitcode=66",
                           "UBSAN_OPTIONS": "halt_on_error=1 print_stacktrace=1 exitcode=66"}),
])
def test_store_under_sanitizers(tmp_path, sanitizer, options):
    flag = f"-fsanitize={sanitizer}"
    if not _sanitizer_works(tmp_path, flag):
        pytest.skip(f"{flag} runtime not available")
    exe = str(tmp_path / "store_san")
    cmd = ["g++", "-std=c++17", "-O1", "-g", flag, "-fno-sanitize-recover=undefined"
           if "undefined" in sanitizer else "-O1", "-I", os.path.join(ROOT, "include"),
           "-I", "/usr/local/cuda/include", os.path.join(ROOT, "expert_streaming_ffn_gb300", "csrc", "store.cpp"),
           os.path.join(ROOT, "expert_streaming_ffn_gb300", "csrc", "host_cache.cpp"),
           os.path.join(ROOT, "tests", "store_sanitize_main.cpp"), "-o", exe, "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    path = str(tmp_path / "layer.experts")
    moe.moe_store_write(path, SHAPES, synth.layer_weights(SHAPES, 3, 5))
    env = dict(os.environ, **options)
    for chunk in (0, 16384):
        r = subprocess.run([exe, path, str(chunk)], capture_output=True, text=True, timeout=300, env=env)
        assert r.returncode == 0, (chunk, r.stdout, r.stderr[-4000:])
        assert "bad 0" in r.stdout
