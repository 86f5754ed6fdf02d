"""The pins catch plausible mistakes in the oracle.

Each case copies oracle/oracle.c to a scratch directory, plants one mistake
(a dropped term, a wrong sign, index, order or tie-break, a transposed or
swapped operand, a wrong cache rule), and runs tests/test_oracle_pins.py
against that copy (MOE_ORACLE_SOURCE): at least one pin must fail. The
unchanged copy, run the same way, must pass. Nothing here touches the
library or a GPU."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from tests.conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "oracle.c")

# name: (text in oracle.c, its replacement); each text occurs exactly once
MUTATIONS = {
    "gelu without the cubic term": (
        "0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)))", "0.5 * z * (1.0 + tanh(c * z))"),
    "silu as the bare sigmoid": (
        "if (act == ACT_SILU) return z / (1.0 + exp(-z));", "if (act == ACT_SILU) return 1.0 / (1.0 + exp(-z));"),
    "nibbles swapped": (
        "return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15u);",
        "return (k & 1) ? (unsigned)(byte & 15u) : (unsigned)(byte >> 4);"),
    "bias subtracted": (
        "* (double)oracle_code_u4(codes, K, n, k) + oracle_f16(bias[g]);",
        "* (double)oracle_code_u4(codes, K, n, k) - oracle_f16(bias[g]);"),
    "groups of 128": (
        "size_t g = (size_t)n * (size_t)(K / 64) + (size_t)(k / 64);\n    return oracle_f16(scale[g]) * (double)oracle_code_u4",
        "size_t g = (size_t)n * (size_t)(K / 64) + (size_t)(k / 128);\n    return oracle_f16(scale[g]) * (double)oracle_code_u4"),
    "router without its bias term": (
        "float w = fmaf(s, (float)codes[(size_t)e * (size_t)d + (size_t)i], b);",
        "float w = s * (float)codes[(size_t)e * (size_t)d + (size_t)i];"),
    "zbias ignored": ("if (zbias) logit = logit + zbias[e];", "(void)zbias;"),
    "bf16 decoded one bit off": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "ties to the higher index": (
        "return l[a] > l[b] || (l[a] == l[b] && a < b);", "return l[a] > l[b] || (l[a] == l[b] && a > b);"),
    "gates not renormalised": (
        "gates[(size_t)t * (size_t)k + (size_t)r] = p / sel;", "gates[(size_t)t * (size_t)k + (size_t)r] = p;"),
    "gate and up swapped": ("h[j] = oracle_act(g, act) * u;", "h[j] = oracle_act(u, act) * g;"),
    "down matrix transposed": (
        "acc += oracle_w4(dc, ds, db, inter, n, j) * h[j];", "acc += oracle_w4(dc, ds, db, d, j, n) * h[j];"),
    "shared expert left out": (
        "oracle_shared_ffn(L, xt, yt);\n        for (int r = 0; r < L->k; ++r) {",
        "memset(yt, 0, sizeof(double) * (size_t)L->d);\n        for (int r = 0; r < L->k; ++r) {"),
    "lfu ties to the higher slot": (
        "c->count[s] < c->count[victim] : c->tick[s] < c->tick[victim]",
        "c->count[s] <= c->count[victim] : c->tick[s] < c->tick[victim]"),
    "lru evicts the newest": (
        "c->count[s] < c->count[victim] : c->tick[s] < c->tick[victim]",
        "c->count[s] < c->count[victim] : c->tick[s] > c->tick[victim]"),
    "new entries start at zero": ("c->count[victim] = 1;", "c->count[victim] = 0;"),
    "highest empty slot first": (
        "for (int s = 0; s < c->S && victim < 0; ++s)\n            if (c->slot_expert[s] < 0) victim = s;",
        "for (int s = c->S - 1; s >= 0 && victim < 0; --s)\n            if (c->slot_expert[s] < 0) victim = s;"),
    "hits not counted": ("                c->count[s] += 1;\n", "                c->count[s] += 0;\n"),
    "grouping not stable": (
        "for (int p = 0; p < n_pairs; ++p)\n            if (ids[p] == e) perm[pos++] = p;",
        "for (int p = n_pairs - 1; p >= 0; --p)\n            if (ids[p] == e) perm[pos++] = p;"),
}


def _run_pins(tmp, name, text):
    d = os.path.join(tmp, name.replace(" ", "_"))
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "oracle.c")
    with open(src, "w") as f:
        f.write(text)
    if subprocess.run(["gcc", "-fsyntax-only", "-std=c11", src], capture_output=True).returncode != 0:
        return name, None, "does not compile"
    env = dict(os.environ, MOE_ORACLE_SOURCE=src)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-q",
                        "-x", "-p", "no:cacheprovider"], capture_output=True, text=True, env=env, cwd=ROOT,
                       timeout=600)
    return name, r.returncode, r.stdout[-600:]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_every_planted_mistake_fails_a_pin(tmp_path):
    original = open(SRC).read()
    cases = {"(unchanged)": original}
    for name, (old, new) in MUTATIONS.items():
        assert original.count(old) == 1, name
        cases[name] = original.replace(old, new)
    with ThreadPoolExecutor(min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda kv: _run_pins(str(tmp_path), *kv), cases.items()))
    for name, rc, out in results:
        assert rc is not None, (name, out)
        if name == "(unchanged)":
            assert rc == 0, out
        else:
            assert rc == 1 and "failed" in out, (name, rc, out)
