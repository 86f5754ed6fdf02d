"""Host-side checks of libmoe that need no GPU.

* the shared library loads and exports every function include/moe.h declares;
* the library's host cache manager reproduces the oracle's cache trace (a
  separate implementation of the same rules) on random id sequences and on
  the hand-replayed golden traces;
* the library's prefill pair grouping equals the oracle's stable grouping.
"""
import json
import os
import re

import numpy as np
import pytest

import expert_streaming_ffn_gb300 as moe
import oracle
from tests.conftest import GOLDEN, ROOT


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = moe.load()
    declared = _declared_functions()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), name
    bound = {n for n, _, _ in moe.SIGNATURES}
    assert set(declared) == bound, set(declared) ^ bound


def test_status_strings():
    assert moe.moe_status_str(moe.MOE_ECOPY) == "MOE_ECOPY"
    assert moe.moe_status_str(moe.MOE_OK) == "MOE_OK"


def test_expert_bytes_matches_canonical_count():
    import synth

    for s in (synth.SHAPES_TINY, synth.SHAPES_2816, synth.SHAPES_2048):
        assert moe.moe_expert_bytes(s) == synth.expert_bytes(s)
    assert moe.moe_expert_bytes(synth.SHAPES_2816) == 3345408


def test_host_cache_rejects_bad_arguments():
    with pytest.raises(moe.MoeError):
        moe.moe_host_cache_create(16, 0, moe.LFU)
    with pytest.raises(moe.MoeError):
        moe.moe_host_cache_create(16, 17, moe.LFU)
    with pytest.raises(moe.MoeError):
        moe.moe_host_cache_create(16, 4, 7)
    c = moe.moe_host_cache_create(16, 4, moe.LFU)
    try:
        with pytest.raises(moe.MoeError):
            moe.moe_host_cache_step(c, [3, 16])
    finally:
        moe.moe_host_cache_destroy(c)


def test_host_cache_golden_traces():
    with open(os.path.join(GOLDEN, "lfu_toy_trace.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        pol = moe.LFU if case["policy"] == "lfu" else moe.LRU
        c = moe.moe_host_cache_create(case["experts"], case["slots"], pol)
        try:
            for step, exp in zip(case["steps"], case["expected"]):
                r = moe.moe_host_cache_step(c, step)
                se, cnt = moe.moe_host_cache_dump(c, case["slots"])
                assert r["hits"] == exp["hits"] and r["misses"] == exp["misses"], (case["name"], step)
                assert r["miss_slots"].tolist() == exp["miss_slots"], (case["name"], step)
                assert se.tolist() == exp["slot_expert"], (case["name"], step)
                if "counts" in exp:
                    assert cnt.tolist() == exp["counts"]
        finally:
            moe.moe_host_cache_destroy(c)


@pytest.mark.parametrize("E,S,policy,batch", [(16, 4, moe.LFU, 2), (256, 16, moe.LFU, 8), (256, 64, moe.LRU, 64),
                                              (256, 16, moe.LRU, 8), (64, 1, moe.LFU, 3), (256, 256, moe.LFU, 8),
                                              (1024, 32, moe.LFU, 128), (256, 16, moe.LRU, 1024),
                                              (256, 256, moe.LFU, 2048)])
def test_host_cache_matches_oracle_trace(E, S, policy, batch):
    rng = np.random.default_rng(E * 7 + S + policy)
    c = moe.moe_host_cache_create(E, S, policy)
    ref = oracle.Cache(E, S, policy)
    try:
        for step in range(400):
            n = int(rng.integers(1, batch + 1))
            # skewed ids so that hits, evictions and bypasses all occur
            ids = (rng.zipf(1.2, n) - 1 + step // 50) % E
            r = moe.moe_host_cache_step(c, ids)
            o = ref.step(ids)
            for key in ("hits", "misses", "bypass"):
                assert r[key] == o[key], (step, key)
            assert (r["slot_of"] == o["slot_of"]).all(), step
            assert (r["miss_experts"] == o["miss_experts"]).all(), step
            assert (r["miss_slots"] == o["miss_slots"]).all(), step
            se, cnt = moe.moe_host_cache_dump(c, S)
            ose, ocnt = ref.dump()
            assert (se == ose).all() and (cnt == ocnt).all(), step
    finally:
        moe.moe_host_cache_destroy(c)


def test_group_pairs_matches_oracle():
    rng = np.random.default_rng(2)
    for E, n in ((16, 8), (256, 1024), (256, 1), (1024, 777)):
        ids = rng.integers(0, E, n).astype(np.int32)
        off, perm = moe.moe_group_pairs(ids, E)
        ooff, operm = oracle.group_pairs(ids, E)
        assert (off == ooff).all() and (perm == operm).all()
    with pytest.raises(moe.MoeError):
        moe.moe_group_pairs(np.array([0, 5], np.int32), 5)


def test_ctx_create_without_device_fails_cleanly():
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_ctx_create(0)
    assert ei.value.status == moe.MOE_EINVAL
