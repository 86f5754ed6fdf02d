"""GPU parity on the stress sweep: the 2816 shapes with uniform routing.

Decode batches of 1, 4, 16 and 64 tokens against caches of 8, 16 and 64
slots, and a 4096-token prefill (32 chunks of 128). Expert ids and the cache
trace must match the oracle exactly at every point; layer outputs are
checked on sampled tokens (same bars as test_gpu_parity.py).
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import expert_streaming_ffn_gb300 as moe  # noqa: E402
from test_gpu_parity import Rig  # noqa: E402

WL = synth.WORKLOADS["stress_2816"]


@pytest.fixture(scope="module")
def ctx():
    moe.load()
    c = moe.moe_ctx_create(0)
    yield c
    moe.moe_ctx_destroy(c)


@pytest.fixture(scope="module")
def weights():
    return synth.layer_weights(WL.shapes, 11, WL.seed)


@pytest.mark.parametrize("S", [8, 16, 64])
@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_stress_decode(ctx, weights, T, S):
    s = WL.shapes
    r = Rig(ctx, s, 11, S, weights=weights)
    try:
        for step in range(3):
            x = synth.tokens(s, 11, 100 * T + step, T, True)
            r.forward(x, None, check_y=step == 2, y_tokens=sorted({0, T // 2, T - 1}))
        st = moe.moe_layer_stats(r.h)
        assert st["steps"] == 3 and st["hits"] + st["misses"] > 0
        if T * s.top_k > S:
            assert st["misses"] > 0
    finally:
        r.close()


def test_stress_prefill_4096(ctx, weights):
    s = WL.shapes
    r = Rig(ctx, s, 11, 16, weights=weights)
    try:
        x = synth.tokens(s, 11, 7, 4096, True)
        r.forward(x, None, y_tokens=[0, 127, 128, 2047, 2100, 4095])
        st = moe.moe_layer_stats(r.h)
        assert st["steps"] == 32 and st["bypass"] > 0
    finally:
        r.close()
