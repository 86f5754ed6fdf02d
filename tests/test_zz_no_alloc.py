"""moe_route_noalloc: the router with library-owned static scratch.

It must give what moe_route gives (same kernel, same fixed summation order)
on two calls in a row (the second call finds the counters the first left
behind), and refuse calls larger than its static scratch before enqueuing
anything. The file sorts last so that it also runs after every other GPU
test has used the library in the same process.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import expert_streaming_ffn_gb300 as moe  # noqa: E402

GATE_TOL = 1e-6


@pytest.fixture(scope="module")
def layer():
    moe.load()
    ctx = moe.moe_ctx_create(0)
    s = synth.WORKLOADS["decode_2816"].shapes
    h = moe.moe_layer_create(ctx, s, 16, moe.LFU)
    moe.moe_layer_set_weights(h, synth.layer_weights(s, 3, 7))
    yield s, h
    moe.moe_layer_destroy(h)
    moe.moe_ctx_destroy(ctx)


def _x(s, T, step):
    xb = synth.tokens(s, 3, step, T, True, 7)
    return torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("T", [1, 8, 13, 64])
def test_noalloc_matches_moe_route_twice(layer, T):
    s, h = layer
    zb = torch.from_numpy(synth.zipf_bias(s, 3, 1.1, 1.0, 7)).cuda()
    for step in range(2):
        x = _x(s, T, step)
        ids_ref, gates_ref = moe.moe_route(h, x, s.top_k, zb)
        ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
        gates = torch.full((T, s.top_k), -1.0, dtype=torch.float32, device="cuda")
        moe.moe_route_noalloc(h, x, zb, ids, gates)
        torch.cuda.synchronize()
        assert torch.equal(ids.cpu(), ids_ref.cpu())
        assert (gates - gates_ref).abs().max().item() <= GATE_TOL


def test_noalloc_rejects_calls_over_its_scratch(layer):
    s, h = layer
    T = 65
    x = _x(s, T, 0)
    ids = torch.empty((T, s.top_k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, s.top_k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError, match="exceeds the static scratch"):
        moe.moe_route_noalloc(h, x, None, ids, gates)
    # the refusal left the scratch usable
    ids_ref, gates_ref = moe.moe_route(h, x[:4], s.top_k)
    moe.moe_route_noalloc(h, x[:4], None, ids[:4], gates[:4])
    torch.cuda.synchronize()
    assert torch.equal(ids[:4].cpu(), ids_ref.cpu())
