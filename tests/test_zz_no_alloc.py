"""moe_route_noalloc: the router with library-owned static scratch.

Callers that cannot allocate device memory (a decode loop on a fixed memory
budget, or one that cannot take the device-wide synchronisation a cudaFree
would add) route through this entry point. It must give the oracle's ids
(bit-exact) and gates (within 1e-6), and what moe_route gives, on calls in a
row: each call finds the static arrays as the previous call left them, and
calls for layers of different widths share them. Calls larger than the
static scratch are refused before anything is enqueued. The file sorts last
so that it also runs after every other GPU test has used the library in the
same process.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import expert_streaming_ffn_gb300 as moe  # noqa: E402

GATE_TOL = 1e-6
SHAPES_WIDE = synth.Shapes(512, 512, 8, 64, 64, synth.GELU_TANH)  # 512 experts: T * E reaches the limit at T = 33


@pytest.fixture(scope="module")
def layers():
    moe.load()
    ctx = moe.moe_ctx_create(0)
    out = {}
    for name, s, seed in (("2816", synth.SHAPES_2816, 7), ("tiny", synth.SHAPES_TINY, 8), ("wide", SHAPES_WIDE, 9)):
        w = synth.layer_weights(s, 3, seed)
        h = moe.moe_layer_create(ctx, s, 16, moe.LFU)
        moe.moe_layer_set_weights(h, w)
        out[name] = (s, h, w, seed)
    yield out
    for s, h, w, seed in out.values():
        moe.moe_layer_destroy(h)
    moe.moe_ctx_destroy(ctx)


def _route_and_check(entry, T, step, zipf=None):
    """One moe_route_noalloc call against the oracle and against moe_route."""
    s, h, w, seed = entry
    xb = synth.tokens(s, 3, step, T, True, seed)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    zb_np = None if zipf is None else synth.zipf_bias(s, 3, zipf, 1.0, seed)
    zb = None if zb_np is None else torch.from_numpy(zb_np).cuda()
    ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
    gates = torch.full((T, s.top_k), -1.0, dtype=torch.float32, device="cuda")
    moe.moe_route_noalloc(h, x, zb, ids, gates)
    torch.cuda.synchronize()
    oids, og = oracle.topk_gates(oracle.router_logits(xb, w.router, s.n_experts, zb_np), s.top_k)
    assert (ids.cpu().numpy() == oids).all(), "expert ids differ from the oracle"
    assert np.abs(gates.cpu().numpy() - og).max() <= GATE_TOL
    ids_ref, gates_ref = moe.moe_route(h, x, s.top_k, zb)
    torch.cuda.synchronize()
    assert torch.equal(ids.cpu(), ids_ref.cpu())
    assert (gates - gates_ref).abs().max().item() <= GATE_TOL


@pytest.mark.parametrize("T", [1, 8, 13, 64])
def test_noalloc_matches_oracle_twice(layers, T):
    for step in range(2):
        _route_and_check(layers["2816"], T, step, zipf=1.1)


def test_noalloc_layers_of_different_width_share_the_scratch(layers):
    # 16 and 256 experts, alternately: each call's logits overwrite a different
    # extent of the same array, and each must still route exactly
    for step in range(3):
        _route_and_check(layers["tiny"], 5, step)
        _route_and_check(layers["2816"], 3, step, zipf=1.1)
        _route_and_check(layers["tiny"], 64, 10 + step)


def test_noalloc_wide_layer_at_its_limit(layers):
    # 512 experts (the top-k path for more than 256 candidates): T = 32 fills
    # the 16384 logits exactly; T = 33 (T <= 64, but T * E over the limit) is
    # refused before anything is enqueued, and the scratch stays usable
    s, h, w, seed = layers["wide"]
    _route_and_check(layers["wide"], 32, 0)
    xb = synth.tokens(s, 3, 1, 33, True, seed)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    ids = torch.full((33, s.top_k), -7, dtype=torch.int32, device="cuda")
    gates = torch.full((33, s.top_k), -7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError, match="exceeds the static scratch"):
        moe.moe_route_noalloc(h, x, None, ids, gates)
    torch.cuda.synchronize()
    assert (ids.cpu() == -7).all() and (gates.cpu() == -7.0).all()  # nothing ran
    _route_and_check(layers["wide"], 32, 2)


def test_noalloc_rejects_calls_over_its_scratch(layers):
    s, h, w, seed = layers["2816"]
    T = 65
    xb = synth.tokens(s, 3, 0, T, True, seed)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    ids = torch.empty((T, s.top_k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, s.top_k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError, match="exceeds the static scratch"):
        moe.moe_route_noalloc(h, x, None, ids, gates)
    # the refusal left the scratch usable
    _route_and_check(layers["2816"], 4, 5)
