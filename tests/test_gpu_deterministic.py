"""The ordered decode combine (moe_layer_set_deterministic) on the GPU.

With it on, a decode call's y is summed in a fixed order (the shared expert's
share, then the routed experts' in rank order), so repeating a call on the
same x gives the same bits even though the cache state differs between the
calls (misses the first time, hits after). Ids, gates and the cache trace must
still match the oracle exactly, and y within the usual tolerance.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import expert_streaming_ffn_gb300 as moe  # noqa: E402

Y_TOL = 2e-3


@pytest.fixture(scope="module")
def ctx():
    moe.load()
    c = moe.moe_ctx_create(0)
    yield c
    moe.moe_ctx_destroy(c)


@pytest.mark.parametrize("shapes,slots,T", [(synth.SHAPES_TINY, 4, 1), (synth.SHAPES_TINY, 4, 5),
                                            (synth.SHAPES_2816, 16, 1), (synth.SHAPES_2816, 16, 8),
                                            (synth.SHAPES_2048, 64, 3)])
def test_ordered_combine_repeats_bit_for_bit(ctx, shapes, slots, T):
    s = shapes
    w = synth.layer_weights(s, 11)
    h = moe.moe_layer_create(ctx, s, slots, moe.LFU)
    try:
        moe.moe_layer_set_weights(h, w)
        moe.moe_layer_set_deterministic(h, True)
        ref = oracle.Layer(w, s)
        cache = oracle.Cache(s.n_experts, slots, moe.LFU)
        rms = s.n_experts != 16
        first = None
        for rep in range(3):
            for step in range(2):  # the same two inputs each round: different cache states
                xb = synth.tokens(s, 11, step, T, rms)
                x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
                ids = torch.empty((T, s.top_k), dtype=torch.int32, device="cuda")
                y = moe.moe_forward(h, x, ids_out=ids)
                torch.cuda.synchronize()
                oids, og = oracle.topk_gates(oracle.router_logits(xb, w.router, s.n_experts, None), s.top_k)
                assert (ids.cpu().numpy() == oids).all()
                cache.step(oids)
                se, cnt = moe.moe_cache_dump(h, slots)
                ose, ocnt = cache.dump()
                assert (se == ose).all() and (cnt == ocnt).all()
                if rep == 0:
                    yg = y.cpu().numpy()
                    for t in sorted({0, T - 1}):
                        yo = ref.combine(xb[t:t + 1], oids[t:t + 1], og[t:t + 1])[0]
                        assert np.abs(yg[t] - yo).max() <= Y_TOL * np.abs(yo).max()
                    if step == 0:
                        first = y.clone()
                elif step == 0:
                    assert torch.equal(y, first), f"round {rep}: y differs in its bits from the first call"
        st = moe.moe_layer_stats(h)
        assert st["hits"] > 0 and st["misses"] > 0
    finally:
        moe.moe_layer_destroy(h)


def test_ordered_and_atomic_combines_agree(ctx):
    # the same layer inputs through both modes: within fp32 rounding of each other
    s = synth.SHAPES_2816
    w = synth.layer_weights(s, 12)
    hs = [moe.moe_layer_create(ctx, s, s.n_experts, moe.LFU) for _ in range(2)]
    try:
        for h in hs:
            moe.moe_layer_set_weights(h, w)
        moe.moe_layer_set_deterministic(hs[1], True)
        xb = synth.tokens(s, 12, 0, 4, True)
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        y0 = moe.moe_forward(hs[0], x)
        y1 = moe.moe_forward(hs[1], x)
        torch.cuda.synchronize()
        assert (y0 - y1).abs().max().item() <= 1e-5 * y0.abs().max().item()
    finally:
        for h in hs:
            moe.moe_layer_destroy(h)
