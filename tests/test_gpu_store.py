"""GPU parity of layers that stream their routed experts from an expert file.

A streamed layer reads each miss from its store (a small host tier filled by
reader threads from the file) before copying it to HBM. Its routing, cache
trace and outputs must equal the oracle's exactly as a pinned-pool layer's do
(same bars as test_gpu_parity.py): the store changes where the bytes come
from, not what is computed. The tiers here are smaller than a call's misses,
so entries are recycled within a call while earlier copies are in flight.
"""
import os

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import expert_streaming_ffn_gb300 as moe  # noqa: E402
from test_gpu_parity import Rig  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    moe.load()
    c = moe.moe_ctx_create(0)
    yield c
    moe.moe_ctx_destroy(c)


class StreamedRig(Rig):
    """A Rig whose layer streams from an expert file in tmp_path."""

    def __init__(self, ctx, shapes, layer, slots, path, host_slots, readers=4, flags=moe.MOE_STORE_DIRECT,
                 policy=moe.LFU, seed=0):
        self.s = shapes
        self.w = synth.layer_weights(shapes, layer, seed)
        self.ref = oracle.Layer(self.w, shapes)
        self.cache = oracle.Cache(shapes.n_experts, slots, policy)
        self.slots = slots
        self.layer = layer
        self.path = path
        moe.moe_store_write(path, shapes, self.w)
        self.store = moe.moe_store_open(path, shapes, host_slots, readers, flags)
        self.h = moe.moe_layer_create_streamed(ctx, shapes, slots, self.store, policy)
        moe.moe_layer_set_weights(self.h, self.w, routed=False)

    def close(self):
        moe.moe_layer_destroy(self.h)
        moe.moe_store_close(self.store)


def test_streamed_tiny_decode_and_prefill(ctx, tmp_path):
    s = synth.SHAPES_TINY
    r = StreamedRig(ctx, s, 0, 4, str(tmp_path / "tiny.experts"), host_slots=2)
    try:
        for step in range(6):
            r.forward(synth.tokens(s, 0, step, 4, False))
        # 200 tokens: chunks of 128 and 72, each missing on most of the 16
        # experts with only 2 tier entries
        r.forward(synth.tokens(s, 0, 99, 200, False), y_tokens=[0, 127, 128, 199])
        st = moe.moe_store_get_stats(r.store)
        lst = moe.moe_layer_stats(r.h)
        assert st["fetches"] == lst["misses"] and st["read_errors"] == 0
        assert lst["bytes_h2d"] == lst["misses"] * moe.moe_expert_bytes(s)
    finally:
        r.close()


def test_streamed_2816_decode_with_readahead(ctx, tmp_path):
    s = synth.SHAPES_2816
    wl = synth.WORKLOADS["decode_2816"]
    r = StreamedRig(ctx, s, 13, wl.cache_slots, str(tmp_path / "l13.experts"), host_slots=12)
    zb = synth.zipf_bias(s, 13, wl.zipf_s)
    try:
        for step in range(10):
            moe.moe_layer_prefetch(r.h, 4)
            r.forward(synth.tokens(s, 13, step, 1, True), zb, check_y=step in (0, 5, 9))
        st = moe.moe_store_get_stats(r.store)
        assert st["reads"] > 0 and st["read_errors"] == 0
    finally:
        r.close()


def test_readahead_picks_routed_experts_outside_slots_and_tier(ctx, tmp_path):
    """One 8-token step on the tiny shapes routes to 11 experts: the 4 lowest
    take the HBM slots, the rest bypass, and the 2-entry tier ends holding the
    last two fetched. Readahead then takes the routed experts in neither, by
    routing count (all 1 here) and then id, one per entry it may use, and
    never evicts an expert read ahead and not yet used."""
    s = synth.SHAPES_TINY
    r = StreamedRig(ctx, s, 2, 4, str(tmp_path / "ra.experts"), host_slots=2, flags=0)
    try:
        assert moe.moe_layer_prefetch(r.h, 3) == 0  # no routing history yet
        xb = synth.tokens(s, 2, 0, 8, False)
        gids, _ = r.forward(xb)
        torch.cuda.synchronize()
        routed = sorted(set(gids.reshape(-1).tolist()))
        slots = set(moe.moe_cache_dump(r.h, 4)[0].tolist())
        tier = set(moe.moe_store_tier(r.store, 2)[0].tolist())
        assert slots == set(routed[:4]) and tier == set(routed[-2:])
        cands = [e for e in routed if e not in slots and e not in tier]
        assert len(cands) >= 2
        assert moe.moe_layer_prefetch(r.h, 1) == 1
        moe.moe_store_wait_idle(r.store)
        assert cands[0] in moe.moe_store_tier(r.store, 2)[0]
        assert moe.moe_layer_prefetch(r.h, 5) == 1  # only the other entry may be taken
        moe.moe_store_wait_idle(r.store)
        assert sorted(moe.moe_store_tier(r.store, 2)[0].tolist()) == cands[:2]
        assert moe.moe_layer_prefetch(r.h, 5) == 0
        st = moe.moe_store_get_stats(r.store)
        assert st["prefetch_reads"] == 2 and st["prefetch_used"] == 0
        # the next step uses what was read ahead (the same tokens route the same way)
        r.forward(xb)
        st = moe.moe_store_get_stats(r.store)
        assert st["prefetch_used"] >= 1 and st["read_errors"] == 0
    finally:
        r.close()


def test_streamed_prompt_layer_major(ctx, tmp_path):
    # one call, every distinct expert fetched once through a 4-entry tier
    s = synth.SHAPES_TINY
    r = StreamedRig(ctx, s, 2, 4, str(tmp_path / "p.experts"), host_slots=4, flags=0)
    try:
        from test_gpu_parity import _prompt_check

        _prompt_check(r, synth.tokens(s, 2, 0, 300, False), [0, 150, 299])
    finally:
        r.close()


def test_streamed_read_failure_is_reported_and_recovers(ctx, tmp_path):
    s = synth.SHAPES_TINY
    path = str(tmp_path / "fail.experts")
    r = StreamedRig(ctx, s, 1, 4, path, host_slots=2, flags=0)
    stride = moe.moe_store_expert_stride(s)
    try:
        xb = synth.tokens(s, 1, 0, 64, False)  # 64 tokens route to nearly every expert
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        os.truncate(path, 4096 + 1 * stride)  # only expert 0 is still readable
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_forward(r.h, x)
        torch.cuda.synchronize()
        assert ei.value.status == moe.MOE_ECOPY
        se, _ = moe.moe_cache_dump(r.h, 4)
        # the slots whose reads failed are empty; only expert 0 may remain
        assert set(se.tolist()) <= {-1, 0}
        moe.moe_store_write(path, s, r.w)  # same file again (same inode)
        # the cache now differs from a fresh oracle trace: compare y and ids only
        ids = torch.empty((64, s.top_k), dtype=torch.int32, device="cuda")
        y = moe.moe_forward(r.h, x, ids_out=ids)
        torch.cuda.synchronize()
        oids, ogates = oracle.topk_gates(oracle.router_logits(xb, r.w.router, s.n_experts, None), s.top_k)
        assert (ids.cpu().numpy() == oids).all()
        yg = y.cpu().numpy()
        for t in (0, 31, 63):
            ref = r.ref.combine(xb[t:t + 1], oids[t:t + 1], ogates[t:t + 1])[0]
            assert np.abs(yg[t] - ref).max() <= 2e-3 * np.abs(ref).max()
    finally:
        r.close()


def test_store_serves_one_layer_and_stays_open_while_used(ctx, tmp_path):
    s = synth.SHAPES_TINY
    r = StreamedRig(ctx, s, 0, 4, str(tmp_path / "one.experts"), host_slots=2, flags=0)
    try:
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_layer_create_streamed(ctx, s, 4, r.store)
        assert ei.value.status == moe.MOE_EINVAL
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_store_close(r.store)
        assert ei.value.status == moe.MOE_ESTATE
        plain = moe.moe_layer_create(ctx, s, 4)
        try:
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_layer_prefetch(plain, 2)
            assert ei.value.status == moe.MOE_ESTATE
        finally:
            moe.moe_layer_destroy(plain)
    finally:
        r.close()
