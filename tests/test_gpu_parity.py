"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Bars (fixed before any kernel ran):
  * expert ids (and so the gates' order) and the cache hit/miss trace: bit-exact;
  * gates: |g_gpu - g_oracle| <= 1e-6 (fp32 softmax of the same fp32 logits);
  * layer outputs: max |y_gpu - y_oracle| <= 2e-3 * max |y_oracle| per call.
The oracle runs the plain definition (double accumulation); the library runs
fp32 fused dequant GEMVs, so only rounding separates them.
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
GATE_TOL = 1e-6


@pytest.fixture(scope="module")
def ctx():
    moe.load()
    c = moe.moe_ctx_create(0)
    yield c
    moe.moe_ctx_destroy(c)


class Rig:
    """One library layer and the oracle's view of the same weights."""

    def __init__(self, ctx, shapes, layer, slots, policy=moe.LFU, seed=0, weights=None):
        self.s = shapes
        self.w = weights if weights is not None else synth.layer_weights(shapes, layer, seed)
        self.ref = oracle.Layer(self.w, shapes)
        self.cache = oracle.Cache(shapes.n_experts, slots, policy)
        self.slots = slots
        self.h = moe.moe_layer_create(ctx, shapes, slots, policy)
        moe.moe_layer_set_weights(self.h, self.w)
        self.layer = layer

    def close(self):
        moe.moe_layer_destroy(self.h)

    def forward(self, x_bits, zbias=None, check_y=True, y_tokens=None):
        """Run the library, check ids/gates/trace exactly and y within tolerance."""
        T = x_bits.shape[0]
        k = self.s.top_k
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
        zb = None if zbias is None else torch.from_numpy(zbias).cuda()
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
        y = moe.moe_forward(self.h, x, zb, ids_out=ids, gates_out=gates)
        torch.cuda.synchronize()
        lg = oracle.router_logits(x_bits, self.w.router, self.s.n_experts, zbias)
        oids, ogates = oracle.topk_gates(lg, k)
        gids = ids.cpu().numpy()
        assert (gids == oids).all(), "expert ids differ from the oracle"
        assert np.abs(gates.cpu().numpy() - ogates).max() <= GATE_TOL
        # the cache trace: the library's table after the call equals the oracle's
        chunk = T if T <= 64 else 128
        for t0 in range(0, T, chunk):
            self.cache.step(oids[t0:t0 + chunk])
        se, cnt = moe.moe_cache_dump(self.h, self.slots)
        ose, ocnt = self.cache.dump()
        assert (se == ose).all() and (cnt == ocnt).all(), "cache table differs from the oracle trace"
        if check_y:
            toks = range(T) if y_tokens is None else y_tokens
            yg = y.cpu().numpy()
            for t in toks:
                ref = self.ref.combine(x_bits[t:t + 1], oids[t:t + 1], ogates[t:t + 1])[0]
                err = np.abs(yg[t] - ref).max()
                assert err <= Y_TOL * np.abs(ref).max(), (t, err, np.abs(ref).max())
        return gids, y


def test_tiny_layer_full_parity(ctx):
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 0, 4)
    try:
        for step in range(6):
            r.forward(synth.tokens(s, 0, step, 4, False))
        st = moe.moe_layer_stats(r.h)
        assert st["steps"] == 6 and st["hits"] + st["misses"] > 0
    finally:
        r.close()


def test_tiny_layer_matches_oracle_layer_output(ctx):
    # the oracle's own fused layer (not only its per-expert pieces)
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 2, 4)
    try:
        xb = synth.tokens(s, 2, 0, 4, False)
        zb = synth.zipf_bias(s, 2, 0.8)
        _, y = r.forward(xb, zb, check_y=False)
        _, _, _, yo = r.ref.forward(xb, zb)
        assert np.abs(y.cpu().numpy() - yo).max() <= Y_TOL * np.abs(yo).max()
    finally:
        r.close()


@pytest.mark.parametrize("T", [1, 3, 16, 64, 65, 128, 200])
def test_tiny_ragged_token_counts(ctx, T):
    # decode (T <= 64) and prefill (chunks of 128 plus a ragged tail)
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 1, 4)
    try:
        r.forward(synth.tokens(s, 1, T, T, False), y_tokens=range(0, T, max(1, T // 7)))
    finally:
        r.close()


@pytest.mark.parametrize("slots,k", [(1, 2), (16, 2), (4, 1), (4, 16)])
def test_tiny_degenerate_caches_and_top_k(ctx, slots, k):
    # one slot (almost everything bypasses), all experts resident, k = 1, k = E
    s = synth.Shapes(512, 16, k, 256, 512, synth.GELU_TANH)
    r = Rig(ctx, s, 0, slots)
    try:
        for step in range(3):
            r.forward(synth.tokens(s, 0, step, 5, False))
    finally:
        r.close()


def test_decode_2816_two_layers(ctx):
    """decode_2816: layer 0 for all 64 decode steps of the workload, with ids,
    gates, the cache table and y checked at every step; and layer 17 for 8
    steps."""
    s = synth.SHAPES_2816
    wl = synth.WORKLOADS["decode_2816"]
    for layer, steps in ((0, wl.steps), (17, 8)):
        r = Rig(ctx, s, layer, wl.cache_slots)
        zb = synth.zipf_bias(s, layer, wl.zipf_s)
        try:
            for step in range(steps):
                x = synth.tokens(s, layer, step, 1, True)
                r.forward(x, zb, check_y=True)
            st = moe.moe_layer_stats(r.h)
            assert st["steps"] == steps and st["hits"] > 0 and st["misses"] > 0
        finally:
            r.close()


@pytest.mark.parametrize("policy", [moe.LFU, moe.LRU])
@pytest.mark.parametrize("T", [1, 8])
def test_decode_2048_silu(ctx, T, policy):
    """decode_2048 (SiLU, 64 slots) at batches 1 and 8 under both policies:
    two layers for 64 steps each, long enough for the 64-slot cache to fill
    and evict. Ids, gates and the cache table are checked at every step, y
    on the first and last token of steps 0, 31 and 63."""
    s = synth.SHAPES_2048
    wl = synth.WORKLOADS["decode_2048"]
    for layer in (3, 22):
        r = Rig(ctx, s, layer, wl.cache_slots, policy)
        zb = synth.zipf_bias(s, layer, wl.zipf_s)
        try:
            for step in range(64):
                x = synth.tokens(s, layer, step, T, True)
                r.forward(x, zb, check_y=step in (0, 31, 63), y_tokens=[0, T - 1])
            st = moe.moe_layer_stats(r.h)
            assert st["steps"] == 64 and st["misses"] > wl.cache_slots  # the slots filled and then evicted
        finally:
            r.close()


def _tied_router(s, layer, tied):
    """The layer's weights with router rows tied[1:] made copies of row tied[0]:
    those experts get bit-identical logits for every input."""
    w = synth.layer_weights(s, layer)
    codes, scale, bias = (a.copy() for a in w.router)
    for e in tied[1:]:
        codes[e], scale[e], bias[e] = codes[tied[0]], scale[tied[0]], bias[tied[0]]
    w.router = (codes, scale, bias)
    return w


@pytest.mark.parametrize("shapes,T", [(synth.SHAPES_TINY, 1), (synth.SHAPES_TINY, 37),
                                      (synth.SHAPES_2816, 1), (synth.SHAPES_2816, 37)])
def test_tied_logits_pick_the_lowest_expert_id(ctx, shapes, T):
    """Equal logits go to the lower expert id first. Three router rows are made
    identical; with a large equal bias on them they outrank every other expert,
    so for top-2 the ids must be exactly [a, b] and for top-8 the first three
    [a, b, c] with equal gates. Without the bias the tied experts compete with
    the rest and the ids must still equal the oracle's stable order."""
    s = shapes
    tied = [3, 9, 14] if s.n_experts == 16 else [3, 9, 20]
    w = _tied_router(s, 7, tied)
    r = Rig(ctx, s, 7, 4 if s.n_experts == 16 else 16, weights=w)
    try:
        xb = synth.tokens(s, 7, 0, T, s.n_experts != 16)
        lg = oracle.router_logits(xb, w.router, s.n_experts, None)
        assert (lg[:, tied[1:]] == lg[:, tied[:1]]).all()  # the ties are exact
        zb = np.zeros(s.n_experts, np.float32)
        zb[tied] = 40.0
        ids, _ = r.forward(xb, zb, check_y=False)
        n = min(s.top_k, len(tied))
        assert (ids[:, :n] == np.array(tied[:n])).all(), ids[:, :n]
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        rid, rg = moe.moe_route(r.h, x, s.top_k, torch.from_numpy(zb).cuda())
        torch.cuda.synchronize()
        rg = rg.cpu().numpy()
        assert (rid.cpu().numpy()[:, :n] == np.array(tied[:n])).all()
        assert (rg[:, 1:n] == rg[:, :1]).all()  # equal logits, equal gates
        # without the bias, and with a small one that puts the tie mid-rank:
        # ties wherever the shared logit makes the top-k
        zmid = np.zeros(s.n_experts, np.float32)
        zmid[tied] = 1.5
        for step in range(1, 7):
            xb = synth.tokens(s, 7, step, T, s.n_experts != 16)
            ids, _ = r.forward(xb, zmid if step % 2 else None, check_y=False)
            both = np.isin(ids, tied).sum(axis=1) >= 2
            for row in ids[both]:
                pos = [int(np.where(row == e)[0][0]) for e in tied if e in row]
                assert pos == sorted(pos)
    finally:
        r.close()


def test_prefill_chunk_2816(ctx):
    s = synth.SHAPES_2816
    r = Rig(ctx, s, 5, 16)
    try:
        x = synth.tokens(s, 5, 0, 128, True)
        r.forward(x, None, y_tokens=[0, 61, 127])
        st = moe.moe_layer_stats(r.h)
        assert st["bypass"] > 0  # a 128-token chunk touches far more than 16 experts
    finally:
        r.close()


@pytest.mark.parametrize("layer", [0, 1, 29])
def test_prefill_prompt_as_chunks_2816(ctx, layer):
    """prefill_2816: the 1024-token prompt as 8 chunks of 128 through a fresh
    16-slot cache, uniform routing; ids, gates and the cache table after every
    chunk, y on tokens of the first and the last chunk."""
    s = synth.SHAPES_2816
    wl = synth.WORKLOADS["prefill_2816"]
    r = Rig(ctx, s, layer, wl.cache_slots)
    try:
        x = synth.tokens(s, layer, 0, wl.tokens * wl.steps, True)
        r.forward(x, None, y_tokens=[0, 127, 896, 1023])
        st = moe.moe_layer_stats(r.h)
        assert st["steps"] == wl.steps and st["bypass"] > 0
    finally:
        r.close()


def test_prefill_prompt_repeated_all_resident(ctx):
    """A 1024-token prompt (8 chunks of 128) through a layer with a slot per
    expert, six times: the first pass copies every expert in, the rest run on
    resident weights. The down GEMM's jobs have 11 K-blocks, so the MMA issuers'
    A stages change owner between jobs; every pass must finish without an
    expired wait and give the same bits (the arithmetic order is fixed)."""
    s = synth.SHAPES_2816
    r = Rig(ctx, s, 6, s.n_experts)
    try:
        xb = synth.tokens(s, 6, 0, 1024, True)
        first, y0 = r.forward(xb, None, y_tokens=[0, 517, 1023])
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        for rep in range(5):
            y = moe.moe_forward(r.h, x)
            torch.cuda.synchronize()
            assert torch.equal(y, y0), f"pass {rep + 1} differs from the first"
        st = moe.moe_layer_stats(r.h)
        assert st["misses"] == len(np.unique(first))
    finally:
        r.close()


def test_prefill_split_k_small_launch(ctx):
    """A layer of d = 2816 with one 64-wide routed expert and the 2816-wide
    shared expert: its prefill launches have too few 128-row tiles to fill the
    GPU, so each tile's K range is split over several CTAs and the parts are
    added by a second kernel. Outputs match the oracle, and a repeat gives the
    same bits."""
    s0 = synth.SHAPES_2816
    s = synth.Shapes(s0.d_model, 1, 1, 64, s0.d_ff_shared, s0.act)
    r = Rig(ctx, s, 2, 1)
    try:
        xb = synth.tokens(s, 2, 0, 128, True)
        _, y0 = r.forward(xb, None, y_tokens=[0, 1, 77, 127])
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        y = moe.moe_forward(r.h, x)
        torch.cuda.synchronize()
        assert torch.equal(y, y0)
    finally:
        r.close()


def test_prefill_chunk_skewed_rows_2816(ctx):
    """A 128-token chunk of d = 2816 whose routing is skewed by the zbias:
    expert 0 is in every token's top-k (one item of 128 rows), expert 1 in
    about half of them, the rest spread thin. The launch still counts as a
    chunk (a few rows per routed expert on average), so the big items go
    through the chunk layout's 64- and 128-row token boxes."""
    s = synth.SHAPES_2816
    r = Rig(ctx, s, 7, 16)
    try:
        xb = synth.tokens(s, 7, 0, 128, True)
        lg = oracle.router_logits(xb, r.w.router, s.n_experts, None)
        k = s.top_k
        kth = np.sort(lg, axis=1)[:, -k]  # each token's k-th largest logit
        zb = np.zeros(s.n_experts, dtype=np.float32)
        zb[0] = float(np.max(kth - lg[:, 0])) + 1.0
        zb[1] = float(np.median(kth - lg[:, 1]))
        ids, _ = r.forward(xb, zb, y_tokens=[0, 1, 63, 64, 127])
        counts = np.bincount(ids.ravel(), minlength=s.n_experts)
        assert counts[0] == 128 and 32 < counts[1] < 128, counts[:2]
        assert ids.size / np.count_nonzero(counts) <= 24
    finally:
        r.close()


def _prompt_check(r, xb, y_tokens):
    """One moe_forward_prompt call checked against the oracle: ids bit-exact,
    gates within 1e-6, the cache table after ONE step over all the call's ids,
    and y on the sampled tokens."""
    T, k = xb.shape[0], r.s.top_k
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    y = moe.moe_forward_prompt(r.h, x, None, ids_out=ids, gates_out=gates)
    torch.cuda.synchronize()
    lg = oracle.router_logits(xb, r.w.router, r.s.n_experts, None)
    oids, ogates = oracle.topk_gates(lg, k)
    assert (ids.cpu().numpy() == oids).all()
    assert np.abs(gates.cpu().numpy() - ogates).max() <= GATE_TOL
    r.cache.step(oids)
    se, cnt = moe.moe_cache_dump(r.h, r.slots)
    ose, ocnt = r.cache.dump()
    assert (se == ose).all() and (cnt == ocnt).all(), "cache table differs from one oracle step"
    yg = y.cpu().numpy()
    for t in y_tokens:
        ref = r.ref.combine(xb[t:t + 1], oids[t:t + 1], ogates[t:t + 1])[0]
        err = np.abs(yg[t] - ref).max()
        assert err <= Y_TOL * np.abs(ref).max(), (t, err, np.abs(ref).max())
    return y


@pytest.mark.parametrize("T", [65, 300, 4096])
def test_prompt_layer_major_tiny(ctx, T):
    """A prompt longer than a chunk in one layer-major call: several shared
    token blocks (the last ragged), one cache step, twice in a row (the second
    call on a warm cache gives the same bits). At the largest prompt (4096
    tokens, ~512 rows per expert) every routed expert is split into pieces of
    128 rows."""
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 0, 4)
    try:
        xb = synth.tokens(s, 0, 0, T, False)
        y0 = _prompt_check(r, xb, [0, T // 2, T - 1])
        y1 = _prompt_check(r, xb, [0, T - 1])
        assert torch.equal(y0, y1)
    finally:
        r.close()


def test_prompt_layer_major_2816(ctx):
    """A 1024-token prompt of d = 2816 in one call: ~32 token rows per routed
    expert, the shared expert in 8 token blocks, most experts bypassing the
    16-slot cache through the staging arena."""
    s = synth.SHAPES_2816
    r = Rig(ctx, s, 4, 16)
    try:
        xb = synth.tokens(s, 4, 0, 1024, True)
        _prompt_check(r, xb, [0, 129, 1023])
        st = moe.moe_layer_stats(r.h)
        assert st["bypass"] > 0 and st["steps"] == 1
    finally:
        r.close()


def test_route_call_matches_oracle(ctx):
    s = synth.SHAPES_2816
    r = Rig(ctx, s, 9, 16)
    try:
        xb = synth.tokens(s, 9, 0, 37, True)
        zb = synth.zipf_bias(s, 9, 1.1)
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        ids, gates = moe.moe_route(r.h, x, s.top_k, torch.from_numpy(zb).cuda())
        torch.cuda.synchronize()
        oids, og = oracle.topk_gates(oracle.router_logits(xb, r.w.router, s.n_experts, zb), s.top_k)
        assert (ids.cpu().numpy() == oids).all()
        assert np.abs(gates.cpu().numpy() - og).max() <= GATE_TOL
    finally:
        r.close()


def test_cache_step_call_and_forward_agree(ctx):
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 0, 4)
    try:
        ids = np.array([[3, 5], [5, 9]], np.int32)
        out = moe.moe_cache_step(r.h, ids)
        o = r.cache.step(ids)
        assert (out["slot_of"] == o["slot_of"]).all()
        assert (out["miss_experts"] == o["miss_experts"]).all() and (out["miss_slots"] == o["miss_slots"]).all()
        # the copies it issued must leave the slots usable by a forward
        for step in range(3):
            r.forward(synth.tokens(s, 0, 10 + step, 4, False))
    finally:
        r.close()


def test_injected_copy_failure_is_reported_and_recovers(ctx):
    # A host-made fault: the next miss copy reports failure instead of being issued.
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 0, 4)
    try:
        x0 = synth.tokens(s, 0, 0, 4, False)
        moe.moe_ctx_inject_copy_failure(ctx, 0)
        x = torch.from_numpy(x0.view(np.int16)).view(torch.bfloat16).cuda()
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_forward(r.h, x)
        assert ei.value.status == moe.MOE_ECOPY
        torch.cuda.synchronize()
        se, _ = moe.moe_cache_dump(r.h, 4)
        assert (se == -1).all()  # every slot whose copy was not issued is left empty
        # the oracle never saw the failed call; reset the library's view to match
        moe.moe_layer_set_weights(r.h, r.w)
        for step in range(3):
            r.forward(synth.tokens(s, 0, 20 + step, 4, False))
    finally:
        r.close()


def test_cache_reset_empties_the_table(ctx):
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 0, 4)
    try:
        for step in range(3):
            r.forward(synth.tokens(s, 0, 30 + step, 4, False))
        moe.moe_cache_reset(r.h)
        se, cnt = moe.moe_cache_dump(r.h, 4)
        assert (se == -1).all() and (cnt == 0).all()
        # from here the library must follow a fresh oracle cache
        r.cache = oracle.Cache(s.n_experts, 4, moe.LFU)
        for step in range(3):
            r.forward(synth.tokens(s, 0, 40 + step, 4, False))
    finally:
        r.close()


# ---- one-token calls: the hits are looked up on the device in a copy of the
# slot table, which every other path that changes the cache must keep current


@pytest.mark.parametrize("slots,k", [(1, 2), (16, 2), (4, 1), (4, 16), (4, 24)])
def test_one_token_degenerate_caches_and_top_k(ctx, slots, k):
    # one slot (the rest bypasses), all resident, k = 1, k = 16, and k = 24 (more
    # pairs than the device-routed list holds: the host-built path)
    s = synth.Shapes(512, 32, k, 256, 512, synth.GELU_TANH)
    r = Rig(ctx, s, 0, slots)
    try:
        for step in range(6):
            r.forward(synth.tokens(s, 0, step, 1, False))
    finally:
        r.close()


def test_one_token_after_cache_step_call(ctx):
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 0, 4)
    try:
        ids = np.array([[3, 5], [5, 9]], np.int32)
        moe.moe_cache_step(r.h, ids)
        r.cache.step(ids)
        for step in range(4):
            r.forward(synth.tokens(s, 0, 30 + step, 1, False))
    finally:
        r.close()


def test_one_token_after_injected_copy_failure(ctx):
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 0, 4)
    try:
        for step in range(2):
            r.forward(synth.tokens(s, 0, 40 + step, 1, False))
        moe.moe_ctx_inject_copy_failure(ctx, 0)
        x = torch.from_numpy(synth.tokens(s, 0, 42, 1, False).view(np.int16)).view(torch.bfloat16).cuda()
        try:
            moe.moe_forward(r.h, x)
            failed = False
        except moe.MoeError as e:
            assert e.status == moe.MOE_ECOPY
            failed = True
        torch.cuda.synchronize()
        if failed:
            # the oracle never saw the failed call: restart both from an empty cache
            moe.moe_layer_set_weights(r.h, r.w)
            r.cache = oracle.Cache(s.n_experts, 4, moe.LFU)
        else:
            moe.moe_ctx_inject_copy_failure(ctx, -1)  # the call had no miss to fail
            r.cache.step(oracle.topk_gates(oracle.router_logits(synth.tokens(s, 0, 42, 1, False), r.w.router,
                                                                s.n_experts, None), s.top_k)[0])
        for step in range(4):
            r.forward(synth.tokens(s, 0, 43 + step, 1, False))
    finally:
        r.close()


def test_one_token_mixed_with_batches_and_prefill(ctx):
    # the host-built paths (a 4-token call, a 130-token prefill) change the cache
    # too; one-token calls after them must see the same table as the host
    s = synth.SHAPES_TINY
    r = Rig(ctx, s, 3, 4)
    try:
        for step, T in enumerate([1, 4, 1, 130, 1, 1, 4, 1]):
            r.forward(synth.tokens(s, 3, 50 + step, T, False), y_tokens=[0, T - 1])
        moe.moe_cache_reset(r.h)
        r.cache = oracle.Cache(s.n_experts, 4, moe.LFU)
        for step in range(3):
            r.forward(synth.tokens(s, 3, 60 + step, 1, False))
    finally:
        r.close()


def test_timeline_trace_file(tmp_path, monkeypatch):
    path = tmp_path / "trace.txt"
    monkeypatch.setenv("MOE_TRACE_FILE", str(path))
    c = moe.moe_ctx_create(0)
    s = synth.SHAPES_TINY
    try:
        r = Rig(c, s, 0, 4)
        try:
            for step in range(3):
                r.forward(synth.tokens(s, 0, 70 + step, 1, False))
        finally:
            r.close()
    finally:
        moe.moe_ctx_destroy(c)
    lines = path.read_text().splitlines()
    assert lines[0].startswith("cal ")
    launches = [l.split() for l in lines if l.startswith("launch ")]
    assert len(launches) >= 6  # a router and a resident launch per call
    for l in launches:
        start, end = int(l[5]), int(l[6])
        assert 0 < start <= end  # every launch ran and recorded its span
    marks = {l.split()[1] for l in lines if l.startswith("host ")}
    assert {"call", "ids", "copies", "end"} <= marks


def test_hbm_prefetch_leaves_every_result_unchanged(ctx):
    """decode_2816 layer 2 with the spare-buffer prefetch on: misses of the
    prefetched expert are copied from HBM instead of host memory, and the
    ids, gates, cache trace and y stay those of the oracle at every step."""
    s = synth.SHAPES_2816
    wl = synth.WORKLOADS["decode_2816"]
    r = Rig(ctx, s, 2, wl.cache_slots)
    zb = synth.zipf_bias(s, 2, wl.zipf_s)
    try:
        moe.moe_layer_set_prefetch(r.h, True)
        for step in range(40):
            r.forward(synth.tokens(s, 2, step, 1, True), zb, check_y=step % 4 == 0)
        st = moe.moe_layer_prefetch_stats(r.h)
        assert st["issued"] > 0 and st["used"] > 0, st
    finally:
        r.close()
