"""Pins of the CPU oracle to things other than itself.

Each test fixes the oracle against a closed form, a textbook or library routine
applied to a special case, an invariant of the definition, brute force on a
tiny input, or a hand-replayed trace under tests/golden/. Each is chosen so that
a plausible slip in the oracle (a dropped term, a wrong sign or index, a swapped
nibble, a transposed operand, a wrong tie-break) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import synth
from tests.conftest import GOLDEN

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _const_matrix(n, k, code, scale_bits, bias_bits):
    codes = np.full((n, k // 2), (code & 15) | ((code & 15) << 4), np.uint8)
    s = np.full((n, k // 64), scale_bits, np.uint16)
    b = np.full((n, k // 64), bias_bits, np.uint16)
    return codes, s, b


class _W:
    """Minimal stand-in with the attributes oracle.Layer reads."""

    def __init__(self, router, shared, experts):
        self.router = router
        self.shared = shared
        stack = lambda i, j: np.stack([e[i][j] for e in experts])
        self.gate_codes, self.gate_scale, self.gate_bias = stack(0, 0), stack(0, 1), stack(0, 2)
        self.up_codes, self.up_scale, self.up_bias = stack(1, 0), stack(1, 1), stack(1, 2)
        self.down_codes, self.down_scale, self.down_bias = stack(2, 0), stack(2, 1), stack(2, 2)


# ---------------------------------------------------------------------------
# generator (input side): published definitions


def test_splitmix64_known_answers():
    # SplitMix64 seeded with state 0 emits mix(gamma), mix(2 gamma), ...; the
    # published first outputs for seed 0 are these three words.
    w = synth.words(0, 0, 3)
    assert [int(v) for v in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_f16_and_bf16_rounding_match_libraries():
    import torch

    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-3e-4, 3e-4, 500), rng.uniform(-70000, 70000, 200),
                           rng.uniform(-1e-7, 1e-7, 200), [0.0, 6.103515625e-05, 2.0 ** -24, 2.0 ** -25]])
    for v in vals:
        assert synth.f64_to_f16_bits(float(v)) == int(np.float16(v).view(np.uint16)), v
    f = rng.standard_normal(2000).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([synth.f32_to_bf16_bits(float(v)) for v in f], np.uint16)
    assert (mine == ref).all()


# ---------------------------------------------------------------------------
# dequantisation


def test_dequant_known_codes_and_nibble_order():
    s_bits = int(np.float16(0.01).view(np.uint16))
    s = oracle.f16(s_bits)
    assert s == 0.01000213623046875  # 1311 * 2^-17, the binary16 nearest 0.01
    b_bits = int(np.float16(-8 * s).view(np.uint16))
    assert oracle.f16(b_bits) == -8 * s
    # one row, K = 64: byte 0 = 0xF0 -> element 0 = 0 (low nibble), element 1 = 15 (high nibble)
    codes = np.zeros((1, 32), np.uint8)
    codes[0, 0] = 0xF0
    codes[0, 1] = 0x08  # element 2 = 8, element 3 = 0
    scale = np.full((1, 1), s_bits, np.uint16)
    bias = np.full((1, 1), b_bits, np.uint16)
    assert oracle.code_u4(codes, 64, 0, 0) == 0 and oracle.code_u4(codes, 64, 0, 1) == 15
    assert oracle.w4(codes, scale, bias, 64, 0, 1) == 7 * s  # q = 15
    assert oracle.w4(codes, scale, bias, 64, 0, 0) == -8 * s  # q = 0
    assert oracle.w4(codes, scale, bias, 64, 0, 2) == 0.0  # q = 8
    # group index: a second group with its own scale
    codes2 = np.zeros((2, 64), np.uint8)
    codes2[1, 32] = 0x01  # row 1, element 64 (group 1) = 1
    sc = np.array([[0x3C00, 0x3C00], [0x3C00, 0x4000]], np.uint16)  # 1.0, 1.0 / 1.0, 2.0
    bi = np.zeros((2, 2), np.uint16)
    assert oracle.w4(codes2, sc, bi, 128, 1, 64) == 2.0
    assert oracle.w4(codes2, sc, bi, 128, 0, 64) == 0.0


def test_activation_against_library_forms():
    z = np.linspace(-8, 8, 401)
    gel = np.array([oracle.act(v, oracle.GELU_TANH) for v in z])
    exact = 0.5 * z * (1 + scipy.special.erf(z / np.sqrt(2)))  # erf form of GELU
    assert np.abs(gel - exact).max() < 1e-3  # the tanh form is within ~5e-4 of it
    assert np.abs(gel - exact).max() > 1e-5  # and is not the erf form
    silu = np.array([oracle.act(v, oracle.SILU) for v in z])
    assert np.allclose(silu, z * scipy.special.expit(z), rtol=1e-14, atol=1e-15)
    assert oracle.act(0.0, oracle.GELU_TANH) == 0.0


# ---------------------------------------------------------------------------
# closed-form worked example


def _two_expert_layer(k):
    one_bf16 = 0x3F80
    s_bits, b_bits = 0x2C00, 0xB800  # 2^-4, -0.5
    e0 = tuple(_const_matrix(n, kk, 9, s_bits, b_bits) for n, kk in ((64, 64), (64, 64), (64, 64)))
    e1 = tuple(_const_matrix(n, kk, 10, s_bits, b_bits) for n, kk in ((64, 64), (64, 64), (64, 64)))
    shared = tuple(_const_matrix(64, 64, 9, s_bits, b_bits) for _ in range(3))
    rc = np.array([[130] * 64, [129] * 64], np.uint8)
    rs = np.full((2, 1), 0x2400, np.uint16)
    rb = np.full((2, 1), 0xC000, np.uint16)
    w = _W((rc, rs, rb), shared, [e0, e1])
    shapes = synth.Shapes(64, 2, k, 64, 64, synth.GELU_TANH)
    x = np.full((1, 64), one_bf16, np.uint16)
    return oracle.Layer(w, shapes), x


def test_two_expert_closed_form():
    with open(os.path.join(GOLDEN, "two_expert_example.json")) as f:
        g = json.load(f)
    for k, key in ((2, "y_k2"), (1, "y_k1")):
        L, x = _two_expert_layer(k)
        logits, ids, gates, y = L.forward(x)
        assert logits[0].tolist() == g["logits"]
        assert ids[0].tolist() == [0, 1][:k]
        if k == 2:
            assert np.allclose(gates[0], g["gates_k2"], rtol=1e-14)
        assert np.allclose(y[0], g[key], rtol=1e-13), (y[0, :3], g[key])
    # the closed form itself, independent of the stored numbers
    gel = lambda z: 0.5 * z * (1 + math.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))
    h0, h1 = 4 * gel(4.0), 8 * gel(8.0)
    g0 = math.e ** 2 / (math.e ** 2 + math.e)
    assert math.isclose(g["y_k2"], 4 * h0 + g0 * 4 * h0 + (1 - g0) * 8 * h1, rel_tol=1e-14)


# ---------------------------------------------------------------------------
# router


def test_router_one_hot_input_reads_one_column():
    s = synth.SHAPES_TINY
    r = synth.router_weights(s, 0)
    for j in (0, 1, 17, 64, 511):
        x = np.zeros((1, s.d_model), np.uint16)
        x[0, j] = 0x3F80  # 1.0
        lg = oracle.router_logits(x, r, s.n_experts)
        for e in range(s.n_experts):
            w = oracle.f16(r[1][e, j // 64]) * float(r[0][e, j]) + oracle.f16(r[2][e, j // 64])
            assert lg[0, e] == np.float32(w)


def test_router_fp32_order_within_rounding_bound():
    for s in (synth.SHAPES_TINY, synth.SHAPES_2048):
        r = synth.router_weights(s, 3)
        x = synth.tokens(s, 3, 0, 3, True)
        zb = synth.zipf_bias(s, 3, 0.9)
        l32 = oracle.router_logits(x, r, s.n_experts, zb).astype(np.float64)
        l64 = oracle.router_logits_f64(x, r, s.n_experts, zb)
        # bound: (d/32 fmas + 5 tree adds + bias add) units of roundoff times sum |w x|
        xf = synth.bf16_to_f32(x).astype(np.float64)
        wf = synth.f16(r[1]).astype(np.float64).repeat(64, 1) * r[0] + synth.f16(r[2]).astype(np.float64).repeat(64, 1)
        mag = np.abs(xf) @ np.abs(wf).T + np.abs(zb)[None, :]
        n_ops = s.d_model // 32 + 6
        assert (np.abs(l32 - l64) <= n_ops * 2.0 ** -24 * mag * 1.01).all()
        assert np.abs(l32 - l64).max() > 0  # fp32 is genuinely fp32
        # against numpy's matmul on the dequantised weights (library routine)
        assert np.allclose(l64, xf @ wf.T + zb[None, :], rtol=1e-12, atol=1e-12)


def test_topk_matches_stable_argsort_and_gate_identities():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((50, 32)).astype(np.float32)
    logits[0, [3, 9, 20]] = 5.0  # exact ties: lower index ranks first
    logits[1, :] = 1.0
    ids, gates = oracle.topk_gates(logits, 6)
    for t in range(logits.shape[0]):
        ref = np.argsort(-logits[t].astype(np.float64), kind="stable")[:6]
        assert ids[t].tolist() == ref.tolist()
    assert ids[0, :3].tolist() == [3, 9, 20]
    assert ids[1].tolist() == [0, 1, 2, 3, 4, 5]
    assert np.allclose(gates.sum(1), 1.0, atol=1e-14)
    assert (np.diff(gates, axis=1) <= 0).all()
    # k = E: the renormalised gates are the full softmax
    ids_all, g_all = oracle.topk_gates(logits, 32)
    sm = scipy.special.softmax(logits.astype(np.float64), axis=1)
    for t in range(logits.shape[0]):
        assert np.allclose(g_all[t], sm[t, ids_all[t]], rtol=1e-13)
    # k < E: the renormalised softmax equals the softmax over the chosen logits alone
    for t in range(5):
        sel = logits[t, ids[t]].astype(np.float64)
        assert np.allclose(gates[t], scipy.special.softmax(sel), rtol=1e-13)
    # shifting every logit by a constant changes neither ids nor gates
    ids2, gates2 = oracle.topk_gates(logits + np.float32(0.5), 6)
    assert (ids2[2:] == ids[2:]).all()
    assert np.allclose(gates2[2:], gates[2:], atol=1e-6)


def test_zero_router_weights_route_by_bias():
    s = synth.SHAPES_2816
    r = (np.zeros((s.n_experts, s.d_model), np.uint8), np.zeros((s.n_experts, 44), np.uint16),
         np.zeros((s.n_experts, 44), np.uint16))
    zb = synth.zipf_bias(s, 5, 1.1)
    x = synth.tokens(s, 5, 0, 2, True)
    lg = oracle.router_logits(x, r, s.n_experts, zb)
    ids, _ = oracle.topk_gates(lg, 8)
    ref = np.argsort(-zb.astype(np.float64), kind="stable")[:8]
    assert (ids == ref[None, :]).all()


# ---------------------------------------------------------------------------
# FFN and layer


def _dequant(m):
    codes, sc, bi = m
    n, kh = codes.shape
    q = np.empty((n, kh * 2), np.float64)
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    return q * synth.f16(sc).astype(np.float64).repeat(64, 1) + synth.f16(bi).astype(np.float64).repeat(64, 1)


@pytest.mark.parametrize("act", [synth.GELU_TANH, synth.SILU])
def test_single_expert_reduces_to_textbook_gated_ffn(act):
    # E = 1, k = 1 makes the gate exactly 1; a shared expert with all codes 8
    # and bias -8 scale is exactly zero. The layer is then the textbook gated
    # FFN W_d (act(W_g x) * (W_u x)), evaluated here with numpy matmul.
    s = synth.Shapes(512, 1, 1, 256, 512, act)
    g, u, dn = synth.ffn_weights(s, 0, 0)
    zero_shared = tuple(_const_matrix(n, k, 8, 0x2400, 0xB000) for n, k in ((512, 512), (512, 512), (512, 512)))
    assert oracle.f16(0xB000) == -8 * oracle.f16(0x2400)
    w = _W(synth.router_weights(s, 0), zero_shared, [(g, u, dn)])
    L = oracle.Layer(w, s)
    x = synth.tokens(s, 0, 0, 3, True)
    _, ids, gates, y = L.forward(x)
    assert (ids == 0).all() and (gates == 1.0).all()
    xf = synth.bf16_to_f32(x).astype(np.float64)
    G, U, D = _dequant(g), _dequant(u), _dequant(dn)
    zg = xf @ G.T
    a = zg * scipy.special.expit(zg) if act == synth.SILU else 0.5 * zg * (
        1 + np.tanh(np.sqrt(2 / np.pi) * (zg + 0.044715 * zg ** 3)))
    ref = (a * (xf @ U.T)) @ D.T
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-10 * np.abs(ref).max())


def test_dense_brute_force_equals_sparse_layer():
    s = synth.SHAPES_TINY
    w = synth.layer_weights(s, 0)
    L = oracle.Layer(w, s)
    x = synth.tokens(s, 0, 0, 4, False)
    zb = synth.zipf_bias(s, 0, 0.7)
    for bias in (None, zb):
        _, _, _, y = L.forward(x, bias)
        yd = L.forward_dense(x, bias)
        assert np.allclose(y, yd, rtol=0, atol=1e-12 * np.abs(y).max())


def test_layer_invariants():
    s = synth.SHAPES_TINY
    w = synth.layer_weights(s, 1)
    L = oracle.Layer(w, s)
    x = synth.tokens(s, 1, 0, 4, False)
    _, ids, gates, y = L.forward(x)
    # tokens are independent
    for t in range(4):
        _, _, _, yt = L.forward(x[t:t + 1])
        assert (yt[0] == y[t]).all()
    # relabelling the experts (router rows and expert weights together) changes nothing
    perm = np.random.default_rng(3).permutation(s.n_experts)
    w2 = synth.layer_weights(s, 1)
    w2.router = tuple(a[perm] for a in w.router)
    for name in ("gate_codes", "gate_scale", "gate_bias", "up_codes", "up_scale", "up_bias", "down_codes",
                 "down_scale", "down_bias"):
        setattr(w2, name, getattr(w, name)[perm])
    _, ids2, gates2, y2 = oracle.Layer(w2, s).forward(x)
    assert (perm[ids2] == ids).all()
    # (the softmax normaliser is summed in expert-index order, so only rounding may differ)
    assert np.allclose(gates2, gates, rtol=1e-13) and np.allclose(y2, y, rtol=0, atol=1e-13 * np.abs(y).max())
    # doubling every down-projection scale and bias doubles y exactly
    w3 = synth.layer_weights(s, 1)
    dbl = lambda b: (synth.f16(b).astype(np.float32) * 2).astype(np.float16).view(np.uint16)
    w3.down_scale, w3.down_bias = dbl(w.down_scale), dbl(w.down_bias)
    g, u, dn = w.shared
    w3.shared = (g, u, (dn[0], dbl(dn[1]), dbl(dn[2])))
    _, _, _, y3 = oracle.Layer(w3, s).forward(x)
    assert (y3 == 2 * y).all()
    # per-token expert terms: y = shared + sum_r g_r o_r, each term checkable alone
    yc = L.combine(x, ids, gates)
    assert np.allclose(yc, y, rtol=0, atol=1e-12 * np.abs(y).max())
    # swapping gate and up changes the output (the operands are not symmetric)
    w4 = synth.layer_weights(s, 1)
    w4.gate_codes, w4.up_codes = w.up_codes, w.gate_codes
    w4.gate_scale, w4.up_scale = w.up_scale, w.gate_scale
    w4.gate_bias, w4.up_bias = w.up_bias, w.gate_bias
    _, _, _, y4 = oracle.Layer(w4, s).forward(x)
    assert np.abs(y4 - y).max() > 1e-3 * np.abs(y).max()


# ---------------------------------------------------------------------------
# cache


def test_cache_golden_traces():
    with open(os.path.join(GOLDEN, "lfu_toy_trace.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        pol = oracle.LFU if case["policy"] == "lfu" else oracle.LRU
        c = oracle.Cache(case["experts"], case["slots"], pol)
        hits = lookups = 0
        for step, exp in zip(case["steps"], case["expected"]):
            r = c.step(step)
            se, cnt = c.dump()
            assert r["hits"] == exp["hits"], (case["name"], step)
            assert r["misses"] == exp["misses"], (case["name"], step)
            assert r["miss_slots"].tolist() == exp["miss_slots"], (case["name"], step)
            assert r["bypass"] == exp.get("bypass", 0)
            assert se.tolist() == exp["slot_expert"], (case["name"], step)
            if "counts" in exp:
                assert cnt.tolist() == exp["counts"], (case["name"], step)
            hits += r["hits"]
            lookups += r["hits"] + r["misses"]
        assert hits == case["total_hits"] and lookups == case["total_lookups"], case["name"]


@pytest.mark.parametrize("policy", [oracle.LFU, oracle.LRU])
def test_cache_random_trace_properties(policy):
    rng = np.random.default_rng(11 + policy)
    E, S = 64, 12
    c = oracle.Cache(E, S, policy)
    for step in range(300):
        n = int(rng.integers(1, 20))
        ids = rng.zipf(1.3, n) % E
        r = c.step(ids)
        distinct = np.unique(ids)
        assert r["hits"] + r["misses"] == len(distinct)
        assert r["miss_experts"].tolist() == sorted(r["miss_experts"].tolist())
        se, _ = c.dump()
        resident = se[se >= 0]
        assert len(set(resident.tolist())) == len(resident)  # no expert twice
        for i, e in enumerate(ids):
            so = r["slot_of"][i]
            if so >= 0:
                assert se[so] == e
        # bypass only when the step's distinct experts exceed the slots
        assert r["bypass"] == max(0, len(distinct) - S)


def test_grouping_is_stable_sort_by_expert():
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 256, (128, 8)).astype(np.int32)
    offsets, perm = oracle.group_pairs(ids, 256)
    ref = np.argsort(ids.reshape(-1), kind="stable")
    assert (perm == ref).all()
    counts = np.bincount(ids.reshape(-1), minlength=256)
    assert (np.diff(offsets) == counts).all() and offsets[0] == 0 and offsets[-1] == ids.size
