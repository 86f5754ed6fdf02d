"""Seeded synthetic workloads for the expert-streaming MoE layer.

This module only draws inputs: weights in the canonical quantised layout, token
activations and the per-expert router bias. It holds none of the layer's
arithmetic, so both the CPU oracle (``oracle``) and the CUDA library
(``expert_streaming_ffn_gb300``) can consume it without sharing any computation.

Canonical layout (what ``moe_layer_set_weights`` and the oracle both read):
  * a matrix W[N][K] is row-major; K is grouped in runs of 64;
  * 4-bit codes: byte j of a row holds element 2j in the low nibble and 2j+1 in
    the high nibble, unsigned 0..15;
  * 8-bit router codes: one unsigned byte per element;
  * per (row, group) an IEEE binary16 scale and bias, arrays [N][K/64].

Value distributions (the workloads' stated recipe):
  * expert and shared codes ~ U{0..15}, scale ~ U(0.005, 0.02) in binary16,
    bias = -8 * scale;
  * router codes ~ U{0..255}, scale ~ U(0.005, 0.02) / sqrt(d) in binary16,
    bias = -128 * scale (keeps router logits near unit spread);
  * x ~ N(0, 1) per element, rows scaled to unit RMS where the workload says so,
    stored as bfloat16; x for each (step, layer, token) is drawn independently;
  * Zipf router bias: a seeded permutation ranks the experts, and the expert of
    rank r (1-based) gets bias -beta * s * ln(r).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None
_lock = threading.Lock()

# tensor ids of the counter streams
T_ROUTER_CODES, T_ROUTER_SCALE = 1, 2
T_GATE_CODES, T_GATE_SCALE, T_UP_CODES, T_UP_SCALE, T_DOWN_CODES, T_DOWN_SCALE = 3, 4, 5, 6, 7, 8
T_SHARED_OFFSET = 10  # shared expert streams are the routed ids + 10
T_X = 30
T_ZIPF_PERM = 31

GELU_TANH, SILU = 0, 1
LFU, LRU = 0, 1


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libsynth.so (plain C, host compiler)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    u64, u32, i32, dbl = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_double
    vp = ctypes.c_void_p
    lib.synth_key.restype = u64
    lib.synth_key.argtypes = [u64, u32, u32, u64]
    lib.synth_words.argtypes = [u64, u64, u64, vp]
    lib.synth_f64_to_f16.restype = ctypes.c_uint16
    lib.synth_f64_to_f16.argtypes = [dbl]
    lib.synth_f32_to_bf16.restype = ctypes.c_uint16
    lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.synth_codes_u4.argtypes = [u64, u64, vp]
    lib.synth_codes_u8.argtypes = [u64, u64, vp]
    lib.synth_scale_bias_f16.argtypes = [u64, u64, dbl, dbl, dbl, dbl, vp, vp]
    lib.synth_normal_bf16.argtypes = [u64, i32, i32, i32, vp, vp]
    lib.synth_permutation.argtypes = [u64, i32, vp]
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def key(seed: int, tensor: int, layer: int, sub: int) -> int:
    """Stream key of (seed, tensor id, layer, expert-or-step)."""
    return _load().synth_key(seed, tensor, layer, sub)


def words(k: int, first: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().synth_words(k, first, n, _ptr(out))
    return out


def f64_to_f16_bits(v: float) -> int:
    return int(_load().synth_f64_to_f16(float(v)))


def f32_to_bf16_bits(v: float) -> int:
    return int(_load().synth_f32_to_bf16(float(v)))


# ---------------------------------------------------------------------------
# workload shapes


@dataclass(frozen=True)
class Shapes:
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    d_ff_shared: int
    act: int  # GELU_TANH or SILU


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: Shapes
    n_layers: int
    tokens: int  # tokens per forward call (decode batch or prefill chunk)
    steps: int  # forward calls per layer
    cache_slots: int
    policy: int
    zipf_s: float | None  # None: no router bias
    zipf_beta: float = 1.0
    rms_normalise: bool = True
    seed: int = 0
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


SHAPES_TINY = Shapes(512, 16, 2, 256, 512, GELU_TANH)
SHAPES_2816 = Shapes(2816, 256, 8, 704, 2816, GELU_TANH)
SHAPES_2048 = Shapes(2048, 256, 8, 512, 512, SILU)

WORKLOADS = {
    # tiny single layer: 4 decode tokens, 4-slot LFU, x ~ N(0,1) without RMS scaling
    "tiny": Workload("tiny", SHAPES_TINY, 1, 4, 1, 4, LFU, None, rms_normalise=False),
    # decode: 30 layers, batch 1, 64 steps, 16-slot LFU, Zipf(1.1) router bias
    "decode_2816": Workload("decode_2816", SHAPES_2816, 30, 1, 64, 16, LFU, 1.1),
    # prefill: 1024-token prompt as 8 chunks of 128 tokens, no router bias
    "prefill_2816": Workload("prefill_2816", SHAPES_2816, 30, 128, 8, 16, LFU, None),
    # decode, 40 layers, SiLU, 64 slots, Zipf(0.9); batches 1 and 8; LFU and LRU
    "decode_2048": Workload("decode_2048", SHAPES_2048, 40, 1, 256, 64, LFU, 0.9),
    # stress sweep on the 2816 shapes, 48 layers, uniform routing
    "stress_2816": Workload("stress_2816", SHAPES_2816, 48, 1, 16, 16, LFU, None),
}


def expert_bytes(s: Shapes) -> int:
    """Bytes of one routed expert (gate + up + down codes, scales and biases)."""
    gu = s.d_ff * (s.d_model // 2 + 4 * (s.d_model // 64))
    dn = s.d_model * (s.d_ff // 2 + 4 * (s.d_ff // 64))
    return 2 * gu + dn


# ---------------------------------------------------------------------------
# generation


def _matrix(seed, layer, sub, t_codes, t_scale, n, k, bits=4, lo=0.005, hi=0.02, div=1.0, bias_mult=-8.0,
            out=None):
    """One quantised matrix; writes into out=(codes, scale, bias) when given."""
    lib = _load()
    if out is None:
        codes = np.empty((n, k // 2 if bits == 4 else k), np.uint8)
        scale = np.empty((n, k // 64), np.uint16)
        bias = np.empty((n, k // 64), np.uint16)
    else:
        codes, scale, bias = out
    if bits == 4:
        lib.synth_codes_u4(key(seed, t_codes, layer, sub), n * k, _ptr(codes))
    else:
        lib.synth_codes_u8(key(seed, t_codes, layer, sub), n * k, _ptr(codes))
    lib.synth_scale_bias_f16(key(seed, t_scale, layer, sub), n * (k // 64), lo, hi, div, bias_mult,
                             _ptr(scale), _ptr(bias))
    return codes, scale, bias


def router_weights(s: Shapes, layer: int, seed: int = 0):
    """Router [E x d]: 8-bit codes, binary16 scale and bias per group of 64."""
    return _matrix(seed, layer, 0, T_ROUTER_CODES, T_ROUTER_SCALE, s.n_experts, s.d_model, bits=8,
                   div=float(np.sqrt(s.d_model)), bias_mult=-128.0)


def ffn_weights(s: Shapes, layer: int, expert: int, seed: int = 0, shared: bool = False, out=None):
    """One gated FFN: (gate, up, down) triples of (codes, scale, bias).

    Routed expert e uses stream sub-index e; the shared expert uses the shared
    tensor ids with sub-index 0. out: optional preallocated triples to fill.
    """
    off = T_SHARED_OFFSET if shared else 0
    inter = s.d_ff_shared if shared else s.d_ff
    sub = 0 if shared else expert
    o = out or (None, None, None)
    g = _matrix(seed, layer, sub, T_GATE_CODES + off, T_GATE_SCALE + off, inter, s.d_model, out=o[0])
    u = _matrix(seed, layer, sub, T_UP_CODES + off, T_UP_SCALE + off, inter, s.d_model, out=o[1])
    dn = _matrix(seed, layer, sub, T_DOWN_CODES + off, T_DOWN_SCALE + off, s.d_model, inter, out=o[2])
    return g, u, dn


@dataclass
class LayerWeights:
    """Canonical-layout weights of one MoE layer (numpy arrays; binary16 as uint16 bits)."""

    shapes: Shapes
    router: tuple  # (codes [E,d] u8, scale [E,d/64], bias [E,d/64])
    shared: tuple  # ((gc,gs,gb),(uc,us,ub),(dc,ds,db))
    # routed experts stacked on a leading E axis
    gate_codes: np.ndarray
    gate_scale: np.ndarray
    gate_bias: np.ndarray
    up_codes: np.ndarray
    up_scale: np.ndarray
    up_bias: np.ndarray
    down_codes: np.ndarray
    down_scale: np.ndarray
    down_bias: np.ndarray

    def expert(self, e: int):
        return ((self.gate_codes[e], self.gate_scale[e], self.gate_bias[e]),
                (self.up_codes[e], self.up_scale[e], self.up_bias[e]),
                (self.down_codes[e], self.down_scale[e], self.down_bias[e]))


def layer_weights(s: Shapes, layer: int, seed: int = 0, threads: int | None = None,
                  reuse: LayerWeights | None = None) -> LayerWeights:
    """All weights of one layer. reuse: a LayerWeights of the same shapes whose
    routed arrays are overwritten (saves the allocation of ~1 GB per layer)."""
    E, d, I = s.n_experts, s.d_model, s.d_ff
    if reuse is not None and reuse.shapes == s:
        gc, gs, gb = reuse.gate_codes, reuse.gate_scale, reuse.gate_bias
        uc, us, ub = reuse.up_codes, reuse.up_scale, reuse.up_bias
        dc, ds, db = reuse.down_codes, reuse.down_scale, reuse.down_bias
    else:
        gc = np.empty((E, I, d // 2), np.uint8)
        gs = np.empty((E, I, d // 64), np.uint16)
        gb = np.empty_like(gs)
        uc = np.empty_like(gc)
        us = np.empty_like(gs)
        ub = np.empty_like(gs)
        dc = np.empty((E, d, I // 2), np.uint8)
        ds = np.empty((E, d, I // 64), np.uint16)
        db = np.empty_like(ds)

    def one(e):
        ffn_weights(s, layer, e, seed, out=((gc[e], gs[e], gb[e]), (uc[e], us[e], ub[e]), (dc[e], ds[e], db[e])))

    nthreads = threads or min(32, os.cpu_count() or 1)
    if E > 1 and nthreads > 1:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(one, range(E)))
    else:
        for e in range(E):
            one(e)
    return LayerWeights(s, router_weights(s, layer, seed), ffn_weights(s, layer, 0, seed, shared=True),
                        gc, gs, gb, uc, us, ub, dc, ds, db)


def tokens(s: Shapes, layer: int, step: int, n_tokens: int, rms_normalise: bool, seed: int = 0) -> np.ndarray:
    """x for (step, layer): [n_tokens x d] bfloat16 bits (uint16)."""
    out = np.empty((n_tokens, s.d_model), np.uint16)
    scratch = np.empty(s.d_model, np.float64)
    _load().synth_normal_bf16(key(seed, T_X, layer, step), n_tokens, s.d_model, int(rms_normalise),
                              _ptr(out), _ptr(scratch))
    return out


def zipf_bias(s: Shapes, layer: int, zipf_s: float, beta: float = 1.0, seed: int = 0) -> np.ndarray:
    """Per-expert additive router bias: expert of rank r gets -beta * s * ln(r)."""
    perm = np.empty(s.n_experts, np.int32)
    _load().synth_permutation(key(seed, T_ZIPF_PERM, layer, 0), s.n_experts, _ptr(perm))
    out = np.empty(s.n_experts, np.float32)
    for r in range(s.n_experts):
        out[perm[r]] = np.float32(-beta * zipf_s * np.log(r + 1.0))
    return out


def f16(bits: np.ndarray) -> np.ndarray:
    """View binary16 bit patterns as numpy float16."""
    return np.asarray(bits, np.uint16).view(np.float16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact bfloat16 -> float32 (bit shift)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
