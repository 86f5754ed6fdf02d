"""CPU oracle for the expert-streaming MoE layer (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never loads it and
shares no code with it. The arithmetic lives in ``oracle.c`` (plain C,
single-threaded, -ffp-contract=off); this module builds it with gcc and
marshals numpy arrays.

Pages cited (by title and section):
  [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
  [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
Every function's citation is in its C counterpart's comment.

Parity pins (tests/test_oracle_pins.py) hold this code to the mathematics:
closed-form examples, textbook special cases, invariants, brute force on tiny
inputs and the hand-replayed cache trace in tests/golden/.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_ORACLE_SOURCE may name another copy of oracle.c (the mutation test plants
# one mistake in a scratch copy to check that the pins catch it); it is built
# beside that copy. Unset, this directory's oracle.c is used.
_SRC = os.environ.get("MOE_ORACLE_SOURCE") or os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(os.path.dirname(_SRC), "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

GELU_TANH, SILU = 0, 1
LFU, LRU = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with the host C compiler."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("d", "E", "k", "I", "Is", "act")] + [
        (n, ctypes.c_void_p) for n in (
            "rc", "rs", "rb",
            "sgc", "suc", "sdc",
            "sgs", "sgb", "sus", "sub", "sds", "sdb",
            "gc", "uc", "dc",
            "gs", "gb", "us", "ub", "ds", "db")]


class _Cache(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("S", ctypes.c_int), ("policy", ctypes.c_int), ("step", ctypes.c_int64),
                ("slot_expert", ctypes.c_int32 * 1024), ("count", ctypes.c_uint32 * 1024),
                ("tick", ctypes.c_int64 * 1024)]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.oracle_f16.restype = dbl
            lib.oracle_f16.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16.restype = ctypes.c_float
            lib.oracle_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_code_u4.restype = ctypes.c_uint
            lib.oracle_code_u4.argtypes = [vp, i32, i32, i32]
            lib.oracle_w4.restype = dbl
            lib.oracle_w4.argtypes = [vp, vp, vp, i32, i32, i32]
            lib.oracle_w8.restype = dbl
            lib.oracle_w8.argtypes = [vp, vp, vp, i32, i32, i32]
            lib.oracle_router_logits.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
            lib.oracle_router_logits_f64.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
            lib.oracle_topk_gates.argtypes = [vp, i32, i32, i32, vp, vp]
            lib.oracle_act.restype = dbl
            lib.oracle_act.argtypes = [dbl, i32]
            lib.oracle_ffn.argtypes = [vp, i32, i32, i32] + [vp] * 9 + [vp]
            lib.oracle_shared_ffn.argtypes = [vp, vp, vp]
            lib.oracle_expert_ffn.argtypes = [vp, i32, vp, vp]
            lib.oracle_moe_layer.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
            lib.oracle_moe_layer_dense.argtypes = [vp, vp, i32, vp, vp]
            lib.oracle_cache_init.restype = i32
            lib.oracle_cache_init.argtypes = [vp, i32, i32, i32]
            lib.oracle_cache_step.restype = i32
            lib.oracle_cache_step.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp]
            lib.oracle_cache_dump.argtypes = [vp, vp, vp]
            lib.oracle_cache_size.restype = i32
            lib.oracle_group_pairs.argtypes = [vp, i32, i32, vp, vp]
            assert lib.oracle_cache_size() == ctypes.sizeof(_Cache)
            _lib = lib
    return _lib


def _c(a, dtype):
    """C-contiguous array of dtype (no copy when already so)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------------------
# scalar helpers


def f16(bits: int) -> float:
    return _load().oracle_f16(int(bits))


def bf16(bits: int) -> float:
    return _load().oracle_bf16(int(bits))


def code_u4(codes: np.ndarray, K: int, n: int, k: int) -> int:
    codes = _c(codes, np.uint8)
    return _load().oracle_code_u4(_p(codes), K, n, k)


def w4(codes, scale, bias, K, n, k) -> float:
    codes, scale, bias = _c(codes, np.uint8), _c(scale, np.uint16), _c(bias, np.uint16)
    return _load().oracle_w4(_p(codes), _p(scale), _p(bias), K, n, k)


def act(z: float, kind: int) -> float:
    return _load().oracle_act(float(z), kind)


# ---------------------------------------------------------------------------
# router


def router_logits(x, router, E: int, zbias=None) -> np.ndarray:
    """fp32 logits [T][E] in the fixed lane-strided order. x: [T][d] bf16 bits."""
    x = _c(x, np.uint16)
    T, d = x.shape
    codes, scale, bias = (_c(router[0], np.uint8), _c(router[1], np.uint16), _c(router[2], np.uint16))
    zb = None if zbias is None else _c(zbias, np.float32)
    out = np.empty((T, E), np.float32)
    _load().oracle_router_logits(_p(x), T, d, E, _p(codes), _p(scale), _p(bias), _p(zb), _p(out))
    return out


def router_logits_f64(x, router, E: int, zbias=None) -> np.ndarray:
    x = _c(x, np.uint16)
    T, d = x.shape
    codes, scale, bias = (_c(router[0], np.uint8), _c(router[1], np.uint16), _c(router[2], np.uint16))
    zb = None if zbias is None else _c(zbias, np.float32)
    out = np.empty((T, E), np.float64)
    _load().oracle_router_logits_f64(_p(x), T, d, E, _p(codes), _p(scale), _p(bias), _p(zb), _p(out))
    return out


def topk_gates(logits, k: int):
    """(ids [T][k] int32, gates [T][k] float64) from fp32 logits [T][E]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    gates = np.empty((T, k), np.float64)
    _load().oracle_topk_gates(_p(logits), T, E, k, _p(ids), _p(gates))
    return ids, gates


# ---------------------------------------------------------------------------
# FFN and layer


def ffn(x_row, gate, up, down, act_kind: int) -> np.ndarray:
    """One gated FFN on one token. gate/up/down are (codes, scale, bias) in canonical layout."""
    x_row = _c(x_row, np.uint16)
    d = x_row.shape[0]
    inter = np.asarray(gate[0]).shape[0]
    arrs = [(_c(m[0], np.uint8), _c(m[1], np.uint16), _c(m[2], np.uint16)) for m in (gate, up, down)]
    out = np.empty(d, np.float64)
    flat = [_p(a) for m in arrs for a in m]
    _load().oracle_ffn(_p(x_row), d, inter, act_kind, *flat, _p(out))
    return out


class Layer:
    """Holds one layer's canonical arrays and the C struct that points at them.

    ``weights`` is any object with the attributes of ``synth.LayerWeights``
    (router, shared, gate_codes, ...); only numpy arrays are read from it.
    """

    def __init__(self, weights, shapes):
        self.shapes = shapes
        keep = {}

        def put(name, a, dtype):
            a = _c(a, dtype)
            keep[name] = a
            return _p(a)

        s = _Layer()
        s.d, s.E, s.k, s.I, s.Is, s.act = (shapes.d_model, shapes.n_experts, shapes.top_k, shapes.d_ff,
                                          shapes.d_ff_shared, shapes.act)
        s.rc = put("rc", weights.router[0], np.uint8)
        s.rs = put("rs", weights.router[1], np.uint16)
        s.rb = put("rb", weights.router[2], np.uint16)
        (g, u, dn) = weights.shared
        s.sgc, s.sgs, s.sgb = put("sgc", g[0], np.uint8), put("sgs", g[1], np.uint16), put("sgb", g[2], np.uint16)
        s.suc, s.sus, s.sub = put("suc", u[0], np.uint8), put("sus", u[1], np.uint16), put("sub", u[2], np.uint16)
        s.sdc, s.sds, s.sdb = put("sdc", dn[0], np.uint8), put("sds", dn[1], np.uint16), put("sdb", dn[2], np.uint16)
        s.gc, s.gs, s.gb = (put("gc", weights.gate_codes, np.uint8), put("gs", weights.gate_scale, np.uint16),
                            put("gb", weights.gate_bias, np.uint16))
        s.uc, s.us, s.ub = (put("uc", weights.up_codes, np.uint8), put("us", weights.up_scale, np.uint16),
                            put("ub", weights.up_bias, np.uint16))
        s.dc, s.ds, s.db = (put("dc", weights.down_codes, np.uint8), put("ds", weights.down_scale, np.uint16),
                            put("db", weights.down_bias, np.uint16))
        self._keep = keep
        self._s = s

    @property
    def ref(self):
        return ctypes.byref(self._s)

    def forward(self, x, zbias=None):
        """Full layer on T tokens: returns (logits fp32 [T][E], ids [T][k], gates f64 [T][k], y f64 [T][d])."""
        x = _c(x, np.uint16)
        T = x.shape[0]
        sh = self.shapes
        zb = None if zbias is None else _c(zbias, np.float32)
        logits = np.empty((T, sh.n_experts), np.float32)
        ids = np.empty((T, sh.top_k), np.int32)
        gates = np.empty((T, sh.top_k), np.float64)
        y = np.empty((T, sh.d_model), np.float64)
        _load().oracle_moe_layer(self.ref, _p(x), T, _p(zb), _p(logits), _p(ids), _p(gates), _p(y))
        return logits, ids, gates, y

    def forward_dense(self, x, zbias=None):
        """Brute-force dense evaluation of the same layer: y f64 [T][d]."""
        x = _c(x, np.uint16)
        T = x.shape[0]
        zb = None if zbias is None else _c(zbias, np.float32)
        y = np.empty((T, self.shapes.d_model), np.float64)
        _load().oracle_moe_layer_dense(self.ref, _p(x), T, _p(zb), _p(y))
        return y

    def shared_ffn(self, x_row):
        x_row = _c(x_row, np.uint16)
        out = np.empty(self.shapes.d_model, np.float64)
        _load().oracle_shared_ffn(self.ref, _p(x_row), _p(out))
        return out

    def expert_ffn(self, e, x_row):
        x_row = _c(x_row, np.uint16)
        out = np.empty(self.shapes.d_model, np.float64)
        _load().oracle_expert_ffn(self.ref, int(e), _p(x_row), _p(out))
        return out

    def combine(self, x, ids, gates):
        """y for given routing (ids, gates): shared + gate-weighted experts in rank order."""
        x = _c(x, np.uint16)
        T = x.shape[0]
        y = np.empty((T, self.shapes.d_model), np.float64)
        for t in range(T):
            y[t] = self.shared_ffn(x[t])
            for r in range(ids.shape[1]):
                y[t] += float(gates[t, r]) * self.expert_ffn(ids[t, r], x[t])
        return y


# ---------------------------------------------------------------------------
# cache


class Cache:
    """The per-layer LFU / LRU expert cache trace (pure function of the id sequence)."""

    def __init__(self, n_experts: int, slots: int, policy: int = LFU):
        self._c = _Cache()
        if _load().oracle_cache_init(ctypes.byref(self._c), n_experts, slots, policy) != 0:
            raise ValueError("bad cache shape")
        self.E, self.S = n_experts, slots

    def step(self, ids):
        """One lookup step. Returns dict(slot_of, miss_experts, miss_slots, hits, misses, bypass)."""
        ids = _c(np.asarray(ids).reshape(-1), np.int32)
        n = ids.shape[0]
        slot_of = np.empty(n, np.int32)
        me = np.empty(max(n, 1), np.int32)
        ms = np.empty(max(n, 1), np.int32)
        nh, nm, nb = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        rc = _load().oracle_cache_step(ctypes.byref(self._c), _p(ids), n, _p(slot_of), _p(me), _p(ms),
                                       ctypes.byref(nh), ctypes.byref(nm), ctypes.byref(nb))
        if rc != 0:
            raise ValueError("expert id out of range")
        return dict(slot_of=slot_of, miss_experts=me[:nm.value].copy(), miss_slots=ms[:nm.value].copy(),
                    hits=nh.value, misses=nm.value, bypass=nb.value)

    def dump(self):
        se = np.empty(self.S, np.int32)
        cnt = np.empty(self.S, np.uint32)
        _load().oracle_cache_dump(ctypes.byref(self._c), _p(se), _p(cnt))
        return se, cnt


def group_pairs(ids, n_experts: int):
    """Stable grouping of (token, rank) pairs by expert: (offsets [E+1], perm [n_pairs])."""
    ids = _c(np.asarray(ids).reshape(-1), np.int32)
    n = ids.shape[0]
    offsets = np.empty(n_experts + 1, np.int32)
    perm = np.empty(max(n, 1), np.int32)
    _load().oracle_group_pairs(_p(ids), n, n_experts, _p(offsets), _p(perm))
    return offsets, perm[:n].copy()
