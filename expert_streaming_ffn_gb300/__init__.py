"""Python binding of libmoe, the expert-streaming MoE layer for GB300.

Argument marshalling only: every step of the layer runs in the CUDA library
(``_build/libmoe.so``, built from ``csrc/`` by ``build.py``). There is no CPU
fallback: if the library is missing and cannot be built, ``load()`` raises.

Functions carry the C ABI's names (see include/moe.h). Device buffers are torch
CUDA tensors (PyTorch provides device memory and streams only); host buffers
are numpy arrays.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB
_lib = None

MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA, MOE_ECOPY, MOE_ETIMEOUT, MOE_ESTATE, MOE_EBUSY, MOE_EIO = range(9)
MOE_STORE_DIRECT = 1
LFU, LRU = 0, 1
GELU_TANH, SILU = 0, 1
KERNEL_KINDS = ("router", "expert_ffn", "combine", "gemm_gateup", "gemm_down", "pf_gather", "expert_ffn_miss")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)}: {message}")
        self.status = status


_STATUS = {0: "MOE_OK", 1: "MOE_EINVAL", 2: "MOE_ENOMEM", 3: "MOE_ECUDA", 4: "MOE_ECOPY", 5: "MOE_ETIMEOUT",
           6: "MOE_ESTATE", 7: "MOE_EBUSY", 8: "MOE_EIO"}


class moe_shapes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("d_model", "n_experts", "top_k", "d_ff", "d_ff_shared", "act")]


class moe_quant_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("w_bits", "w_group", "r_bits", "r_group")]


class moe_qmatrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class moe_host_weights(ctypes.Structure):
    _fields_ = [(n, moe_qmatrix) for n in ("router", "shared_gate", "shared_up", "shared_down", "gate", "up",
                                             "down")]


class moe_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("bypass", ctypes.c_uint64), ("bytes_h2d", ctypes.c_uint64), ("bytes_resident", ctypes.c_uint64),
                ("exposed_copy_us", ctypes.c_double), ("host_wait_us", ctypes.c_double),
                ("host_issue_us", ctypes.c_double)]


class moe_store_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("fetches", "tier_hits", "reads", "prefetch_reads", "prefetch_used",
                                                "bytes_read", "read_errors")] + \
               [("read_us", ctypes.c_double), ("wait_us", ctypes.c_double), ("direct", ctypes.c_int32),
                ("host_slots", ctypes.c_int32), ("readers", ctypes.c_int32)]


# (name, restype, argtypes) of every exported symbol in include/moe.h
_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_P = ctypes.POINTER
SIGNATURES = [
    ("moe_ctx_create", _i32, [ctypes.c_int, _P(_vp)]),
    ("moe_ctx_destroy", None, [_vp]),
    ("moe_layer_create", _i32, [_vp, _P(moe_shapes), _P(moe_quant_layout), _i32, _i32, _P(_vp)]),
    ("moe_layer_set_weights", _i32, [_vp, _P(moe_host_weights)]),
    ("moe_expert_bytes", _sz, [_P(moe_shapes)]),
    ("moe_route", _i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    ("moe_route_noalloc", _i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    ("moe_cache_step", _i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    ("moe_forward", _i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    ("moe_forward_prompt", _i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    ("moe_cache_reset", _i32, [_vp]),
    ("moe_layer_stats", _i32, [_vp, _P(moe_stats)]),
    ("moe_layer_reset_stats", _i32, [_vp]),
    ("moe_cache_dump", _i32, [_vp, _vp, _vp]),
    ("moe_layer_destroy", None, [_vp]),
    ("moe_host_cache_create", _i32, [_i32, _i32, _i32, _P(_vp)]),
    ("moe_host_cache_step", _i32, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    ("moe_host_cache_dump", _i32, [_vp, _vp, _vp]),
    ("moe_host_cache_destroy", None, [_vp]),
    ("moe_group_pairs", _i32, [_vp, _i32, _i32, _vp, _vp]),
    ("moe_status_str", ctypes.c_char_p, [_i32]),
    ("moe_last_error", ctypes.c_char_p, []),
    ("moe_ctx_set_profiling", _i32, [_vp, _i32]),
    ("moe_ctx_kernel_times", _i32, [_vp, _i32, _P(ctypes.c_uint64), _P(ctypes.c_double), _P(ctypes.c_double),
                                    _P(ctypes.c_double)]),
    ("moe_ctx_reset_kernel_times", _i32, [_vp]),
    ("moe_ctx_launches", _i32, [_vp, _P(ctypes.c_uint64)]),
    ("moe_ctx_inject_copy_failure", _i32, [_vp, _i64]),
    ("moe_store_expert_stride", _sz, [_P(moe_shapes)]),
    ("moe_store_write", _i32, [ctypes.c_char_p, _P(moe_shapes), _P(moe_host_weights)]),
    ("moe_store_open", _i32, [ctypes.c_char_p, _P(moe_shapes), _i32, _i32, _i32, _P(_vp)]),
    ("moe_store_close", _i32, [_vp]),
    ("moe_store_fetch", _i32, [_vp, _i32, _P(_vp)]),
    ("moe_store_release", _i32, [_vp, _i32]),
    ("moe_store_prefetch", _i32, [_vp, _vp, _i32, _P(_i32)]),
    ("moe_store_wait_idle", _i32, [_vp]),
    ("moe_store_set_read_chunk", _i32, [_vp, _sz]),
    ("moe_store_get_stats", _i32, [_vp, _P(moe_store_stats)]),
    ("moe_store_reset_stats", _i32, [_vp]),
    ("moe_store_tier", _i32, [_vp, _vp, _vp]),
    ("moe_layer_create_streamed", _i32, [_vp, _P(moe_shapes), _P(moe_quant_layout), _i32, _i32, _vp, _P(_vp)]),
    ("moe_layer_prefetch", _i32, [_vp, _i32, _P(_i32)]),
    ("moe_layers_replay_resident", _i32, [_P(_vp), _i32, _i32, _vp, _P(ctypes.c_double)]),
    ("moe_layer_set_deterministic", _i32, [_vp, _i32]),
    ("moe_layer_set_prefetch", _i32, [_vp, _i32]),
    ("moe_layer_prefetch_stats", _i32, [_vp, _P(ctypes.c_uint64), _P(ctypes.c_uint64)]),
]


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmoe.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmoe.so not found at {LIB_PATH}; build it with expert_streaming_ffn_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where, load().moe_last_error().decode(errors="replace"))


def _dptr(t) -> int | None:
    """Device pointer of a torch CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def _hptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ---------------------------------------------------------------------------
# context and layer


def moe_ctx_create(device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load().moe_ctx_create(device, ctypes.byref(h)), "moe_ctx_create")
    return h.value


def moe_ctx_destroy(ctx: int) -> None:
    load().moe_ctx_destroy(ctx)


def make_shapes(s) -> moe_shapes:
    return moe_shapes(s.d_model, s.n_experts, s.top_k, s.d_ff, s.d_ff_shared, s.act)


def moe_expert_bytes(shapes) -> int:
    sh = make_shapes(shapes)
    return load().moe_expert_bytes(ctypes.byref(sh))


def moe_layer_create(ctx: int, shapes, cache_slots: int, policy: int = LFU) -> int:
    sh = make_shapes(shapes)
    q = moe_quant_layout(4, 64, 8, 64)
    h = ctypes.c_void_p()
    _check(load().moe_layer_create(ctx, ctypes.byref(sh), ctypes.byref(q), cache_slots, policy, ctypes.byref(h)),
           "moe_layer_create")
    return h.value


def moe_layer_destroy(layer: int) -> None:
    load().moe_layer_destroy(layer)


def _qm(codes, scale, bias, keep) -> moe_qmatrix:
    c = np.ascontiguousarray(codes, np.uint8)
    s = np.ascontiguousarray(scale, np.uint16)
    b = np.ascontiguousarray(bias, np.uint16)
    keep += [c, s, b]
    return moe_qmatrix(_hptr(c), _hptr(s), _hptr(b))


def _host_weights(w, keep: list, routed: bool = True, resident: bool = True) -> moe_host_weights:
    """moe_host_weights over canonical-layout arrays (the attributes of
    synth.LayerWeights); the routed or the resident matrices may be left NULL."""
    null = moe_qmatrix(None, None, None)
    g, u, d = w.shared
    res = [_qm(*w.router, keep), _qm(*g, keep), _qm(*u, keep), _qm(*d, keep)] if resident else [null] * 4
    rt = [_qm(w.gate_codes, w.gate_scale, w.gate_bias, keep), _qm(w.up_codes, w.up_scale, w.up_bias, keep),
          _qm(w.down_codes, w.down_scale, w.down_bias, keep)] if routed else [null] * 3
    return moe_host_weights(*res, *rt)


def moe_layer_set_weights(layer: int, w, routed: bool = True) -> None:
    """w: canonical-layout arrays with the attributes of synth.LayerWeights.
    routed=False passes NULL routed matrices (a streamed layer reads them from
    its store)."""
    keep: list = []
    hw = _host_weights(w, keep, routed=routed)
    _check(load().moe_layer_set_weights(layer, ctypes.byref(hw)), "moe_layer_set_weights")


def moe_route(layer: int, x, top_k: int, zbias=None, ids=None, gates=None, stream=None):
    """x: CUDA bf16 [T][d]. Returns (ids int32 [T][k], gates f32 [T][k]) CUDA tensors."""
    import torch

    T = x.shape[0]
    if ids is None:
        ids = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if gates is None:
        gates = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    _check(load().moe_route(layer, _dptr(x), T, _dptr(zbias), _dptr(ids), _dptr(gates), _stream(stream)),
           "moe_route")
    return ids, gates


def moe_route_noalloc(layer: int, x, zbias, ids, gates, stream=None):
    """moe_route into caller-provided CUDA buffers, with no allocation anywhere:
    x bf16 [T][d], ids int32 [T][k], gates f32 [T][k] (T <= 64)."""
    _check(load().moe_route_noalloc(layer, _dptr(x), x.shape[0], _dptr(zbias), _dptr(ids), _dptr(gates),
                                    _stream(stream)), "moe_route_noalloc")


def moe_layer_set_prefetch(layer: int, on: bool = True):
    """Keep one spare expert buffer in HBM, refilled with the most-routed expert not cached."""
    _check(load().moe_layer_set_prefetch(layer, int(bool(on))), "moe_layer_set_prefetch")


def moe_layer_prefetch_stats(layer: int) -> dict:
    issued, used = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check(load().moe_layer_prefetch_stats(layer, ctypes.byref(issued), ctypes.byref(used)), "moe_layer_prefetch_stats")
    return {"issued": issued.value, "used": used.value}


def moe_layer_set_deterministic(layer: int, on: bool = True):
    """Decode calls sum their output in a fixed order (bit-identical repeats)."""
    _check(load().moe_layer_set_deterministic(layer, int(bool(on))), "moe_layer_set_deterministic")


def moe_layers_replay_resident(layers, rounds: int = 1, stream=None) -> float:
    """Enqueue, `rounds` times, each layer's last one-token resident FFN launch
    (kernel timing only: each adds into its call's y again). Returns the
    weight bytes all the launches read."""
    arr = (_vp * len(layers))(*layers)
    by = ctypes.c_double(0.0)
    _check(load().moe_layers_replay_resident(arr, len(layers), rounds, _stream(stream), ctypes.byref(by)),
           "moe_layers_replay_resident")
    return by.value


def moe_cache_reset(layer: int):
    """Empty the layer's expert cache (slots free, counts zero)."""
    _check(load().moe_cache_reset(layer), "moe_cache_reset")


def moe_cache_step(layer: int, ids) -> dict:
    """ids: host int array (any shape). Returns slot map and miss list (numpy)."""
    ids = np.ascontiguousarray(np.asarray(ids).reshape(-1), np.int32)
    n = ids.shape[0]
    slot_of = np.empty(n, np.int32)
    me = np.empty(max(n, 1), np.int32)
    ms = np.empty(max(n, 1), np.int32)
    nm = ctypes.c_int32()
    _check(load().moe_cache_step(layer, _hptr(ids), n, _hptr(slot_of), _hptr(me), _hptr(ms), ctypes.byref(nm)),
           "moe_cache_step")
    return dict(slot_of=slot_of, miss_experts=me[:nm.value].copy(), miss_slots=ms[:nm.value].copy())


def moe_forward(layer: int, x, zbias=None, y=None, ids_out=None, gates_out=None, stream=None):
    """x: CUDA bf16 [T][d]. Returns y (CUDA f32 [T][d])."""
    import torch

    T, d = x.shape
    if y is None:
        y = torch.empty((T, d), dtype=torch.float32, device=x.device)
    _check(load().moe_forward(layer, _dptr(x), T, _dptr(zbias), _dptr(y), _dptr(ids_out), _dptr(gates_out),
                              _stream(stream)), "moe_forward")
    return y


def moe_forward_prompt(layer: int, x, zbias=None, y=None, ids_out=None, gates_out=None, stream=None):
    """The whole prompt x (CUDA bf16 [T][d]) in one layer-major call: one
    routing, one cache step, grouped GEMMs over all of it. Returns y."""
    import torch

    T, d = x.shape
    if y is None:
        y = torch.empty((T, d), dtype=torch.float32, device=x.device)
    _check(load().moe_forward_prompt(layer, _dptr(x), T, _dptr(zbias), _dptr(y), _dptr(ids_out), _dptr(gates_out),
                                     _stream(stream)), "moe_forward_prompt")
    return y


def moe_forward_ptr(layer: int, x_ptr: int, T: int, zbias_ptr, y_ptr: int, stream) -> None:
    """moe_forward on raw device pointers (no tensor checks)."""
    _check(load().moe_forward(layer, x_ptr, T, zbias_ptr, y_ptr, None, None, stream), "moe_forward")


def moe_layer_stats(layer: int) -> dict:
    st = moe_stats()
    _check(load().moe_layer_stats(layer, ctypes.byref(st)), "moe_layer_stats")
    return {n: getattr(st, n) for n, _ in moe_stats._fields_}


def moe_layer_reset_stats(layer: int) -> None:
    _check(load().moe_layer_reset_stats(layer), "moe_layer_reset_stats")


def moe_cache_dump(layer: int, slots: int):
    se = np.empty(slots, np.int32)
    cnt = np.empty(slots, np.uint32)
    _check(load().moe_cache_dump(layer, _hptr(se), _hptr(cnt)), "moe_cache_dump")
    return se, cnt


# ---------------------------------------------------------------------------
# host cache manager (no GPU needed)


def moe_host_cache_create(n_experts: int, slots: int, policy: int = LFU) -> int:
    h = ctypes.c_void_p()
    _check(load().moe_host_cache_create(n_experts, slots, policy, ctypes.byref(h)), "moe_host_cache_create")
    return h.value


def moe_host_cache_step(cache: int, ids) -> dict:
    ids = np.ascontiguousarray(np.asarray(ids).reshape(-1), np.int32)
    n = ids.shape[0]
    slot_of = np.empty(n, np.int32)
    me = np.empty(max(n, 1), np.int32)
    ms = np.empty(max(n, 1), np.int32)
    nm, nh, nb = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().moe_host_cache_step(cache, _hptr(ids), n, _hptr(slot_of), _hptr(me), _hptr(ms), ctypes.byref(nm),
                                      ctypes.byref(nh), ctypes.byref(nb)), "moe_host_cache_step")
    return dict(slot_of=slot_of, miss_experts=me[:nm.value].copy(), miss_slots=ms[:nm.value].copy(), hits=nh.value,
                misses=nm.value, bypass=nb.value)


def moe_host_cache_dump(cache: int, slots: int):
    se = np.empty(slots, np.int32)
    cnt = np.empty(slots, np.uint32)
    _check(load().moe_host_cache_dump(cache, _hptr(se), _hptr(cnt)), "moe_host_cache_dump")
    return se, cnt


def moe_host_cache_destroy(cache: int) -> None:
    load().moe_host_cache_destroy(cache)


def moe_group_pairs(ids, n_experts: int):
    ids = np.ascontiguousarray(np.asarray(ids).reshape(-1), np.int32)
    n = ids.shape[0]
    offsets = np.empty(n_experts + 1, np.int32)
    perm = np.empty(max(n, 1), np.int32)
    _check(load().moe_group_pairs(_hptr(ids), n, n_experts, _hptr(offsets), _hptr(perm)), "moe_group_pairs")
    return offsets, perm[:n].copy()


# ---------------------------------------------------------------------------
# storage tier (expert files; no GPU needed except for streamed layers)


def moe_store_expert_stride(shapes) -> int:
    sh = make_shapes(shapes)
    return load().moe_store_expert_stride(ctypes.byref(sh))


def moe_store_write(path: str, shapes, w) -> None:
    """Write the routed experts of w (canonical layout) as an expert file."""
    sh = make_shapes(shapes)
    keep: list = []
    hw = _host_weights(w, keep, resident=False)
    _check(load().moe_store_write(os.fsencode(path), ctypes.byref(sh), ctypes.byref(hw)), "moe_store_write")


def moe_store_open(path: str, shapes, host_slots: int, readers: int = 4, flags: int = 0) -> int:
    sh = make_shapes(shapes)
    h = ctypes.c_void_p()
    _check(load().moe_store_open(os.fsencode(path), ctypes.byref(sh), host_slots, readers, flags, ctypes.byref(h)),
           "moe_store_open")
    return h.value


def moe_store_close(store: int) -> None:
    _check(load().moe_store_close(store), "moe_store_close")


def moe_store_fetch(store: int, expert: int, nbytes: int) -> np.ndarray:
    """Fetch (and pin) an expert; returns a copy of its first nbytes bytes."""
    p = ctypes.c_void_p()
    _check(load().moe_store_fetch(store, expert, ctypes.byref(p)), "moe_store_fetch")
    return np.ctypeslib.as_array(ctypes.cast(p, ctypes.POINTER(ctypes.c_uint8)), shape=(nbytes,)).copy()


def moe_store_release(store: int, expert: int) -> None:
    _check(load().moe_store_release(store, expert), "moe_store_release")


def moe_store_prefetch(store: int, experts) -> int:
    e = np.ascontiguousarray(np.asarray(experts).reshape(-1), np.int32)
    q = ctypes.c_int32()
    _check(load().moe_store_prefetch(store, _hptr(e) if e.size else None, e.size, ctypes.byref(q)),
           "moe_store_prefetch")
    return q.value


def moe_store_set_read_chunk(store: int, nbytes: int) -> None:
    """Read experts as pieces of nbytes (a multiple of 4096; 0 = whole) spread over the readers."""
    _check(load().moe_store_set_read_chunk(store, nbytes), "moe_store_set_read_chunk")


def moe_store_wait_idle(store: int) -> None:
    _check(load().moe_store_wait_idle(store), "moe_store_wait_idle")


def moe_store_get_stats(store: int) -> dict:
    st = moe_store_stats()
    _check(load().moe_store_get_stats(store, ctypes.byref(st)), "moe_store_get_stats")
    return {n: getattr(st, n) for n, _ in moe_store_stats._fields_}


def moe_store_reset_stats(store: int) -> None:
    _check(load().moe_store_reset_stats(store), "moe_store_reset_stats")


def moe_store_tier(store: int, host_slots: int):
    """(expert per entry, state per entry): 0 empty, 1 being read, 2 ready, 3 failed."""
    ex = np.empty(host_slots, np.int32)
    stt = np.empty(host_slots, np.int32)
    _check(load().moe_store_tier(store, _hptr(ex), _hptr(stt)), "moe_store_tier")
    return ex, stt


def moe_layer_create_streamed(ctx: int, shapes, cache_slots: int, store: int, policy: int = LFU) -> int:
    sh = make_shapes(shapes)
    q = moe_quant_layout(4, 64, 8, 64)
    h = ctypes.c_void_p()
    _check(load().moe_layer_create_streamed(ctx, ctypes.byref(sh), ctypes.byref(q), cache_slots, policy, store,
                                            ctypes.byref(h)), "moe_layer_create_streamed")
    return h.value


def moe_layer_prefetch(layer: int, n: int) -> int:
    q = ctypes.c_int32()
    _check(load().moe_layer_prefetch(layer, n, ctypes.byref(q)), "moe_layer_prefetch")
    return q.value


# ---------------------------------------------------------------------------
# diagnostics


def moe_status_str(status: int) -> str:
    return load().moe_status_str(status).decode()


def moe_last_error() -> str:
    return load().moe_last_error().decode(errors="replace")


def moe_ctx_set_profiling(ctx: int, on: bool) -> None:
    _check(load().moe_ctx_set_profiling(ctx, int(bool(on))), "moe_ctx_set_profiling")


def moe_ctx_kernel_times(ctx: int) -> dict:
    """{kind: (launches, total_ms, bytes, flops)} for every kernel kind."""
    out = {}
    for i, name in enumerate(KERNEL_KINDS):
        n, ms, by, fl = ctypes.c_uint64(), ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        _check(load().moe_ctx_kernel_times(ctx, i, ctypes.byref(n), ctypes.byref(ms), ctypes.byref(by),
                                           ctypes.byref(fl)), "moe_ctx_kernel_times")
        out[name] = (n.value, ms.value, by.value, fl.value)
    return out


def moe_ctx_reset_kernel_times(ctx: int) -> None:
    _check(load().moe_ctx_reset_kernel_times(ctx), "moe_ctx_reset_kernel_times")


def moe_ctx_launches(ctx: int) -> int:
    n = ctypes.c_uint64()
    _check(load().moe_ctx_launches(ctx, ctypes.byref(n)), "moe_ctx_launches")
    return n.value


def moe_ctx_inject_copy_failure(ctx: int, nth: int) -> None:
    _check(load().moe_ctx_inject_copy_failure(ctx, nth), "moe_ctx_inject_copy_failure")
