#!/usr/bin/env python
"""Benchmark of the expert-streaming MoE layer on GB300.

Workload (default): decode_2816 — 30 MoE layers, one token per step, d=2816,
256 routed experts (top-8, FFN 2816->704->2816), shared expert 2816->2816->2816,
int4 affine g64 experts, 8-bit router, a 16-slot LFU expert cache per layer in
HBM with every other expert in pinned host memory, Zipf(1.1) router bias.
Inputs are seeded and synthetic (see synth/). A step is one token through all
30 layers: route, cache step, miss copies, shared expert, routed experts and
combine, for every layer.

Prints one JSON line. Metric: decode tokens/s (whole job); also the achieved
HBM bandwidth of the dominant kernel against the measured peak, the prefill
chunk rate and expert TFLOP/s, 4 layers streamed from expert files (the
storage tier), the CPU oracle as a baseline, and the same decode metric end
to end with host buffers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --prefill-only | --storage-only | --stress   (one leg, its own JSON)

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer does not shard); value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE decode tok/s + achieved HBM GB/s vs peak; prefill-chunk expert TFLOP/s"
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # The host->device copy path runs up to several times slower for the first
    # ~0.1-0.5 s of sparse copies after setup or idle (measured: the same steps
    # replayed run 2-4x faster), and LFU counts need steps to settle: the
    # default warm-up covers both, so the timed steps measure the steady state.
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--prime-steps", type=int, default=256,
                    help="untimed steps on other inputs that warm the caches before every pass")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (testing only)")
    ap.add_argument("--prefill-layers", type=int, default=2)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill leg and print its JSON (for profiling; not the bench line)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--prefill-resident-only", action="store_true",
                    help="prefill leg: skip the streaming pass (profiling the grouped GEMMs on resident weights)")
    ap.add_argument("--resident", action="store_true",
                    help="every expert resident (one slot per expert, all loaded before the warm-up): "
                         "the decode FFN launches then read HBM only (profiling)")
    ap.add_argument("--no-storage", action="store_true", help="skip the storage-tier leg")
    ap.add_argument("--storage-only", action="store_true",
                    help="run only the storage-tier leg and print its JSON (not the bench line)")
    ap.add_argument("--storage-layers", type=int, default=4)
    ap.add_argument("--storage-steps", type=int, default=64)
    ap.add_argument("--storage-warmup", type=int, default=48)
    ap.add_argument("--storage-host-slots", type=int, default=32)
    ap.add_argument("--storage-readers", type=int, default=8)
    ap.add_argument("--storage-readahead", type=int, default=4)
    ap.add_argument("--storage-dir", default=None, help="where the expert files go (default: the temp dir)")
    ap.add_argument("--stress", action="store_true",
                    help="run the stress sweep (2816 shapes, uniform routing) and print its JSON (not the bench line)")
    ap.add_argument("--stress-layers", type=int, default=8)
    ap.add_argument("--stress-steps", type=int, default=16)
    ap.add_argument("--no-legs", action="store_true",
                    help="skip the decode_2048, all-resident and stress legs of the default line")
    ap.add_argument("--no-stress", action="store_true", help="skip the stress subset of the default line")
    ap.add_argument("--resident-layers", type=int, default=8)
    ap.add_argument("--layers-2048", type=int, default=40)
    ap.add_argument("--stress-layers-line", type=int, default=4)
    ap.add_argument("--stress-steps-line", type=int, default=6)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: a barrier and a max, no data exchange)


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.rows = []
        self.proc = None
        self.bus_id = bus_id

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu=pci.bus_id,{self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.15)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = self.rows
        if self.bus_id:
            mine = [r for r in rows if r[0].lower().endswith(self.bus_id.lower()[-12:])]
            rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def gpu_bus_id(dev: int) -> str | None:
    try:
        import torch

        p = torch.cuda.get_device_properties(dev)
        dom, bus, devid = getattr(p, "pci_domain_id", None), getattr(p, "pci_bus_id", None), getattr(p, "pci_device_id", None)
        if bus is None:
            return None
        return f"{dom or 0:08X}:{bus:02X}:{devid or 0:02X}.0"
    except Exception:
        return None


def ncu_traffic(kernel: str, algorithmic_bytes_per_launch=None):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None
    when the kernel's source has changed since the counters were taken. A
    record taken on a different launch size gives DRAM bytes per algorithmic
    byte, scaled here to this run's launches."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
        if not rec:
            return None
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        if "dram_bytes_per_algorithmic_byte" in rec:
            if algorithmic_bytes_per_launch is None:
                return None
            return rec["dram_bytes_per_algorithmic_byte"] * algorithmic_bytes_per_launch
        return rec["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)


def oracle_layer_tokens(n_max: int, seconds: float, wl, layers=(0, 1)):
    """Time the oracle on whole layer-tokens of the workload (single thread)."""
    import oracle
    import synth

    s = wl.shapes
    times = []
    done = 0
    for li, layer in enumerate(layers):
        w = synth.layer_weights(s, layer, wl.seed)
        L = oracle.Layer(w, s)
        zb = synth.zipf_bias(s, layer, wl.zipf_s, wl.zipf_beta, wl.seed) if wl.zipf_s else None
        per_layer = max(1, n_max // len(layers))
        for step in range(per_layer):
            x = synth.tokens(s, layer, step, 1, wl.rms_normalise, wl.seed)
            t = time.perf_counter()
            L.forward(x, zb)
            times.append(time.perf_counter() - t)
            done += 1
            if sum(times) >= seconds and done >= 2:
                return times
        del L, w
    return times


_ORACLE_STATE = None


def _oracle_worker(seconds: float):
    """One forked worker: whole layer-tokens of the oracle for `seconds`."""
    L, xs, zb = _ORACLE_STATE
    n, t0 = 0, time.perf_counter()
    while True:
        L.forward(xs[n % len(xs)], zb)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            return n, time.perf_counter() - t0


def oracle_all_cores(wl, seconds: float):
    """The oracle as it stands, one single-threaded copy per host core: layer
    0 of the workload is built once and the workers are forked from it (before
    any GPU call in this process), each running whole layer-tokens for
    `seconds`. Returns (layer-tokens per second over all workers, workers)."""
    import multiprocessing

    import oracle
    import synth

    global _ORACLE_STATE
    s = wl.shapes
    w = synth.layer_weights(s, 0, wl.seed)
    zb = synth.zipf_bias(s, 0, wl.zipf_s, wl.zipf_beta, wl.seed) if wl.zipf_s else None
    xs = [synth.tokens(s, 0, st, 1, wl.rms_normalise, wl.seed) for st in range(8)]
    _ORACLE_STATE = (oracle.Layer(w, s), xs, zb)
    P = os.cpu_count() or 1
    try:
        with multiprocessing.get_context("fork").Pool(P) as pool:
            res = pool.map(_oracle_worker, [seconds] * P)
    finally:
        _ORACLE_STATE = None
    return sum(n / t for n, t in res), P


def workload_config(wl, n_layers: int, slots: int, world: int, resident: bool = False) -> dict:
    """The `config` object of a decode bench line (both arms)."""
    s = wl.shapes
    return {"workload": wl.name + (" (every expert resident)" if resident else ""),
            "layers": n_layers, "tokens_per_step": wl.tokens, "d_model": s.d_model,
            "experts": s.n_experts, "top_k": s.top_k, "d_ff": s.d_ff, "d_ff_shared": s.d_ff_shared,
            "cache_slots": slots, "policy": "LFU" if wl.policy == 0 else "LRU", "zipf_s": wl.zipf_s,
            "l2": "inputs larger than L2: 1.23 GB of weights read per token vs 129 MiB L2",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def _oracle_step_worker(task):
    """One forked worker's share of a reference step: the given layer-tokens
    (x of (step, layer)) through layer 0's weights."""
    import synth

    step, layers = task
    L, zb, wl = _ORACLE_STATE
    for layer in layers:
        L.forward(synth.tokens(wl.shapes, layer, step, 1, wl.rms_normalise, wl.seed), zb)
    return len(layers)


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores.

    A step is one token through the workload's layers, split over one forked
    single-threaded copy of the oracle per core (each copy takes every P-th
    layer-token). Each layer-token runs the oracle's whole layer (router,
    top-k, shared expert, the 8 routed experts, combine) on layer 0's weights
    with the x of its own (step, layer); the per-layer work does not depend
    on which layer's weights it reads. When --warmup + --steps whole tokens
    would take more than about two minutes, a step is a bounded sample of
    fewer layer-tokens, and the rate is scaled to tokens. Only rank 0 runs."""
    import multiprocessing

    import oracle
    import synth

    if rank != 0:
        return
    global _ORACLE_STATE
    wl = synth.WORKLOADS["decode_2816"]
    s = wl.shapes
    n_layers = args.layers or wl.n_layers
    w = synth.layer_weights(s, 0, wl.seed)
    zb = synth.zipf_bias(s, 0, wl.zipf_s, wl.zipf_beta, wl.seed) if wl.zipf_s else None
    _ORACLE_STATE = (oracle.Layer(w, s), zb, wl)
    P = os.cpu_count() or 1
    t = time.perf_counter()
    _ORACLE_STATE[0].forward(synth.tokens(s, 0, 0, 1, wl.rms_normalise, wl.seed), zb)
    t_lt = time.perf_counter() - t  # one layer-token, single-threaded
    n_steps = max(1, args.warmup + args.steps)
    budget_s = 120.0
    per_step = n_layers
    if n_steps * -(-per_step // P) * t_lt > budget_s:
        per_step = max(1, min(n_layers, int(budget_s / (n_steps * t_lt)) * P))
    try:
        with multiprocessing.get_context("fork").Pool(min(P, per_step)) as pool:
            def one(step):
                layers = list(range(per_step))
                shares = [(step, layers[i::P]) for i in range(min(P, per_step))]
                return sum(pool.map(_oracle_step_worker, shares))

            for st in range(args.warmup):
                one(st)
            t0 = time.perf_counter()
            for st in range(args.warmup, args.warmup + args.steps):
                one(st)
            elapsed = time.perf_counter() - t0
    finally:
        _ORACLE_STATE = None
    tokens = args.steps * per_step / n_layers
    tok_s = tokens / elapsed
    sample = (f"each step: {per_step} of the {n_layers} layer-tokens of one decode_2816 token, split over "
              f"{min(P, per_step)} forked single-threaded copies of the oracle (layer 0's weights, x per "
              f"(step, layer)); tokens/s = steps x {per_step}/{n_layers} tokens / timed seconds")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * elapsed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded int4/int8 weights and N(0,1) RMS-normalised bf16 activations)",
        "config": workload_config(wl, n_layers, wl.cache_slots, world),
        "cpu_baseline": {"value": tok_s, "unit": "tok/s", "cores": min(P, per_step), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tok_s, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# our arm


class DecodeRig:
    """A stack of decode layers of one workload, their inputs resident in HBM
    (x[step][layer][T][d] bf16, drawn per (step, layer)), and the passes the
    bench times over them."""

    def __init__(self, ctx, dev, stream, wl, n_layers, slots, policy, T, n_steps, seed, resident=False,
                 weights=None, n_prime=0):
        import torch

        import expert_streaming_ffn_gb300 as moe
        import synth

        self.moe, self.torch, self.ctx, self.dev, self.stream = moe, torch, ctx, dev, stream
        self.wl, self.s, self.L, self.T, self.resident = wl, wl.shapes, n_layers, T, resident
        s = self.s
        self.slots = s.n_experts if resident else slots
        self.layers, self.zbs = [], []
        w = weights
        for l in range(n_layers):
            w = synth.layer_weights(s, l, seed, reuse=w)
            h = moe.moe_layer_create(ctx, s, self.slots, policy)
            moe.moe_layer_set_weights(h, w)
            self.layers.append(h)
            self.zbs.append(torch.from_numpy(synth.zipf_bias(s, l, wl.zipf_s, wl.zipf_beta, seed)).to(dev)
                            if wl.zipf_s else None)
        self.last_weights = w
        self.reset()
        self.n_prime = 0 if resident else n_prime
        # inputs of the timed steps, then of the priming steps (other draws)
        xs = np.empty((n_steps + self.n_prime, n_layers, T, s.d_model), np.uint16)
        for st in range(n_steps + self.n_prime):
            draw = st if st < n_steps else 1_000_000 + st - n_steps
            for l in range(n_layers):
                xs[st, l] = synth.tokens(s, l, draw, T, wl.rms_normalise, seed)
        self.xs_np = xs[:n_steps]
        self.n_steps = n_steps
        self.x_dev = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
        self.y_dev = torch.empty((n_layers, T, s.d_model), dtype=torch.float32, device=dev)
        self.row = T * s.d_model * 2
        self.primed_once = False

    def reset(self):
        """Empty caches (the cache trajectory starts again), or with every
        expert resident, every expert copied back in."""
        for h in self.layers:
            self.moe.moe_cache_reset(h)
            if self.resident:
                self.moe.moe_cache_step(h, np.arange(self.s.n_experts))
        self.torch.cuda.synchronize(self.dev)

    def step(self, st):
        base = self.x_dev.data_ptr() + st * self.L * self.row
        sptr = self.stream.cuda_stream
        for l in range(self.L):
            zb = self.zbs[l]
            self.moe.moe_forward_ptr(self.layers[l], base + l * self.row, self.T,
                                     zb.data_ptr() if zb is not None else None, self.y_dev[l].data_ptr(), sptr)

    def prime(self, seconds=1.0):
        """Untimed, before every pass: empty caches, then the priming steps
        (inputs drawn apart from the timed steps'), which leave the caches in
        their steady state whatever the counted warm-up. The first time, the
        priming steps repeat (from empty caches each time) until `seconds`
        have passed: the host-to-device path runs slowly for the first few
        hundred milliseconds of sparse copies after set-up."""
        t0 = time.perf_counter()
        while True:
            self.reset()
            for st in range(self.n_prime):
                self.step(self.n_steps + st)
            self.torch.cuda.synchronize(self.dev)
            if self.primed_once or time.perf_counter() - t0 >= seconds or not self.n_prime:
                break
        self.primed_once = True

    def run(self, warmup, steps, profile=False, clocks=None):
        """Warm-up steps, then `steps` timed ones with CUDA events on the
        launching stream. Returns (ms, stats per layer, kernel times or None,
        launches)."""
        moe, torch = self.moe, self.torch
        for st in range(warmup):
            self.step(st)
        torch.cuda.synchronize(self.dev)
        for h in self.layers:
            moe.moe_layer_reset_stats(h)
        if profile:
            moe.moe_ctx_set_profiling(self.ctx, True)
            moe.moe_ctx_reset_kernel_times(self.ctx)
        launches0 = moe.moe_ctx_launches(self.ctx)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        ctxm = clocks if clocks is not None else _Null()
        with ctxm:
            ev0.record(self.stream)
            for st in range(warmup, warmup + steps):
                self.step(st)
            ev1.record(self.stream)
            torch.cuda.synchronize(self.dev)
        launches = moe.moe_ctx_launches(self.ctx) - launches0
        kt = None
        if profile:
            kt = moe.moe_ctx_kernel_times(self.ctx)
            moe.moe_ctx_set_profiling(self.ctx, False)
        return ev0.elapsed_time(ev1), [moe.moe_layer_stats(h) for h in self.layers], kt, launches

    def close(self):
        for h in self.layers:
            self.moe.moe_layer_destroy(h)
        self.layers = []
        del self.x_dev, self.y_dev


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def _totals(stats):
    keys = ("hits", "misses", "bypass", "bytes_h2d", "bytes_resident", "exposed_copy_us", "host_wait_us",
            "host_issue_us")
    return {k: sum(x[k] for x in stats) for k in keys}


def _kernel_table(kt):
    all_ms = sum(v[1] for v in kt.values())
    return {k: {"launches": v[0], "ms": round(v[1], 4), "share": round(v[1] / all_ms, 4) if all_ms else 0,
                "GB_s": round(v[2] / (v[1] * 1e-3) / 1e9, 1) if v[1] > 0 else None}
            for k, v in kt.items() if v[0] > 0}


def _leg_summary(rig, ms, stats, kt, steps, peaks):
    """tokens/s and what moved, for one timed pass of a decode leg."""
    tot = _totals(stats)
    tokens = steps * rig.T
    lookups = tot["hits"] + tot["misses"]
    out = {"tok_s": tokens / (ms * 1e-3), "ms_per_layer_step": ms / steps / rig.L,
           "hit_rate": tot["hits"] / lookups if lookups else None,
           "resident_MB_per_token": tot["bytes_resident"] / tokens / 1e6,
           "h2d_MB_per_token": tot["bytes_h2d"] / tokens / 1e6,
           "hbm_GBs_over_wall": tot["bytes_resident"] / (ms * 1e-3) / 1e9}
    if kt:
        ffn = kt.get("expert_ffn")
        if ffn and ffn[1] > 0:
            gbs = ffn[2] / (ffn[1] * 1e-3) / 1e9
            out["expert_ffn"] = {"GB_s": gbs, "frac": gbs / peaks["hbm_gbs"], "launches": ffn[0],
                                 "mean_us": 1000 * ffn[1] / ffn[0], "bytes_per_launch": ffn[2] / ffn[0]}
        out["kernels"] = _kernel_table(kt)
    return out


def ffn_replay_timing(layers, stream, rounds=4):
    """Duration of the decode FFN launch without the per-launch overhead of a
    pair of CUDA events (several microseconds on this part): each layer's last
    one-token resident launch is replayed back to back, layer after layer (each
    layer its own weights, so no launch finds them in L2), all enqueued by one
    library call, and one pair of events on the launching stream brackets
    `rounds` passes over the layers. Returns bytes per launch, microseconds per
    launch and GB/s."""
    import torch

    import expert_streaming_ffn_gb300 as moe

    torch.cuda.synchronize()
    rs = torch.cuda.Stream()  # a stream of its own: the launches wait on nothing else
    sptr = rs.cuda_stream
    moe.moe_layers_replay_resident(layers, 1, sptr)  # one untimed pass
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(rs)
    by = moe.moe_layers_replay_resident(layers, rounds, sptr)
    ev1.record(rs)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    n = rounds * len(layers)
    return {"launches": n, "bytes_per_launch": by / n, "us_per_launch": 1000.0 * ms / n,
            "GB_s": by / (ms * 1e-3) / 1e9}


def run_ours(args, world, rank, local):
    import torch

    import expert_streaming_ffn_gb300 as moe
    import synth

    wl = synth.WORKLOADS["decode_2816"]
    s = wl.shapes
    n_layers = args.layers or wl.n_layers
    # the oracle on every host core, forked before this process makes any GPU call
    cpu_par = None
    if rank == 0 and world == 1 and not args.no_cpu:
        try:
            cpu_par = oracle_all_cores(wl, args.cpu_seconds)
        except Exception as ex:  # noqa: BLE001 - the single-thread figure below still stands
            cpu_par = ex
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.load()
    steps_total = args.warmup + args.steps
    seed = wl.seed + 1000 * rank  # independent replicas
    peaks, peak_src = measured_peaks()

    ctx = moe.moe_ctx_create(local)
    stream = torch.cuda.current_stream(dev)
    rig = DecodeRig(ctx, dev, stream, wl, n_layers, wl.cache_slots, wl.policy, 1, steps_total, seed,
                    resident=args.resident, n_prime=args.prime_steps)
    slots = rig.slots
    e2e = None
    if not args.no_e2e:
        x_host = torch.from_numpy(rig.xs_np.view(np.int16)).view(torch.bfloat16).pin_memory()
        x_stage = torch.empty((n_layers, s.d_model), dtype=torch.bfloat16, device=dev)
        y_host = torch.empty((n_layers, s.d_model), dtype=torch.float32).pin_memory()
        sptr = stream.cuda_stream

        def e2e_step(st):
            x_stage.copy_(x_host[st].view(n_layers, s.d_model), non_blocking=True)
            for l in range(n_layers):
                zb = rig.zbs[l]
                moe.moe_forward_ptr(rig.layers[l], x_stage[l].data_ptr(), 1,
                                    zb.data_ptr() if zb is not None else None, rig.y_dev[l].data_ptr(), sptr)
            y_host.copy_(rig.y_dev.view(n_layers, s.d_model), non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
            return float(y_host[0, 0])

        # the same cache trajectory as the timed loop: primed caches, the
        # same warm-up steps, then the same timed steps
        rig.prime()
        for st in range(args.warmup):
            e2e_step(st)
        barrier(world)
        t0 = time.perf_counter()
        for st in range(args.warmup, steps_total):
            e2e_step(st)
        t_e2e = max_over_ranks(time.perf_counter() - t0, world)
        e2e = {"value": world * args.steps / t_e2e, "unit": "tok/s",
               "h2d_bytes_per_step": n_layers * s.d_model * 2, "d2h_bytes_per_step": n_layers * s.d_model * 4}
    rig.prime()
    barrier(world)
    with ClockSampler(gpu_bus_id(local)) as clocks:
        t_wall = time.perf_counter()
        ms, stats, _, launches = rig.run(args.warmup, args.steps)
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    ms_max = max_over_ranks(ms, world)
    tot = _totals(stats)

    # end to end through the public call with host buffers, measured first
    # (before the device-timed loop, next to it in time: the host link's speed
    # drifts over a run): per step, the step's x (all layers) host->device
    # from pinned memory, the 30 layer calls, and y device->host read back
    # same steps again, from the same cache state (primed caches, the same
    # warm-up), with per-kernel CUDA events on the launching stream; the
    # exposed copy time is measured in this pass too (it needs events)
    rig.prime()
    _, pstats, kt, _ = rig.run(args.warmup, args.steps, profile=True)
    exposed = sum(x["exposed_copy_us"] for x in pstats)
    # The roofline kernel: the one with the most device time among those whose
    # duration is HBM work. The decode launch over the experts copied in by
    # the call (expert_ffn_miss) waits for the host-to-device copies, so its
    # time is the host link's, reported beside the roofline instead.
    hbm_kinds = {k: v for k, v in kt.items() if k != "expert_ffn_miss" and v[0] > 0}
    dom = max(hbm_kinds.items(), key=lambda kv: kv[1][1])
    name, (n_l, tot_ms, by, fl) = dom
    single = {"GB_s": by / (tot_ms * 1e-3) / 1e9 if tot_ms > 0 else 0.0,
              "us_per_launch": 1000.0 * tot_ms / n_l if n_l else None,
              "bytes_per_launch": by / n_l if n_l else None,
              "how": "a pair of CUDA events around every launch in a replay of the timed steps"}
    replay = ffn_replay_timing(rig.layers, stream) if name == "expert_ffn" else None
    if replay:
        achieved, bpl = replay["GB_s"], replay["bytes_per_launch"]
    else:
        achieved, bpl = single["GB_s"], single["bytes_per_launch"]
    all_ms = sum(v[1] for v in kt.values())
    all_bytes = sum(v[2] for v in kt.values())

    # predictive prefetch into HBM (one spare expert buffer per layer): the
    # same steps from the same primed caches, so the hit rate is the same;
    # what can change is the exposed copy time
    prefetch = None
    if not args.resident and not args.no_legs:
        for h in rig.layers:
            moe.moe_layer_set_prefetch(h, True)
        rig.prime()
        ms_p, st_p, _, _ = rig.run(args.warmup, args.steps)
        rig.prime()
        pf0 = [moe.moe_layer_prefetch_stats(h) for h in rig.layers]
        _, pst_p, _, _ = rig.run(args.warmup, args.steps, profile=True)
        pf1 = [moe.moe_layer_prefetch_stats(h) for h in rig.layers]
        n_ls = rig.L * (args.warmup + args.steps)  # layer-steps of that pass
        pf_issued = sum(b["issued"] - a["issued"] for a, b in zip(pf0, pf1)) / n_ls
        pf_used = sum(b["used"] - a["used"] for a, b in zip(pf0, pf1)) / n_ls
        tp = _totals(st_p)
        for h in rig.layers:
            moe.moe_layer_set_prefetch(h, False)
        prefetch = {"spare_buffers_per_layer": 1,
                    "off": {"tok_s": world * args.steps / (ms_max * 1e-3), "hit_rate": tot["hits"] / max(1, tot["hits"] + tot["misses"]),
                            "exposed_copy_us_per_token": exposed / args.steps,
                            "h2d_MB_per_token": tot["bytes_h2d"] / args.steps / 1e6},
                    "on": {"tok_s": args.steps / (ms_p * 1e-3), "hit_rate": tp["hits"] / max(1, tp["hits"] + tp["misses"]),
                           "exposed_copy_us_per_token": sum(x["exposed_copy_us"] for x in pst_p) / args.steps,
                           "h2d_MB_per_token": tp["bytes_h2d"] / args.steps / 1e6,
                           "prefetches_per_layer_step": pf_issued,
                           "misses_served_from_hbm_per_layer_step": pf_used}}

    weights = rig.last_weights
    rig.close()

    extra = {}
    if not args.resident and world == 1 and not args.no_legs:
        extra["tiny_latency"] = run_tiny_latency(args, ctx, dev, stream, seed)
        extra["resident_upper_bound"] = run_resident_bound(args, ctx, dev, stream, seed, peaks, weights)
        extra["decode_2048"] = run_decode_2048(args, ctx, dev, stream, seed, peaks)
    prefill = None
    if not args.no_prefill and args.prefill_layers > 0:
        prefill = run_prefill(args, ctx, dev, stream, seed)

    storage = None
    if not args.no_storage and args.storage_layers > 0 and world == 1:
        try:
            storage = run_storage(args, ctx, dev, stream, seed)
            storage["pinned_pool_ms_per_layer_token"] = ms_max / args.steps / n_layers
        except Exception as ex:  # noqa: BLE001 - the leg reports its failure; the bench line stands
            storage = {"error": f"{type(ex).__name__}: {ex}"}
    if not args.no_stress and world == 1 and not args.resident and not args.no_legs:
        extra["stress"] = run_stress(args, ctx, dev, stream, seed, layers=args.stress_layers_line,
                                     steps=args.stress_steps_line)

    moe.moe_ctx_destroy(ctx)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        times = oracle_layer_tokens(64, args.cpu_seconds, wl)
        layer_s = statistics.mean(times)
        cpu_single = {"value": 1.0 / (layer_s * n_layers), "unit": "tok/s", "cores": 1, "kind": "oracle",
                  "sample": f"{len(times)} layer-tokens of decode_2816 (layers 0-1) single-threaded, "
                            f"extrapolated to {n_layers} layers per token"}
        if isinstance(cpu_par, tuple):
            rate, P = cpu_par
            cpu = {"value": rate / n_layers, "unit": "tok/s", "cores": P, "kind": "oracle",
                   "sample": f"{P} forked single-threaded copies of the oracle, each running whole layer-tokens "
                             f"of decode_2816 (layer 0) for {args.cpu_seconds:g} s; layer-tokens per second "
                             f"over all copies, divided by {n_layers} layers per token",
                   "single_thread": cpu_single}
        else:
            cpu = dict(cpu_single, all_cores_error=None if cpu_par is None else repr(cpu_par))

    if rank != 0:
        return
    tok_s = world * args.steps / (ms_max * 1e-3)
    lookups = tot["hits"] + tot["misses"]
    out = {
        "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded int4/int8 weights and N(0,1) RMS-normalised bf16 activations)",
        "config": workload_config(wl, n_layers, slots, world, resident=args.resident),
        "hit_rate": tot["hits"] / lookups if lookups else None,
        "h2d_MB_per_token": tot["bytes_h2d"] / args.steps / 1e6,
        "exposed_copy_us_per_token": exposed / args.steps,
        "host_wait_us_per_token": tot["host_wait_us"] / args.steps,
        "host_issue_us_per_token": tot["host_issue_us"] / args.steps,
        "resident_GB_per_token": tot["bytes_resident"] / args.steps / 1e9,
        "hbm_GBs_all_kernels": all_bytes / (all_ms * 1e-3) / 1e9 if all_ms else None,
        "roofline": {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(name, bpl),
                     "algorithmic_bytes_per_launch": bpl,
                     "timing": ("each layer's last resident launch replayed back to back, "
                                f"{replay['launches']} launches between one pair of CUDA events")
                     if replay else single["how"],
                     "replay": replay, "single_launch_events": single,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s"},
        "kernels": _kernel_table(kt),
        "miss_launches": ({"kernel": "expert_ffn_miss", "bound": "host link (copies of missed experts)",
                           "launches": kt["expert_ffn_miss"][0], "ms": round(kt["expert_ffn_miss"][1], 4)}
                          if kt.get("expert_ffn_miss", (0, 0))[1] > 0 else None),
        **extra,
        "hbm_prefetch": prefetch,
        "prefill": prefill,
        "storage": storage,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(out), flush=True)


def run_resident_bound(args, ctx, dev, stream, seed, peaks, weights=None):
    """decode_2816 with every expert resident (S = E): the upper bound of the
    decode layer with no host link in the way (the analogue of the pages'
    all-in-memory baseline). --resident-layers layers (their weights, 0.9 GB
    each, exceed L2 many times over), one token per step."""
    import synth

    wl = synth.WORKLOADS["decode_2816"]
    L = args.resident_layers
    warm, steps = 16, 64
    rig = DecodeRig(ctx, dev, stream, wl, L, wl.cache_slots, wl.policy, 1, warm + steps, seed, resident=True,
                    weights=weights)
    try:
        ms, stats, _, _ = rig.run(warm, steps)
        _, pstats, kt, _ = rig.run(warm, steps, profile=True)
        out = _leg_summary(rig, ms, stats, kt, steps, peaks)
        rep = ffn_replay_timing(rig.layers, stream)
        rep["frac"] = rep["GB_s"] / peaks["hbm_gbs"]
        out.update({"workload": "decode_2816, every expert resident", "layers": L, "steps": steps,
                    "tok_s_30_layers": out["tok_s"] * L / wl.n_layers, "expert_ffn_replay": rep})
        # the ordered combine (bit-identical repeats): the same steps, its cost per layer
        import expert_streaming_ffn_gb300 as moe

        for h in rig.layers:
            moe.moe_layer_set_deterministic(h, True)
        rig.run(warm, steps)  # allocates the partial rows
        ms_d, _, _, _ = rig.run(warm, steps)
        out["ordered_combine"] = {"tok_s": steps / (ms_d * 1e-3), "ms_per_layer_step": ms_d / steps / L,
                                  "extra_us_per_layer": 1000.0 * (ms_d - ms) / steps / L}
        return out
    finally:
        rig.close()


def run_tiny_latency(args, ctx, dev, stream, seed):
    """tiny (config 0): one layer of d = 512, 16 experts (top-2), 4-slot LFU,
    4 decode tokens per call, x ~ N(0, 1): latency per call, through the
    public call, device-timed over 256 consecutive calls (after 64 warm-up
    calls); the cache trajectory is that of the calls, misses included."""
    import torch

    import expert_streaming_ffn_gb300 as moe
    import synth

    wl = synth.WORKLOADS["tiny"]
    s = wl.shapes
    h = moe.moe_layer_create(ctx, s, wl.cache_slots, wl.policy)
    try:
        moe.moe_layer_set_weights(h, synth.layer_weights(s, 0, seed))
        n = 320
        xs = np.stack([synth.tokens(s, 0, st, wl.tokens, wl.rms_normalise, seed) for st in range(n)])
        x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
        y = torch.empty((wl.tokens, s.d_model), dtype=torch.float32, device=dev)
        row = wl.tokens * s.d_model * 2
        sptr = stream.cuda_stream

        def call(i):
            moe.moe_forward_ptr(h, x.data_ptr() + i * row, wl.tokens, None, y.data_ptr(), sptr)

        for i in range(64):
            call(i)
        torch.cuda.synchronize(dev)
        moe.moe_layer_reset_stats(h)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        t0 = time.perf_counter()
        for i in range(64, n):
            call(i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        st = moe.moe_layer_stats(h)
        calls = n - 64
        return {"workload": "tiny", "tokens_per_call": wl.tokens, "calls": calls,
                "us_per_call": 1000.0 * ev0.elapsed_time(ev1) / calls, "wall_us_per_call": 1e6 * wall / calls,
                "hit_rate": st["hits"] / max(1, st["hits"] + st["misses"]),
                "host_wait_us_per_call": st["host_wait_us"] / calls}
    finally:
        moe.moe_layer_destroy(h)


def run_decode_2048(args, ctx, dev, stream, seed, peaks):
    """decode_2048: 40 layers (--layers-2048), SiLU, 64 slots, Zipf(0.9),
    batches 1 and 8, under LFU and under LRU. 256 decode steps per run, the
    first 64 as warm-up, after a priming pass."""
    import synth

    wl = synth.WORKLOADS["decode_2048"]
    L = args.layers_2048
    warm, steps = 64, 192
    runs = []
    weights = None
    for policy, pname in ((0, "LFU"), (1, "LRU")):
        for T in (1, 8):
            rig = DecodeRig(ctx, dev, stream, wl.with_(tokens=T, policy=policy), L, wl.cache_slots, policy, T,
                            warm + steps, seed, weights=weights, n_prime=16)
            try:
                # the host link out of its slow start, then the workload's 256
                # steps from empty caches: the first 64 warm them
                rig.prime(seconds=0.5)
                rig.reset()
                ms, stats, _, _ = rig.run(warm, steps)
                rig.reset()
                _, pstats, kt, _ = rig.run(warm, steps, profile=True)
                out = _leg_summary(rig, ms, stats, kt, steps, peaks)
                out["exposed_copy_us_per_token"] = sum(x["exposed_copy_us"] for x in pstats) / (steps * T)
                out.update({"policy": pname, "batch": T})
                runs.append(out)
                weights = rig.last_weights
            finally:
                rig.close()
    return {"workload": "decode_2048", "layers": L, "steps": steps, "warmup": warm, "slots": wl.cache_slots,
            "runs": runs}


def _prefill_pass(ctx, dev, stream, layers, xs, y, prompt=False):
    """One pass of every layer's prompt (8 chunks of 128, or one layer-major
    call with prompt=True) with per-kernel events."""
    import torch

    import expert_streaming_ffn_gb300 as moe

    moe.moe_ctx_set_profiling(ctx, True)
    moe.moe_ctx_reset_kernel_times(ctx)
    for h in layers:
        moe.moe_layer_reset_stats(h)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for h, x in zip(layers, xs):
        if prompt:
            moe.moe_forward_prompt(h, x, y=y)
        else:
            moe.moe_forward(h, x, y=y)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    kt = moe.moe_ctx_kernel_times(ctx)
    moe.moe_ctx_set_profiling(ctx, False)
    return ev0.elapsed_time(ev1), kt, [moe.moe_layer_stats(h) for h in layers]


def _gemm_summary(kt, peaks):
    out = {}
    for k in ("gemm_gateup", "gemm_down"):
        n, ms, by, fl = kt[k]
        if n == 0 or ms <= 0:
            continue
        tf = fl / (ms * 1e-3) / 1e12
        gbs = by / (ms * 1e-3) / 1e9
        out[k] = {"launches": n, "ms": round(ms, 4), "TFLOPs": round(tf, 2), "GB_s": round(gbs, 1),
                  "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                  "frac_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)}
    return out


def run_prefill(args, ctx, dev, stream, seed):
    """prefill_2816: a 1024-token prompt as 8 chunks of 128 tokens per layer.

    Four runs: (1) streaming, as configured (16-slot LFU, misses copied from
    pinned host memory); (2) all-resident (256 slots, prompt run once to fill
    the slots, then timed), which times the grouped GEMMs on weights already in
    HBM; (3) the shared-expert GEMM alone (a layer of the same d and shared
    expert with a single 64-wide routed expert), the dense contraction the
    tensor-core roofline applies to; (4) `layer_major`: the whole prompt in one
    moe_forward_prompt call per layer (one routing, one cache step, ~32 token
    rows per routed expert), streaming and all-resident."""
    import torch

    import expert_streaming_ffn_gb300 as moe
    import synth

    wl = synth.WORKLOADS["prefill_2816"]
    s = wl.shapes
    P = args.prefill_layers
    prompt = wl.tokens * wl.steps  # 1024
    peaks, _ = measured_peaks()
    y = torch.empty((prompt, s.d_model), dtype=torch.float32, device=dev)
    xs = [torch.from_numpy(synth.tokens(s, l, 0, prompt, wl.rms_normalise, seed).view(np.int16))
          .view(torch.bfloat16).to(dev) for l in range(P)]

    def make(shapes, slots, l, w):
        w = synth.layer_weights(shapes, l, seed, reuse=w)
        h = moe.moe_layer_create(ctx, shapes, slots, wl.policy)
        moe.moe_layer_set_weights(h, w)
        return h, w

    # (1) streaming
    layers, w = [], None
    if args.prefill_resident_only:
        P = 0
    for l in range(P):
        h, w = make(s, wl.cache_slots, l, w)
        layers.append(h)
    if P:
        moe.moe_forward(layers[0], xs[0][:128], y=y[:128])  # load the kernels
        torch.cuda.synchronize(dev)
        moe.moe_layer_destroy(layers[0])  # a fresh cache for the timed pass
        layers[0], w = make(s, wl.cache_slots, 0, w)
    ms, kt, stats = _prefill_pass(ctx, dev, stream, layers, xs, y) if P else (0.0, moe.moe_ctx_kernel_times(ctx), [])
    for h in layers:
        moe.moe_layer_destroy(h)
    kinds = ("gemm_gateup", "gemm_down", "pf_gather", "combine", "router")
    kms = sum(kt[k][1] for k in ("gemm_gateup", "gemm_down"))
    fl = sum(kt[k][3] for k in ("gemm_gateup", "gemm_down"))
    hits = sum(x["hits"] for x in stats)
    misses = sum(x["misses"] for x in stats)
    out = {
        "workload": "prefill_2816", "layers_measured": P, "prompt_tokens": prompt, "chunk": wl.tokens,
        "tok_s_per_layer": prompt * P / (ms * 1e-3) if P else None,
        "tok_s_30_layers": prompt / (ms * 1e-3 / P * 30) if P else None,
        "expert_TFLOPs": fl / (kms * 1e-3) / 1e12 if kms else None,
        "expert_kernel_ms": kms, "wall_ms": ms,
        "hit_rate": hits / (hits + misses) if hits + misses else None,
        "h2d_GB": sum(x["bytes_h2d"] for x in stats) / 1e9,
        "exposed_copy_ms": sum(x["exposed_copy_us"] for x in stats) / 1e3,
        "kernels": {k: {"launches": kt[k][0], "ms": round(kt[k][1], 3)} for k in kinds if kt[k][0] > 0},
    }

    # (2) all-resident: 256 slots, filled by a first pass
    h, w = make(s, s.n_experts, 0, w)
    _prefill_pass(ctx, dev, stream, [h], xs[:1], y)
    ms2, kt2, st2 = _prefill_pass(ctx, dev, stream, [h], xs[:1], y)
    moe.moe_layer_destroy(h)
    out["all_resident"] = {"tok_s_per_layer": prompt / (ms2 * 1e-3), "wall_ms": ms2,
                           "hit_rate": st2[0]["hits"] / max(1, st2[0]["hits"] + st2[0]["misses"]),
                           "kernels": _gemm_summary(kt2, peaks)}

    # (4) layer-major: the same prompt through moe_forward_prompt (one routing,
    # one cache step and one grouped GEMM pair per layer), streaming from a
    # fresh 16-slot cache and with every expert resident
    lm = {}
    for name, slots in (("streaming", wl.cache_slots), ("all_resident", s.n_experts)):
        h, w = make(s, slots, 0, w)
        if slots == s.n_experts:
            moe.moe_cache_step(h, np.arange(s.n_experts))
        moe.moe_forward_prompt(h, xs[0], y=y)  # loads the kernels, fills the resident slots
        torch.cuda.synchronize(dev)
        if slots != s.n_experts:
            moe.moe_layer_destroy(h)
            h, w = make(s, slots, 0, w)
        # all resident: the mean of 3 calls (the same work each time); streaming:
        # one call on the fresh cache (a repeat would find it warm)
        reps = 3 if slots == s.n_experts else 1
        ms4, kt4, st4 = _prefill_pass(ctx, dev, stream, [h] * reps, xs[:1] * reps, y, prompt=True)
        moe.moe_layer_destroy(h)
        ms4 /= reps
        kms4 = sum(kt4[k][1] for k in ("gemm_gateup", "gemm_down"))
        fl4 = sum(kt4[k][3] for k in ("gemm_gateup", "gemm_down"))
        lm[name] = {"tok_s_per_layer": prompt / (ms4 * 1e-3), "wall_ms": ms4, "calls": reps,
                    "expert_TFLOPs": fl4 / (kms4 * 1e-3) / 1e12 if kms4 else None,
                    "h2d_GB": st4[-1]["bytes_h2d"] / reps / 1e9,
                    "exposed_copy_ms": st4[-1]["exposed_copy_us"] / reps / 1e3,
                    "kernels": _gemm_summary(kt4, peaks)}
    out["layer_major"] = lm
    # (5) a 4096-token prompt in one layer-major call, every expert resident:
    # ~128 token rows per routed expert, so the grouped GEMM's MMAs are full
    # width (the large-chunk case the tensor-core roofline applies to)
    try:
        big = 4096
        xb = torch.from_numpy(synth.tokens(s, 0, 1, big, wl.rms_normalise, seed).view(np.int16)).view(
            torch.bfloat16).to(dev)
        yb = torch.empty((big, s.d_model), dtype=torch.float32, device=dev)
        h, w = make(s, s.n_experts, 0, w)
        moe.moe_cache_step(h, np.arange(s.n_experts))
        moe.moe_forward_prompt(h, xb, y=yb)  # loads the kernels, fills the resident slots
        torch.cuda.synchronize(dev)
        reps = 3
        ms5, kt5, _ = _prefill_pass(ctx, dev, stream, [h] * reps, [xb] * reps, yb, prompt=True)
        moe.moe_layer_destroy(h)
        ms5 /= reps
        kms5 = sum(kt5[k][1] for k in ("gemm_gateup", "gemm_down"))
        fl5 = sum(kt5[k][3] for k in ("gemm_gateup", "gemm_down"))
        out["prompt_4096"] = {"tokens": big, "calls": reps, "wall_ms": ms5, "tok_s_per_layer": big / (ms5 * 1e-3),
                              "expert_TFLOPs": fl5 / (kms5 * 1e-3) / 1e12 if kms5 else None,
                              "kernels": _gemm_summary(kt5, peaks)}
    except Exception as ex:  # noqa: BLE001 - the leg reports its failure; the bench line stands
        out["prompt_4096"] = {"error": f"{type(ex).__name__}: {ex}"}

    # (3) the shared-expert GEMM: 128 x 2816 x 2816 (gate, up) and 128 x 2816 x 2816 (down) per chunk
    s3 = synth.Shapes(s.d_model, 1, 1, 64, s.d_ff_shared, s.act)
    h, _ = make(s3, 1, 0, None)
    _prefill_pass(ctx, dev, stream, [h], xs[:1], y)
    ms3, kt3, _ = _prefill_pass(ctx, dev, stream, [h], xs[:1], y)
    moe.moe_layer_destroy(h)
    out["shared_gemm"] = {"shape": f"{prompt}x{s.d_model}x{s.d_ff_shared} in chunks of {wl.tokens}",
                          "wall_ms": ms3, "kernels": _gemm_summary(kt3, peaks)}
    return out


def _fs_type(path: str) -> str | None:
    """File system type of the mount holding path (from /proc/mounts)."""
    try:
        path = os.path.realpath(path)
        best, typ = "", None
        with open("/proc/mounts") as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and (path == parts[1] or path.startswith(parts[1].rstrip("/") + "/")) \
                        and len(parts[1]) >= len(best):
                    best, typ = parts[1], parts[2]
        return typ
    except OSError:
        return None


def run_storage(args, ctx, dev, stream, seed):
    """decode_2816 with the routed experts streamed from expert files.

    The storage tier in place of the pinned pool: one expert file per layer
    (moe_store_write), each layer's misses read by reader threads (O_DIRECT
    where the file system allows it) into a host tier of
    --storage-host-slots experts, then copied to the layer's 16 HBM slots.
    --storage-layers layers, one token per step, Zipf(1.1) routing as in the
    decode bench. Three runs from fresh stores and caches: `demand` (reads
    only when a miss needs them, one pread per expert), `demand_1MiB_pieces`
    (the same, each expert read as 1 MiB pieces spread over the readers) and
    `readahead` (before each layer, the next layer's --storage-readahead
    most-routed experts that are in neither its slots nor its tier are read
    ahead)."""
    import shutil
    import tempfile
    import types

    import torch

    import expert_streaming_ffn_gb300 as moe
    import synth

    wl = synth.WORKLOADS["decode_2816"]
    s = wl.shapes
    L = args.storage_layers
    H = args.storage_host_slots
    steps = args.storage_warmup + args.storage_steps
    root = tempfile.mkdtemp(prefix="moe_store_", dir=args.storage_dir)
    out = {"workload": "decode_2816 streamed from expert files", "layers": L, "cache_slots": wl.cache_slots,
           "host_slots": H, "readers": args.storage_readers, "steps": args.storage_steps,
           "warmup": args.storage_warmup, "file_system": _fs_type(root)}
    try:
        t0 = time.perf_counter()
        paths, w = [], None
        for l in range(L):
            w = synth.layer_weights(s, l, seed, reuse=w)
            paths.append(os.path.join(root, f"layer{l}.experts"))
            moe.moe_store_write(paths[-1], s, w)
        del w
        out["write_s"] = time.perf_counter() - t0
        out["file_GB"] = sum(os.path.getsize(p) for p in paths) / 1e9
        zbs = [torch.from_numpy(synth.zipf_bias(s, l, wl.zipf_s, wl.zipf_beta, seed)).to(dev) for l in range(L)]
        xs_np = np.empty((steps, L, s.d_model), np.uint16)
        for st in range(steps):
            for l in range(L):
                xs_np[st, l] = synth.tokens(s, l, st, 1, wl.rms_normalise, seed)[0]
        x_dev = torch.from_numpy(xs_np.view(np.int16)).view(torch.bfloat16).to(dev)
        y_dev = torch.empty((L, s.d_model), dtype=torch.float32, device=dev)
        row = s.d_model * 2
        sptr = stream.cuda_stream
        for mode, pf, chunk in (("demand", 0, 0), ("demand_1MiB_pieces", 0, 1 << 20),
                                ("readahead", args.storage_readahead, 0)):
            stores, layers = [], []
            for l in range(L):
                stores.append(moe.moe_store_open(paths[l], s, H, args.storage_readers, moe.MOE_STORE_DIRECT))
                moe.moe_store_set_read_chunk(stores[-1], chunk)
                layers.append(moe.moe_layer_create_streamed(ctx, s, wl.cache_slots, stores[-1], wl.policy))
                resident = types.SimpleNamespace(router=synth.router_weights(s, l, seed),
                                                 shared=synth.ffn_weights(s, l, 0, seed, shared=True))
                moe.moe_layer_set_weights(layers[-1], resident, routed=False)

            def step(st):
                base = x_dev.data_ptr() + st * L * row
                for l in range(L):
                    if pf:
                        moe.moe_layer_prefetch(layers[(l + 1) % L], pf)
                    moe.moe_forward_ptr(layers[l], base + l * row, 1, zbs[l].data_ptr(), y_dev[l].data_ptr(),
                                        sptr)

            for st in range(args.storage_warmup):
                step(st)
            torch.cuda.synchronize(dev)
            for h, sto in zip(layers, stores):
                moe.moe_layer_reset_stats(h)
                moe.moe_store_reset_stats(sto)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t_wall = time.perf_counter()
            ev0.record(stream)
            for st in range(args.storage_warmup, steps):
                step(st)
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            t_wall = time.perf_counter() - t_wall
            ms = ev0.elapsed_time(ev1)
            ls = [moe.moe_layer_stats(h) for h in layers]
            ss = [moe.moe_store_get_stats(x) for x in stores]
            for h in layers:
                moe.moe_layer_destroy(h)
            for x in stores:
                moe.moe_store_close(x)
            K = args.storage_steps
            hits = sum(x["hits"] for x in ls)
            misses = sum(x["misses"] for x in ls)
            tot = {k: sum(x[k] for x in ss) for k in ("fetches", "tier_hits", "reads", "prefetch_reads",
                                                       "prefetch_used", "bytes_read", "read_errors")}
            read_us = sum(x["read_us"] for x in ss)
            wait_us = sum(x["wait_us"] for x in ss)
            out[mode] = {
                "tok_s": K / (ms * 1e-3), "ms_per_layer_token": ms / K / L,
                "hbm_hit_rate": hits / (hits + misses) if hits + misses else None,
                "tier_hit_rate": tot["tier_hits"] / tot["fetches"] if tot["fetches"] else None,
                "reads_per_token": tot["reads"] / K, "read_MB_per_token": tot["bytes_read"] / K / 1e6,
                "read_GBs": tot["bytes_read"] / t_wall / 1e9,
                "mean_read_ms": read_us / tot["reads"] / 1e3 if tot["reads"] else None,
                "fetch_wait_ms_per_token": wait_us / K / 1e3,
                "prefetch_reads": tot["prefetch_reads"], "prefetch_used": tot["prefetch_used"],
                "read_errors": tot["read_errors"], "direct_io": bool(ss[0]["direct"]),
            }
    finally:
        shutil.rmtree(root, ignore_errors=True)
    return out


def run_stress(args, ctx, dev, stream, seed, layers=None, steps=None):
    """stress_2816: the 2816 shapes with uniform routing (no bias), decode
    batches of 1, 4, 16 and 64 tokens against caches of 8, 16 and 64 slots
    per layer, and a 4096-token prompt in chunks of 128 per cache size.
    --stress-layers layers (the workload names 48; each holds an 856 MB
    pinned pool), fresh caches per point, --stress-steps timed steps after as
    many warm-up steps. Per point: tokens/s, weight bytes the kernels read
    from HBM and bytes copied host-to-device per token, the hit rate, and the
    exposed copy time per token (the miss launches' wait for their copies,
    from a second, event-timed pass over the same steps)."""
    import torch

    import expert_streaming_ffn_gb300 as moe
    import synth

    wl = synth.WORKLOADS["stress_2816"]
    s = wl.shapes
    L = layers or args.stress_layers
    K = steps or args.stress_steps
    ws, w = [], None
    for l in range(L):
        w = synth.layer_weights(s, l, seed, reuse=None)
        ws.append(w)
    sptr = stream.cuda_stream
    row = s.d_model * 2
    points = []
    for S in (8, 16, 64):
        layers = []
        for l in range(L):
            h = moe.moe_layer_create(ctx, s, S, wl.policy)
            moe.moe_layer_set_weights(h, ws[l])
            layers.append(h)
        for T in (1, 4, 16, 64):
            xs_np = np.empty((2 * K, L, T, s.d_model), np.uint16)
            for st in range(2 * K):
                for l in range(L):
                    xs_np[st, l] = synth.tokens(s, l, 1000 * T + st, T, wl.rms_normalise, seed)
            x_dev = torch.from_numpy(xs_np.view(np.int16)).view(torch.bfloat16).to(dev)
            y_dev = torch.empty((L, T, s.d_model), dtype=torch.float32, device=dev)

            def step(st):
                base = x_dev.data_ptr() + st * L * T * row
                for l in range(L):
                    moe.moe_forward_ptr(layers[l], base + l * T * row, T, None, y_dev[l].data_ptr(), sptr)

            def run(profile):
                for h in layers:
                    moe.moe_cache_reset(h)
                for st in range(K):
                    step(st)
                torch.cuda.synchronize(dev)
                for h in layers:
                    moe.moe_layer_reset_stats(h)
                moe.moe_ctx_set_profiling(ctx, profile)
                ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ev0.record(stream)
                for st in range(K, 2 * K):
                    step(st)
                ev1.record(stream)
                torch.cuda.synchronize(dev)
                moe.moe_ctx_set_profiling(ctx, False)
                return ev0.elapsed_time(ev1), [moe.moe_layer_stats(h) for h in layers]

            ms, stats = run(False)
            _, pstats = run(True)
            tokens = K * T
            hits = sum(x["hits"] for x in stats)
            misses = sum(x["misses"] for x in stats)
            points.append({
                "slots": S, "batch": T, "tok_s": tokens / (ms * 1e-3), "ms_per_layer_step": ms / K / L,
                "hit_rate": hits / (hits + misses) if hits + misses else None,
                "bypass_per_layer_step": sum(x["bypass"] for x in stats) / K / L,
                "hbm_MB_per_token": sum(x["bytes_resident"] for x in stats) / tokens / 1e6,
                "h2d_MB_per_token": sum(x["bytes_h2d"] for x in stats) / tokens / 1e6,
                "exposed_copy_us_per_token": sum(x["exposed_copy_us"] for x in pstats) / tokens,
            })
            del x_dev, y_dev
        # the 4096-token prompt in chunks of 128, from a fresh cache
        P = 4096
        x = torch.from_numpy(synth.tokens(s, 0, 7, P, wl.rms_normalise, seed).view(np.int16)) \
            .view(torch.bfloat16).to(dev)
        y = torch.empty((P, s.d_model), dtype=torch.float32, device=dev)
        moe.moe_cache_reset(layers[0])
        moe.moe_layer_reset_stats(layers[0])
        ms, _, st = _prefill_pass(ctx, dev, stream, layers[:1], [x], y)
        st = st[0]
        points.append({
            "slots": S, "prefill_tokens": P, "tok_s": P / (ms * 1e-3), "ms_per_layer": ms,
            "hit_rate": st["hits"] / max(1, st["hits"] + st["misses"]),
            "hbm_MB_per_token": st["bytes_resident"] / P / 1e6, "h2d_MB_per_token": st["bytes_h2d"] / P / 1e6,
            "exposed_copy_us_per_token": st["exposed_copy_us"] / P,
        })
        for h in layers:
            moe.moe_layer_destroy(h)
    return {"workload": "stress_2816", "layers": L, "steps": K, "points": points}


def main():
    args = parse()
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.prefill_only:
        import torch

        import expert_streaming_ffn_gb300 as moe

        torch.cuda.set_device(local)
        moe.load()
        ctx = moe.moe_ctx_create(local)
        out = run_prefill(args, ctx, torch.device("cuda", local), torch.cuda.current_stream(), 1000 * rank)
        moe.moe_ctx_destroy(ctx)
        if rank == 0:
            print(json.dumps({"prefill": out}), flush=True)
    elif args.stress:
        import torch

        import expert_streaming_ffn_gb300 as moe

        torch.cuda.set_device(local)
        moe.load()
        ctx = moe.moe_ctx_create(local)
        out = run_stress(args, ctx, torch.device("cuda", local), torch.cuda.current_stream(), 1000 * rank)
        moe.moe_ctx_destroy(ctx)
        if rank == 0:
            print(json.dumps({"stress": out}), flush=True)
    elif args.storage_only:
        import torch

        import expert_streaming_ffn_gb300 as moe

        torch.cuda.set_device(local)
        moe.load()
        ctx = moe.moe_ctx_create(local)
        out = run_storage(args, ctx, torch.device("cuda", local), torch.cuda.current_stream(), 1000 * rank)
        moe.moe_ctx_destroy(ctx)
        if rank == 0:
            print(json.dumps({"storage": out}), flush=True)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
