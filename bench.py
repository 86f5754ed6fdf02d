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
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=256)
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


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores (one
    forked single-threaded copy per core, as cpu_baseline)."""
    import synth

    if rank != 0:
        return
    wl = synth.WORKLOADS["decode_2816"]
    n_layers = args.layers or wl.n_layers
    warm = oracle_layer_tokens(1, 0.0, wl, layers=(0,)) if args.warmup > 0 else []
    seconds = float(min(60, max(10, args.steps)))
    rate, P = oracle_all_cores(wl, seconds)  # layer-tokens per second over P cores
    tok_s = rate / n_layers
    sample = (f"{P} forked single-threaded copies of the oracle, each running whole layer-tokens of decode_2816 "
              f"(layer 0) for {seconds:g} s; layer-tokens per second over all copies, divided by {n_layers} "
              f"layers per token")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": int(rate * seconds), "warmup": len(warm), "ms_per_step": 1000.0 / tok_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": "decode_2816", "layers": n_layers, "tokens_per_step": 1,
                                        "cache_slots": 16, "policy": "LFU", "zipf_s": 1.1},
        "cpu_baseline": {"value": tok_s, "unit": "tok/s", "cores": P, "kind": "oracle", "sample": sample},
        "e2e": {"value": tok_s, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# our arm


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

    ctx = moe.moe_ctx_create(local)
    layers, zbs = [], []
    w = None
    slots = s.n_experts if args.resident else wl.cache_slots
    for l in range(n_layers):
        w = synth.layer_weights(s, l, seed, reuse=w)
        h = moe.moe_layer_create(ctx, s, slots, wl.policy)
        moe.moe_layer_set_weights(h, w)
        if args.resident:
            moe.moe_cache_step(h, np.arange(s.n_experts))  # copies every expert into its slot
        layers.append(h)
        zbs.append(torch.from_numpy(synth.zipf_bias(s, l, wl.zipf_s, wl.zipf_beta, seed)).to(dev))
    # inputs resident in HBM: x[step][layer][d] bf16, drawn per (step, layer)
    xs_np = np.empty((steps_total, n_layers, s.d_model), np.uint16)
    for st in range(steps_total):
        for l in range(n_layers):
            xs_np[st, l] = synth.tokens(s, l, st, 1, wl.rms_normalise, seed)[0]
    x_dev = torch.from_numpy(xs_np.view(np.int16)).view(torch.bfloat16).to(dev)
    y_dev = torch.empty((n_layers, s.d_model), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    row = s.d_model * 2

    def reset_caches():
        # empty caches (the cache trajectory starts again), or with --resident
        # every expert copied back in
        for h in layers:
            moe.moe_cache_reset(h)
            if args.resident:
                moe.moe_cache_step(h, np.arange(s.n_experts))

    def step(st):
        base = x_dev.data_ptr() + st * n_layers * row
        for l in range(n_layers):
            moe.moe_forward_ptr(layers[l], base + l * row, 1, zbs[l].data_ptr(), y_dev[l].data_ptr(), sptr)

    for st in range(args.warmup):
        step(st)
    torch.cuda.synchronize(dev)
    for h in layers:
        moe.moe_layer_reset_stats(h)
    launches0 = moe.moe_ctx_launches(ctx)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_bus_id(local)) as clocks:
        t_wall = time.perf_counter()
        ev0.record(stream)
        for st in range(args.warmup, steps_total):
            step(st)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    launches = moe.moe_ctx_launches(ctx) - launches0
    ms_max = max_over_ranks(ms, world)
    stats = [moe.moe_layer_stats(h) for h in layers]
    hits = sum(x["hits"] for x in stats)
    misses = sum(x["misses"] for x in stats)
    h2d = sum(x["bytes_h2d"] for x in stats)
    resident = sum(x["bytes_resident"] for x in stats)
    host_wait = sum(x["host_wait_us"] for x in stats)
    host_issue = sum(x["host_issue_us"] for x in stats)

    # same steps again, from the same cache state (empty caches, the same
    # warm-up), with per-kernel CUDA events on the launching stream; the
    # exposed copy time is measured in this pass too (it needs events)
    reset_caches()
    for st in range(args.warmup):
        step(st)
    torch.cuda.synchronize(dev)
    for h in layers:
        moe.moe_layer_reset_stats(h)
    moe.moe_ctx_set_profiling(ctx, True)
    moe.moe_ctx_reset_kernel_times(ctx)
    for st in range(args.warmup, steps_total):
        step(st)
    torch.cuda.synchronize(dev)
    kt = moe.moe_ctx_kernel_times(ctx)
    moe.moe_ctx_set_profiling(ctx, False)
    exposed = sum(moe.moe_layer_stats(h)["exposed_copy_us"] for h in layers)
    peaks, peak_src = measured_peaks()
    # The roofline kernel: the one with the most device time among those whose
    # duration is HBM work. The decode launch over the experts copied in by
    # the call (expert_ffn_miss) waits for the host-to-device copies, so its
    # time is the host link's, reported beside the roofline instead.
    hbm_kinds = {k: v for k, v in kt.items() if k != "expert_ffn_miss" and v[0] > 0}
    dom = max(hbm_kinds.items(), key=lambda kv: kv[1][1])
    name, (n_l, tot_ms, by, fl) = dom
    achieved = by / (tot_ms * 1e-3) / 1e9 if tot_ms > 0 else 0.0
    all_ms = sum(v[1] for v in kt.values())
    all_bytes = sum(v[2] for v in kt.values())
    kernels = {k: {"launches": v[0], "ms": round(v[1], 4), "share": round(v[1] / all_ms, 4) if all_ms else 0,
                   "GB_s": round(v[2] / (v[1] * 1e-3) / 1e9, 1) if v[1] > 0 else None}
               for k, v in kt.items() if v[0] > 0}

    # end to end through the public call with host buffers: per step, the
    # step's x (all layers) host->device from pinned memory, the 30 layer
    # calls, and y device->host read back
    e2e = None
    if not args.no_e2e:
        x_host = torch.from_numpy(xs_np.view(np.int16)).view(torch.bfloat16).pin_memory()
        x_stage = torch.empty((n_layers, s.d_model), dtype=torch.bfloat16, device=dev)
        y_host = torch.empty((n_layers, s.d_model), dtype=torch.float32).pin_memory()

        def e2e_step(st):
            x_stage.copy_(x_host[st], non_blocking=True)
            for l in range(n_layers):
                moe.moe_forward_ptr(layers[l], x_stage[l].data_ptr(), 1, zbs[l].data_ptr(), y_dev[l].data_ptr(), sptr)
            y_host.copy_(y_dev, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
            return float(y_host[0, 0])

        # the same cache trajectory as the timed loop: empty caches, the same
        # warm-up steps, then the same timed steps
        reset_caches()
        for st in range(args.warmup):
            e2e_step(st)
        barrier(world)
        t0 = time.perf_counter()
        for st in range(args.warmup, steps_total):
            e2e_step(st)
        t_e2e = max_over_ranks(time.perf_counter() - t0, world)
        e2e = {"value": world * args.steps / t_e2e, "unit": "tok/s",
               "h2d_bytes_per_step": n_layers * s.d_model * 2, "d2h_bytes_per_step": n_layers * s.d_model * 4}

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

    for h in layers:
        moe.moe_layer_destroy(h)
    moe.moe_ctx_destroy(ctx)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        times = oracle_layer_tokens(64, args.cpu_seconds, wl)
        layer_s = statistics.mean(times)
        single = {"value": 1.0 / (layer_s * n_layers), "unit": "tok/s", "cores": 1, "kind": "oracle",
                  "sample": f"{len(times)} layer-tokens of decode_2816 (layers 0-1) single-threaded, "
                            f"extrapolated to {n_layers} layers per token"}
        if isinstance(cpu_par, tuple):
            rate, P = cpu_par
            cpu = {"value": rate / n_layers, "unit": "tok/s", "cores": P, "kind": "oracle",
                   "sample": f"{P} forked single-threaded copies of the oracle, each running whole layer-tokens "
                             f"of decode_2816 (layer 0) for {args.cpu_seconds:g} s; layer-tokens per second "
                             f"over all copies, divided by {n_layers} layers per token",
                   "single_thread": single}
        else:
            cpu = dict(single, all_cores_error=None if cpu_par is None else repr(cpu_par))

    if rank != 0:
        return
    tok_s = world * args.steps / (ms_max * 1e-3)
    lookups = hits + misses
    out = {
        "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded int4/int8 weights and N(0,1) RMS-normalised bf16 activations)",
        "config": {"workload": "decode_2816" + (" (every expert resident)" if args.resident else ""),
                   "layers": n_layers, "tokens_per_step": 1, "d_model": s.d_model,
                   "experts": s.n_experts, "top_k": s.top_k, "d_ff": s.d_ff, "d_ff_shared": s.d_ff_shared,
                   "cache_slots": slots, "policy": "LFU", "zipf_s": wl.zipf_s,
                   "l2": f"inputs larger than L2: {resident / args.steps / 1e9:.2f} GB of weights read per step "
                         f"vs {L2_BYTES / 2**20:.0f} MiB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hit_rate": hits / lookups if lookups else None,
        "h2d_MB_per_token": h2d / args.steps / 1e6,
        "exposed_copy_us_per_token": exposed / args.steps,
        "host_wait_us_per_token": host_wait / args.steps,
        "host_issue_us_per_token": host_issue / args.steps,
        "resident_GB_per_token": resident / args.steps / 1e9,
        "hbm_GBs_all_kernels": all_bytes / (all_ms * 1e-3) / 1e9 if all_ms else None,
        "roofline": {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(name, by / n_l if n_l else None),
                     "algorithmic_bytes_per_launch": by / n_l if n_l else None,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s"},
        "kernels": kernels,
        "miss_launches": ({"kernel": "expert_ffn_miss", "bound": "host link (copies of missed experts)",
                           "launches": kt["expert_ffn_miss"][0], "ms": round(kt["expert_ffn_miss"][1], 4)}
                          if kt.get("expert_ffn_miss", (0, 0))[1] > 0 else None),
        "prefill": prefill,
        "storage": storage,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
    }
    print(json.dumps(out), flush=True)


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
        ms4, kt4, st4 = _prefill_pass(ctx, dev, stream, [h], xs[:1], y, prompt=True)
        moe.moe_layer_destroy(h)
        kms4 = sum(kt4[k][1] for k in ("gemm_gateup", "gemm_down"))
        fl4 = sum(kt4[k][3] for k in ("gemm_gateup", "gemm_down"))
        lm[name] = {"tok_s_per_layer": prompt / (ms4 * 1e-3), "wall_ms": ms4,
                    "expert_TFLOPs": fl4 / (kms4 * 1e-3) / 1e12 if kms4 else None,
                    "h2d_GB": st4[0]["bytes_h2d"] / 1e9,
                    "exposed_copy_ms": st4[0]["exposed_copy_us"] / 1e3,
                    "kernels": _gemm_summary(kt4, peaks)}
    out["layer_major"] = lm

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


def run_stress(args, ctx, dev, stream, seed):
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
    L = args.stress_layers
    K = args.stress_steps
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
