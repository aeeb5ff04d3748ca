#!/usr/bin/env python
"""Benchmark of the int4 routed-expert MoE layer on GB300.

A step is one pass of the whole hot path over one batch. For the default
workload (Qwen3-Next-80B-A3B-shaped decode: H=2048, 10 of 512 experts, T=1,
a stack of 48 independent layers, slot table a random permutation) a step is
one moe_decode_stack launch (router, top-k, experts and the weighted combine
of all 48 layers, residual chained), captured in a CUDA graph and replayed.

Prints one JSON line. value = MoE-layer tokens/s = T * layers * steps / time
(whole job: summed over ranks). The expert pool (43.5 GB at this shape) is far
larger than the 129 MB L2 and each step streams 934 MB of distinct expert
blobs, so no L2 flush is needed between steps. After the headline the other
target configurations (--extra: T=8192 prefill, Zipf-skewed T=64, 35B-shaped
decode, 8-bit experts, and the 80B Gated DeltaNet recurrence step) are
measured the same way and reported under "configs" in the same line; a
configuration whose distinct blobs fit twice in L2 is timed step by step with
a 256 MB write between steps.

--impl reference times the CPU oracle (oracle/, one thread) on the same
workload and metric, each step one layer for one token.
"""
from __future__ import annotations

import argparse
import ctypes as C
import dataclasses
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DECODE_SOURCES = ["int4_routed_expert_router_gb300/csrc/decode.cu",
                  "int4_routed_expert_router_gb300/csrc/decode_common.cuh",
                  "int4_routed_expert_router_gb300/csrc/smoe_dev.cuh",
                  "int4_routed_expert_router_gb300/csrc/smoe_internal.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode80b")
    ap.add_argument("--extra", default="prefill80b,zipf80b_t64,decode35b,decode80b_int8,prefill80b_int8,gdn80b",
                    help="comma-separated workloads measured after the headline, as sub-records of the same "
                         "line (N = 1 only; empty: none)")
    ap.add_argument("--layers", type=int, default=0, help="override the stack depth (profiling of small cases)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="stack", choices=["stack", "layers", "cached"],
                    help="one-token steps: one moe_decode_stack launch (default), moe_route + moe_forward per "
                         "layer, or per layer through the streaming slot pool (cached)")
    ap.add_argument("--cache-fraction", type=float, default=0.25,
                    help="cached path: device slots as a fraction of all experts of the stack")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


# --------------------------------------------------------------- clock sampler

REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
           0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler(threading.Thread):
    """Reads the SM clock, the max SM clock and the clock-event reasons
    through NVML (read only) every few ms while running."""

    def __init__(self, period=0.002):
        super().__init__(daemon=True)
        self.period = period
        self.samples = []
        self.stop_flag = threading.Event()
        self.ok = False
        try:
            import torch
            nv = C.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(torch.cuda.current_device())
            bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            h = C.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), C.byref(h)) != 0:
                return
            self.nv, self.h = nv, h
            mx = C.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, 1, C.byref(mx))
            self.max_mhz = mx.value
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except Exception:                                 # noqa: BLE001
            self.ok = False

    def run(self):
        if not self.ok:
            return
        mhz, mask = C.c_uint(), C.c_ulonglong()
        while not self.stop_flag.is_set():
            self.nv.nvmlDeviceGetClockInfo(self.h, 1, C.byref(mhz))
            self.reasons_fn(self.h, C.byref(mask))
            self.samples.append((mhz.value, mask.value))
            time.sleep(self.period)

    def stop(self):
        self.stop_flag.set()
        if self.is_alive():
            self.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": getattr(self, "max_mhz", None), "reasons": [],
                    "samples": len(self.samples), "source": "nvml" if self.ok else "unavailable"}
        bits = 0
        for _, m in self.samples:
            bits |= m
        return {"sm_mhz": statistics.median(s for s, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in REASONS.items() if bits & b and n != "gpu_idle"],
                "samples": len(self.samples), "source": "nvml"}


# ---------------------------------------------------------------- helpers

def src_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


STACK_SOURCES = ["int4_routed_expert_router_gb300/csrc/decode_stack.cu",
                 "int4_routed_expert_router_gb300/csrc/decode_common.cuh",
                 "int4_routed_expert_router_gb300/csrc/route_common.cuh",
                 "int4_routed_expert_router_gb300/csrc/smoe_dev.cuh",
                 "int4_routed_expert_router_gb300/csrc/smoe_internal.h"]


def _traffic_record(name: str, sources, workload: str, key: str):
    """Field `key` of workload's record in profiles/<name> (a committed ncu
    capture: {"source_sha256": ..., "records": {workload: {...}}}), only if
    the kernel's sources are unchanged since it was taken."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_sha256") != src_hash(sources):
        return None
    return d.get("records", {}).get(workload, {}).get(key)


def stack_traffic(workload: str):
    """DRAM bytes per layer of the stack kernel (captured on a shorter stack;
    the traffic is per layer)."""
    return _traffic_record("decode_stack_kernel_traffic.json", STACK_SOURCES, workload, "dram_bytes_per_layer")


def recorded_traffic(workload: str):
    """DRAM bytes per launch (one layer) of the decode kernel."""
    return _traffic_record("decode_kernel_traffic.json", DECODE_SOURCES, workload, "dram_bytes_per_launch")


PREFILL_SOURCES = ["int4_routed_expert_router_gb300/csrc/prefill.cu",
                   "int4_routed_expert_router_gb300/csrc/smoe_dev.cuh",
                   "int4_routed_expert_router_gb300/csrc/smoe_internal.h"]


def prefill_traffic(workload: str):
    """DRAM bytes per launch of the gate/up expert GEMM."""
    return _traffic_record("expert_gemm_traffic.json", PREFILL_SOURCES, workload, "dram_bytes_per_launch")


L2_BYTES = 129 * 10**6


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest value over all ranks (the slowest rank's time), or value
    itself when there is one process."""
    if not dist:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_of(wl, note="", blobs=None, flushed=False):
    """blobs: distinct expert blobs one step streams (routed + shared, all layers)."""
    if blobs is None:
        blobs = wl.n_layers * (min(wl.E, wl.k * wl.T) + 1)
    mb = blobs * 1769472 / 1e6
    if flushed:
        l2 = ("L2 flushed between timed steps (a 256 MB write outside the timed events): one step "
              "streams only %d distinct expert blobs (%.0f MB)" % (blobs, mb))
    else:
        l2 = "no flush: each step streams %d distinct expert blobs (%.0f MB) through the 129 MB L2" % (blobs, mb)
    return {"workload": wl.name + ": " + wl.description, "H": wl.H, "E": wl.E, "k": wl.k, "I": wl.I,
            "I_shared": wl.I_shared, "T": wl.T, "layers": wl.n_layers, "seed": wl.seed, "l2": l2,
            "note": note}


def cpu_baseline(wl, budget_s: float):
    """The oracle as it stands (one thread) on a bounded sample of the
    workload: for one-token stacks, the token through consecutive layers; for
    batches, tokens of the first layer in order, until the budget is used."""
    import numpy as np

    import oracle
    import synthetic
    bias = synthetic.zipf_bias(wl.seed, wl.E) if wl.zipf else None
    done, spent, layer = 0, 0.0, 0
    if wl.T == 1:
        x = synthetic.activations(wl.seed, 1, wl.H, tag=4242)
        while spent < budget_s and layer < wl.n_layers:
            Wr = synthetic.router_weights(wl.seed, layer, wl.E, wl.H)
            ws = synthetic.shared_gate_weights(wl.seed, layer, wl.H)
            t0 = time.perf_counter()
            ids, w, gate = oracle.route(x, Wr, ws, wl.k, bias=bias)
            t_route = time.perf_counter() - t0
            experts = {int(e): synthetic.expert_triples(wl.seed, layer, int(e), wl.H, wl.I) for e in np.unique(ids)}
            shared = synthetic.expert_triples(wl.seed, layer, None, wl.H, wl.I_shared)
            t0 = time.perf_counter()
            out64, _ = oracle.combine(x, ids, w, gate, experts, shared, wl.E, wl.I, wl.I_shared)
            spent += t_route + time.perf_counter() - t0
            x = oracle.residual(x, out64)
            done += 1
            layer += 1
        what = "1 token through %d of %d layers" % (layer, wl.n_layers)
    else:
        x = synthetic.activations(wl.seed, wl.T, wl.H, tag=4242)
        Wr = synthetic.router_weights(wl.seed, 0, wl.E, wl.H)
        ws = synthetic.shared_gate_weights(wl.seed, 0, wl.H)
        shared = synthetic.expert_triples(wl.seed, 0, None, wl.H, wl.I_shared)
        cache = {}
        while spent < budget_s and done < wl.T:
            xt = x[done:done + 8]
            t0 = time.perf_counter()
            ids, w, gate = oracle.route(xt, Wr, ws, wl.k, bias=bias)
            t_route = time.perf_counter() - t0
            for e in np.unique(ids):
                if int(e) not in cache:
                    cache[int(e)] = synthetic.expert_triples(wl.seed, 0, int(e), wl.H, wl.I)
            experts = {int(e): cache[int(e)] for e in np.unique(ids)}
            t0 = time.perf_counter()
            oracle.combine(xt, ids, w, gate, experts, shared, wl.E, wl.I, wl.I_shared)
            spent += t_route + time.perf_counter() - t0
            done += xt.shape[0]
        what = "first %d of %d tokens of layer 0" % (done, wl.T)
    value = done / spent           # (token, layer) passes per second
    return {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%s (expert regeneration excluded), %.1f s on one core" % (what, spent)}


# ------------------------------------------------------------------ arms

def run_reference(args, wl, world, rank):
    """The oracle timed on the host cores: each step one layer for one token."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    import synthetic
    pre = []
    x = synthetic.activations(wl.seed, wl.T, wl.H, tag=4242)
    for i in range(min(args.warmup + args.steps, wl.n_layers)):
        Wr = synthetic.router_weights(wl.seed, i, wl.E, wl.H)
        ws = synthetic.shared_gate_weights(wl.seed, i, wl.H)
        bias = synthetic.zipf_bias(wl.seed, wl.E) if wl.zipf else None
        ids, w, gate = oracle.route(x, Wr, ws, wl.k, bias=bias)
        experts = {int(e): synthetic.expert_triples(wl.seed, i, int(e), wl.H, wl.I) for e in np.unique(ids)}
        shared = synthetic.expert_triples(wl.seed, i, None, wl.H, wl.I_shared)
        pre.append((x, Wr, ws, bias, experts, shared))
        out64, _ = oracle.combine(x, ids, w, gate, experts, shared, wl.E, wl.I, wl.I_shared)
        x = oracle.residual(x, out64)

    def step(i):
        x, Wr, ws, bias, experts, shared = pre[i % len(pre)]
        ids, w, gate = oracle.route(x, Wr, ws, wl.k, bias=bias)
        oracle.combine(x, ids, w, gate, experts, shared, wl.E, wl.I, wl.I_shared)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = args.steps * wl.T / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(wl, "oracle: one layer for one token per step"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "each step: one layer for one token (router + experts); expert "
                                       "regeneration outside the timed region"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(args, wl, dev, dist=None, e2e=False, cached_pool=None):
    """Builds the workload on the device, captures one step in a CUDA graph
    and times it: K replays after W warm-up replays (bracketed by a barrier
    and synchronize), the dominant kernel(s) by event nodes inside an
    instrumented copy of the graph, and optionally end to end (x from pinned
    host memory, the step, the result back). Returns a dict of raw figures."""
    import numpy as np
    import torch

    import int4_routed_expert_router_gb300 as smoe
    import synthetic
    import workload as W

    pool = W.DevicePool(wl)
    inp = W.LayerInputs(wl, wl.n_layers)
    # one-token steps run as one moe_decode_stack launch when the GPU supports it
    stacked = wl.T == 1 and args.path == "stack" and pool.ctx.stack_workspace_bytes(wl.n_layers) > 0
    st = W.DecodeStep(pool, inp) if stacked else W.Stack(pool, inp, wl.T)
    x0 = synthetic.activations(wl.seed, wl.T, wl.H, tag=4242)
    st.xs[0].copy_(W.bf16_tensor(x0))
    g = st.capture()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if smoe.check(st.err) != 0:
        raise RuntimeError("device error word set during warm-up")

    # distinct expert blobs per step (the routing is the same every replay)
    uniq = [len(np.unique((st.ids[l] if not stacked else st.ids[l]).cpu().numpy())) for l in range(wl.n_layers)]
    blobs = sum(u + 1 for u in uniq)
    flush = blobs * int(pool.layout.blob_bytes) < 2 * L2_BYTES

    # ---- timed region: K replays of the whole step (each bracketed by its own
    # events when L2 is flushed in between)
    sampler = ClockSampler()
    sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if flush:
        scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        evs_t = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for a, b in evs_t:
            scratch.fill_(1)
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        ms = float(sum(a.elapsed_time(b) for a, b in evs_t))
        del scratch
    else:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1)
    if dist:
        dist.barrier()
    sampler.stop()
    ms = max_over_ranks(ms, dist, dev)
    if smoe.check(st.err) != 0:
        raise RuntimeError("device error word set during the timed region")

    # ---- the dominant kernel, bracketed by event nodes that the library's
    # profiling hook records inside an instrumented copy of the graph
    prefill = wl.T > 8
    kern_ms = down_ms = None
    try:
        nev = 3 if prefill else 2
        nrow = 1 if stacked else wl.n_layers
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(nev)] for _ in range(nrow)]
        for row in evs:
            for e in row:
                e.record()                      # creates the events
        torch.cuda.synchronize()
        gi = st.capture(prof_events=evs[0] if stacked else evs)
        reps = max(3, min(args.steps, 100))
        tot, tot_down = [], []
        scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
        for _ in range(reps):
            if scratch is not None:
                scratch.fill_(1)
            gi.replay()
            torch.cuda.synchronize()
            tot.extend(row[0].elapsed_time(row[1]) for row in evs)
            if prefill:
                tot_down.extend(row[1].elapsed_time(row[2]) for row in evs)
        kern_ms = float(np.mean(tot))
        down_ms = float(np.mean(tot_down)) if prefill else None
        del gi, scratch
    except Exception as e:                               # noqa: BLE001
        print("kernel timing unavailable: %r" % (e,), file=sys.stderr)

    out = dict(ms=ms, stacked=stacked, prefill=prefill, kern_ms=kern_ms, down_ms=down_ms, uniq=uniq, blobs=blobs,
               flush=flush, blob=int(pool.layout.blob_bytes), clocks=sampler.summary())

    # ---- end to end: x from pinned host memory, the step, the result back
    if e2e:
        xh = torch.from_numpy(x0.view(np.int16)).view(torch.bfloat16).pin_memory()
        oh = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            st.xs[0].copy_(xh, non_blocking=True)
            g.replay()
            oh.copy_(st.xs[wl.n_layers], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        out["e2e_ms"] = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    del g, st, pool
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def roofline_of(wl, m, pk, pk_src):
    """The roofline record of one measurement. One-token and small batches
    (T <= 64) are bounded by HBM: the algorithmic bytes are the distinct
    routed experts' blobs plus the shared expert's, per layer; for the
    one-launch stack the achieved rate uses that kernel's launch time, for a
    T = 64 layer the whole layer's time (router, bucketing, GEMMs and
    combine). T = 8192 prefill is a dense contraction bounded by the tensor
    cores: gate/up 2 (2 I) H and down 2 I H FLOPs per (token, expert) pair,
    pairs = T k routed + T shared, against the bf16 dense peak (the fp16
    rate is the same)."""
    import numpy as np
    blob = m["blob"]
    hbm = "MEASURED_PEAKS.json hbm_gbs (measured)" if pk_src == "measured" else "fallback 6.8 TB/s"
    if wl.T <= 64:
        per_layer = float(np.mean(m["uniq"]) + 1) * blob
        if m["stacked"]:
            alg, t_ms, kern = per_layer * wl.n_layers, m["kern_ms"], \
                "decode_stack_kernel (moe_decode_stack: %d layers per launch)" % wl.n_layers
        elif wl.T <= 8:
            alg, t_ms, kern = per_layer, m["kern_ms"], "decode_kernel (moe_forward, T <= 8)"
        else:
            alg, t_ms = per_layer, m["ms"] / m.get("steps", 1) / wl.n_layers
            kern = "whole layer (moe_route + moe_forward on the token-bucketed path)"
        if not t_ms:
            return None
        ach = alg / (t_ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "kernel": kern, "bytes_per_launch": int(alg),
                "us_per_launch": round(t_ms * 1e3, 3), "peak_source": hbm}
    if not m["kern_ms"]:
        return None
    pairs = wl.T * wl.k + wl.T
    f_gu = 2.0 * pairs * 2 * wl.I * wl.H
    f_dn = 2.0 * pairs * wl.I * wl.H
    peak = pk["bf16_tflops"]
    t_gu, t_dn = m["kern_ms"] / 1e3, (m["down_ms"] or 0) / 1e3
    comb = (f_gu + f_dn) / (t_gu + t_dn) / 1e12 if m["down_ms"] else None
    return {"bound": "tensor", "achieved": round(comb or f_gu / t_gu / 1e12, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round((comb or f_gu / t_gu / 1e12) / peak, 4),
            "kernel": "expert_gemm_kernel, gate/up and down launches together (fp16 operands, A in TMEM, fp32 "
                      "accumulate)",
            "flops_per_launch": f_gu + f_dn, "us_per_launch": round((t_gu + t_dn) * 1e6, 3),
            "gate_up_us": round(t_gu * 1e6, 3), "gate_up_tflops": round(f_gu / t_gu / 1e12, 1),
            "gate_up_frac": round(f_gu / t_gu / 1e12 / peak, 4),
            "down_us": round(t_dn * 1e6, 3) if m["down_ms"] else None,
            "down_tflops": round(f_dn / t_dn / 1e12, 1) if m["down_ms"] else None,
            "layer_us": round(m["ms"] / m.get("steps", 1) / wl.n_layers * 1e3, 3),
            "peak_source": "MEASURED_PEAKS.json bf16_tflops (measured; fp16 dense rate = bf16)"
            if pk_src == "measured" else "fallback 1.9 PFLOP/s"}


GDN_SOURCES = ["int4_routed_expert_router_gb300/csrc/deltanet.cu",
               "int4_routed_expert_router_gb300/csrc/smoe_dev.cuh",
               "int4_routed_expert_router_gb300/csrc/smoe_internal.h"]


def gdn_traffic(workload: str):
    """DRAM bytes per launch of the DeltaNet step kernel."""
    return _traffic_record("gdn_step_kernel_traffic.json", GDN_SOURCES, workload, "dram_bytes_per_launch")


def measure_gdn(args, gs, dev, pk, pk_src):
    """The Gated DeltaNet recurrence step of one layer (gdn_step) on the
    state of gs.B sequences: K launches after W warm-up launches, timed with
    events on the launching stream; the state (far larger than L2 at the 80B
    shape) is updated in place by every launch. HBM-bound: the algorithmic
    bytes are the fp32 state read and written once, plus q, k, v, the gates
    and the bf16 output."""
    import torch

    import int4_routed_expert_router_gb300 as smoe
    import synthetic
    from workload import bf16_tensor

    q, k, v, g, beta, S0 = synthetic.gdn_inputs(gs.seed, gs.T, gs.B, gs.nk, gs.nv, gs.dk, gs.dv, tag=11)
    qd, kd, vd = bf16_tensor(q), bf16_tensor(k), bf16_tensor(v)
    gd, bd = torch.from_numpy(g).to(dev), torch.from_numpy(beta).to(dev)
    S = torch.from_numpy(S0).to(dev)
    out = torch.empty((gs.T, gs.B, gs.nv, gs.dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        smoe.gdn_step(gs.nk, gs.nv, qd, kd, vd, gd, bd, S, out, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    state_bytes = S.numel() * 4
    flush = 2 * state_bytes < 2 * L2_BYTES
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    sampler = ClockSampler()
    sampler.start()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in evs:
        if scratch is not None:
            scratch.fill_(1)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    ms = float(sum(a.elapsed_time(b) for a, b in evs))
    alg = 2 * state_bytes + (q.nbytes + k.nbytes + v.nbytes) + g.nbytes + beta.nbytes + out.numel() * 2
    t = ms / 1e3 / args.steps
    ach = alg / t / 1e9
    del S, out, scratch
    torch.cuda.empty_cache()
    return {"workload": gs.description, "value": round(gs.B * gs.T * args.steps / (ms / 1e3), 1),
            "unit": "DeltaNet-layer tokens/s", "us_per_launch": round(t * 1e6, 3),
            "l2": "flushed between timed steps" if flush else "no flush (state larger than L2)",
            "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(ach / pk["hbm_gbs"], 4), "kernel": "gdn_step_kernel (gdn_step)",
                         "bytes_per_launch": int(alg), "us_per_launch": round(t * 1e6, 3),
                         "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)" if pk_src == "measured"
                         else "fallback 6.8 TB/s", "traffic": gdn_traffic(gs.name)},
            "clocks": sampler.summary()}


def traffic_of(wl, m):
    if m["stacked"]:
        t = stack_traffic(wl.name)
        return t * wl.n_layers if t else None
    if wl.T <= 8:
        return recorded_traffic(wl.name)
    if wl.T > 64:
        return prefill_traffic(wl.name)
    return None


def run_ours(args, wl, world, rank, dist):
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    m = measure(args, wl, dev, dist, e2e=True)
    m["steps"] = args.steps
    ms = m["ms"]
    step_s = ms / 1e3 / args.steps
    value = world * wl.T * wl.n_layers / step_s
    e2e = {"value": round(world * wl.T * wl.n_layers * args.steps / (m["e2e_ms"] / 1e3), 1), "unit": UNIT,
           "h2d_bytes_per_step": wl.T * wl.H * 2, "d2h_bytes_per_step": wl.T * wl.H * 2}
    pk, pk_src = peaks()
    roof = roofline_of(wl, m, pk, pk_src)
    if roof is not None:
        roof["traffic"] = traffic_of(wl, m)

    # ---- the other target configurations, each measured the same way on this
    # GPU after the headline (same steps and warm-up), as sub-records
    extra = {}
    if world == 1 and args.extra:
        import synthetic
        for name in [n for n in args.extra.split(",") if n and n != wl.name]:
            if name in synthetic.GDN_WORKLOADS:
                extra[name] = measure_gdn(args, synthetic.GDN_WORKLOADS[name], dev, pk, pk_src)
                continue
            w2 = synthetic.WORKLOADS[name]
            m2 = measure(args, w2, dev)
            m2["steps"] = args.steps
            r2 = roofline_of(w2, m2, pk, pk_src)
            if r2 is not None:
                r2["traffic"] = traffic_of(w2, m2)
            extra[name] = {"workload": w2.description, "value": round(w2.T * w2.n_layers * args.steps /
                                                                        (m2["ms"] / 1e3), 1), "unit": UNIT,
                           "us_per_layer": round(1e3 * m2["ms"] / args.steps / w2.n_layers, 3),
                           "l2": "flushed between timed steps" if m2["flush"] else "no flush",
                           "distinct_blobs_per_step": m2["blobs"], "roofline": r2, "clocks": m2["clocks"]}

    if rank != 0:
        return
    stacked, prefill = m["stacked"], m["prefill"]
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16" if prefill else "bf16", "data": "synthetic",
            "config": config_of(wl, ("CUDA graph of one moe_decode_stack call (%d layers in one launch); us per layer "
                                     "%.3f" if stacked else "CUDA graph of %d x (moe_route + moe_forward); us per "
                                     "layer %.3f") % (wl.n_layers, 1e3 * ms / args.steps / wl.n_layers), m["blobs"],
                                m["flush"]),
            "roofline": roof, "e2e": e2e,
            # per step: the one stack kernel; else per layer: decode = router + fused expert kernel;
            # bucketed path = router GEMM + top-k, 3 bucketing kernels, row gather, 2 grouped GEMMs, combine
            "gpu_launches": (1 if stacked else (9 if prefill else 2) * wl.n_layers) * args.steps,
            "clocks": m["clocks"]}
    if extra:
        line["configs"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_cached(args, wl, world, rank):
    """One token per step through the stack, per layer: moe_route, its ids read
    to the host, smoe_cache_prepare (misses copied from pinned host memory into
    the bounded device pool), moe_forward. The steps cycle through 64 seeded
    token inputs (a decoded sequence), so the routing changes from step to step."""
    import numpy as np
    import torch

    import int4_routed_expert_router_gb300 as smoe
    import synthetic
    import workload as W

    full = W.DevicePool(wl)
    inp = W.LayerInputs(wl, wl.n_layers)
    L, E, stride = wl.n_layers, wl.E, full.stride
    idx = torch.from_numpy(full.table.astype(np.int64)).cuda().reshape(-1)
    store = torch.empty(L * E * stride, dtype=torch.uint8).pin_memory()
    for l in range(L):                                   # every expert's blob, [layer][expert] order
        store[l * E * stride:(l + 1) * E * stride].copy_(full.pool.view(-1, stride).index_select(0, idx[l * E:(l + 1) * E]).reshape(-1))
    shared = full.shared
    del full
    torch.cuda.empty_cache()
    n_slots = max(4 * wl.k, int(args.cache_fraction * L * E))
    pool = torch.empty(n_slots * stride, dtype=torch.uint8, device="cuda")
    table = torch.zeros((L, E), dtype=torch.int32, device="cuda")
    ctx = smoe.Context(smoe.make_shape(wl.H, wl.E, wl.k, wl.I, wl.I_shared), L, n_slots, table)
    cache = smoe.Cache(ctx, store, pool)
    xs = torch.zeros((L + 1, 1, wl.H), dtype=torch.bfloat16, device="cuda")
    tokens = W.bf16_tensor(synthetic.activations(wl.seed, 64, wl.H, tag=4243))      # [64, H]
    ids = torch.zeros((1, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((1, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros((1,), dtype=torch.float32, device="cuda")
    ws = W.workspace(ctx, 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids_h = torch.zeros((1, wl.k), dtype=torch.int32).pin_memory()

    def step(i):
        xs[0].copy_(tokens[i % 64:i % 64 + 1])
        for l in range(L):
            smoe.moe_route(ctx, inp.Wr[l], inp.ws[l], xs[l], ids, w, gate, ws, logit_bias=inp.bias)
            ids_h.copy_(ids)                                 # waits for the routing
            cache.prepare(l, ids_h.numpy())
            smoe.moe_forward(ctx, l, xs[l], ids, w, gate, pool, shared[l], xs[l + 1], ws, err, residual=xs[l])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    h0, m0, b0 = cache.stats()
    sampler = ClockSampler()
    sampler.start()
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    sampler.stop()
    if smoe.check(err) != 0:
        raise RuntimeError("device error word set during the cached run")
    h1, m1, b1 = cache.stats()
    hits, misses, nbytes = h1 - h0, m1 - m0, b1 - b0
    value = args.steps * L / el
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(wl, "streaming slot pool: %d of %d experts resident, per layer moe_route, ids to "
                                    "the host, smoe_cache_prepare, moe_forward; steps cycle through 64 token "
                                    "inputs" % (n_slots, L * E), None, False),
            "cache": {"slots": n_slots, "experts": L * E, "hit_rate": round(hits / max(1, hits + misses), 4),
                      "copied_bytes_per_step": nbytes // max(1, args.steps),
                      "host_to_device_GBps": round(nbytes / el / 1e9, 2), "us_per_layer": round(1e6 * el / args.steps / L, 3)},
            "gpu_launches": 2 * L * args.steps, "clocks": sampler.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    import synthetic
    wl = synthetic.WORKLOADS[args.workload]
    if args.layers:
        wl = dataclasses.replace(wl, n_layers=args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl" if args.impl == "ours" else "gloo")
        dist = tdist
    try:
        if args.impl == "reference":
            run_reference(args, wl, world, rank)
        elif args.path == "cached":
            run_cached(args, wl, world, rank)
        else:
            run_ours(args, wl, world, rank, dist)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
