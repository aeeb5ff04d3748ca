"""Synthetic workloads on the device, for the tests and the benchmark.

Glue only: draws inputs with ``synthetic`` (host numpy and the device
generator ``synthetic/libsynth.so``) and lays the expert pool out with the
library's own ``pack_experts``. Holds none of the layer's arithmetic.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

import int4_routed_expert_router_gb300 as smoe
import synthetic
from synthetic import _build as synth_build

_synth = None


def synth_lib():
    global _synth
    if _synth is None:
        L = C.CDLL(synth_build.build())
        L.synth_expert_triples.argtypes = [C.c_uint64, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int] + \
            [C.c_void_p] * 10
        L.synth_expert_triples.restype = C.c_int
        L.synth_expert_triples_bits.argtypes = [C.c_uint64] + [C.c_int] * 6 + [C.c_void_p] * 10
        L.synth_expert_triples_bits.restype = C.c_int
        _synth = L
    return _synth


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).to(device).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def device_triples(seed: int, layer: int, code0: int, n: int, H: int, I: int, stream=None, bits: int = 4):
    """Triples of n consecutive experts generated on the device: 9 tensors with
    a leading expert dimension, in ExpertTriples order (4-bit or 8-bit q)."""
    dev = torch.device("cuda")
    per = 32 // bits
    shapes = [(I, H // per), (I, H // 64), (I, H // 64)] * 2 + [(H, I // per), (H, I // 64), (H, I // 64)]
    dts = [torch.int32, torch.int16, torch.int16] * 3
    ts = [torch.empty((n,) + s, dtype=d, device=dev) for s, d in zip(shapes, dts)]
    st = torch.cuda.current_stream().cuda_stream if stream is None else stream.cuda_stream
    rc = synth_lib().synth_expert_triples_bits(seed, layer, code0, n, H, I, bits, *[t.data_ptr() for t in ts], st)
    if rc != 0:
        raise RuntimeError("synth_expert_triples failed: %d" % rc)
    return ts


class DevicePool:
    """Expert pool of a workload on the device, with its slot table and shared blobs."""

    def __init__(self, wl: synthetic.Workload, n_layers: int | None = None, table: np.ndarray | None = None):
        self.wl = wl
        L = wl.n_layers if n_layers is None else n_layers
        self.n_layers = L
        self.shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I, wl.I_shared, bits=wl.bits)
        self.layout = smoe.layout_of(self.shape)
        self.stride = int(self.layout.blob_bytes)
        self.table = synthetic.slot_table(wl.seed, L, wl.E, wl.permuted_slots) if table is None else table
        self.n_slots = L * wl.E
        self.pool = torch.empty(self.n_slots * self.stride, dtype=torch.uint8, device="cuda")
        self.shared = torch.empty((L, self.stride), dtype=torch.uint8, device="cuda")
        self.table_dev = torch.zeros((L, wl.E), dtype=torch.int32, device="cuda")
        self.ctx = smoe.Context(self.shape, L, self.n_slots, self.table_dev)
        for layer in range(L):
            smoe.set_slot_table(self.ctx, layer, self.table[layer])
            self._fill_layer(layer)
        torch.cuda.synchronize()

    def _fill_layer(self, layer: int):
        wl = self.wl
        chunk = 128
        for e0 in range(0, wl.E, chunk):
            n = min(chunk, wl.E - e0)
            ts = device_triples(wl.seed, layer, e0, n, wl.H, wl.I, bits=wl.bits)
            experts = [[t[i] for t in ts] for i in range(n)]
            slots = [int(self.table[layer, e0 + i]) for i in range(n)]
            smoe.pack_experts(self.shape, experts, slots, self.pool, self.pool.numel(), smoe.DEVICE)
            torch.cuda.synchronize()
        ts = device_triples(wl.seed, layer, synthetic.SHARED_EXPERT_CODE, 1, wl.H, wl.I_shared, bits=wl.bits)
        smoe.pack_experts(self.shape, [[t[0] for t in ts]], [0], self.shared[layer],
                          self.stride, smoe.DEVICE)

    def set_table(self, layer: int, table_row: np.ndarray):
        smoe.set_slot_table(self.ctx, layer, table_row)


class LayerInputs:
    """Router weights, shared-gate vector and (optional) Zipf offsets of a layer stack."""

    def __init__(self, wl: synthetic.Workload, n_layers: int):
        self.Wr_bits = [synthetic.router_weights(wl.seed, l, wl.E, wl.H) for l in range(n_layers)]
        self.ws_bits = [synthetic.shared_gate_weights(wl.seed, l, wl.H) for l in range(n_layers)]
        self.Wr = [bf16_tensor(b) for b in self.Wr_bits]
        self.ws = [bf16_tensor(b) for b in self.ws_bits]
        self.bias_np = synthetic.zipf_bias(wl.seed, wl.E) if wl.zipf else None
        self.bias = None if self.bias_np is None else torch.from_numpy(self.bias_np).cuda()


def workspace(ctx: smoe.Context, T: int) -> torch.Tensor:
    n = ctx.workspace_bytes(T)
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device="cuda")


class Stack:
    """A decode step through an L-layer stack: per layer moe_route then
    moe_forward with the residual fused, x_{l+1} = bf16(x_l + layer_l(x_l)).
    Buffers are preallocated so the step can be captured in a CUDA graph."""

    def __init__(self, pool: DevicePool, inputs: LayerInputs, T: int):
        wl = pool.wl
        self.pool, self.inputs, self.T = pool, inputs, T
        L = pool.n_layers
        dev = "cuda"
        self.xs = [torch.zeros((T, wl.H), dtype=torch.bfloat16, device=dev) for _ in range(L + 1)]
        self.ids = [torch.zeros((T, wl.k), dtype=torch.int32, device=dev) for _ in range(L)]
        self.w = [torch.zeros((T, wl.k), dtype=torch.float32, device=dev) for _ in range(L)]
        self.gate = [torch.zeros((T,), dtype=torch.float32, device=dev) for _ in range(L)]
        self.ws = workspace(pool.ctx, T)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def enqueue(self, stream=None, prof_events=None):
        """prof_events: optional per-layer lists of events for the profiling hook."""
        p, inp = self.pool, self.inputs
        for l in range(p.n_layers):
            smoe.moe_route(p.ctx, inp.Wr[l], inp.ws[l], self.xs[l], self.ids[l], self.w[l], self.gate[l],
                           self.ws, logit_bias=inp.bias, stream=stream)
            if prof_events is not None:
                p.ctx.set_profile_events(prof_events[l])
            smoe.moe_forward(p.ctx, l, self.xs[l], self.ids[l], self.w[l], self.gate[l], p.pool, p.shared[l],
                             self.xs[l + 1], self.ws, self.err, residual=self.xs[l], stream=stream)
        if prof_events is not None:
            p.ctx.set_profile_events([])

    def capture(self, prof_events=None):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue(s)            # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.enqueue(s, prof_events)
        torch.cuda.synchronize()
        if prof_events is None:
            self.graph = g
        return g


class DecodeStep:
    """A one-token decode step through the whole stack as one moe_decode_stack
    call (one persistent launch): xs_buf [L + 1][1][H] holds the input and
    each layer's output; ids/w/gate [L][k], [L]."""

    def __init__(self, pool: DevicePool, inputs: LayerInputs):
        wl = pool.wl
        L = pool.n_layers
        self.pool, self.inputs, self.T = pool, inputs, 1
        self.xs_buf = torch.zeros((L + 1, 1, wl.H), dtype=torch.bfloat16, device="cuda")
        self.xs = [self.xs_buf[l] for l in range(L + 1)]      # [1][H] views, as in Stack
        self.ids = torch.zeros((L, wl.k), dtype=torch.int32, device="cuda")
        self.w = torch.zeros((L, wl.k), dtype=torch.float32, device="cuda")
        self.gate = torch.zeros((L,), dtype=torch.float32, device="cuda")
        n = pool.ctx.stack_workspace_bytes(L)
        if n == 0:
            raise RuntimeError("moe_decode_stack is not available for this shape / GPU")
        self.ws = torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.shared = [pool.shared[l] for l in range(L)]
        self.graph = None

    def enqueue(self, stream=None, prof_events=None):
        """prof_events: optional [before, after] events for the profiling hook."""
        p, inp = self.pool, self.inputs
        if prof_events is not None:
            p.ctx.set_profile_events(prof_events)
        smoe.moe_decode_stack(p.ctx, 0, inp.Wr, inp.ws, self.shared, self.xs_buf, self.ids, self.w, self.gate, p.pool,
                              self.ws, self.err, logit_bias=inp.bias, stream=stream)
        if prof_events is not None:
            p.ctx.set_profile_events([])

    capture = Stack.capture

