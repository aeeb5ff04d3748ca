"""Python binding of libsmoe.so, the int4 routed-expert MoE layer for GB300.

Argument marshalling only: every step of the layer runs in the CUDA kernels
behind the C ABI (``include/smoe.h``). Device tensors are torch tensors (used
for device memory and streams); host buffers are numpy arrays. If the library
is not built this module raises on first use: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsmoe.so")

OK, EINVAL, ERANGE, ENOMEM, ECUDA, EDEVICE, ENOTSUP = 0, -1, -2, -3, -4, -5, -6
DEV_BAD_SLOT, DEV_BAD_EXPERT, DEV_TIMEOUT, DEV_RANGE = 1, 2, 3, 4
MAX_TOKENS = 1 << 20          # SMOE_MAX_TOKENS: most tokens of one moe_route / moe_forward call
HOST, DEVICE = 0, 1
EXPORTS = ["smoe_layout_of", "pack_experts", "smoe_ctx_create", "smoe_ctx_destroy", "set_slot_table",
           "smoe_workspace_bytes", "moe_route", "moe_forward", "moe_forward_noalloc", "moe_decode_stack",
           "smoe_stack_workspace_bytes", "smoe_check", "smoe_ctx_describe", "smoe_set_profile_events",
           "smoe_status_string", "smoe_cache_create", "smoe_cache_destroy", "smoe_cache_prepare",
           "smoe_cache_stats", "smoe_cache_simulate", "moe_forward_debug", "smoe_set_stack_wait", "gdn_step",
           "smoe_quantize_mlx"]


class SmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (%d)" % (what, status_string(status), status))
        self.status = status


class Shape(C.Structure):
    _fields_ = [("H", C.c_int32), ("E", C.c_int32), ("k", C.c_int32), ("I", C.c_int32),
                ("I_shared", C.c_int32), ("group", C.c_int32), ("bits", C.c_int32)]


class Layout(C.Structure):
    _fields_ = [("blob_bytes", C.c_uint64), ("gu_offset", C.c_uint64), ("gu_bytes", C.c_uint64),
                ("down_offset", C.c_uint64), ("down_bytes", C.c_uint64), ("atom_bytes", C.c_uint32),
                ("atom_rows", C.c_uint32), ("group", C.c_uint32), ("reserved", C.c_uint32)]


class GdnShape(C.Structure):
    _fields_ = [("nk", C.c_int32), ("nv", C.c_int32), ("dk", C.c_int32), ("dv", C.c_int32)]


class ExpertSrc(C.Structure):
    _fields_ = [("q", C.c_void_p * 3), ("s", C.c_void_p * 3), ("b", C.c_void_p * 3)]


_lib = None


def lib():
    """The loaded libsmoe.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libsmoe.so is not built (run __graft_entry__.build() or "
                               "python int4_routed_expert_router_gb300/_build.py)")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, u64 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64
        L.smoe_layout_of.argtypes = [C.POINTER(Shape), C.POINTER(Layout)]
        L.pack_experts.argtypes = [C.POINTER(Shape), C.POINTER(ExpertSrc), i32, C.POINTER(C.c_int64), vp, u64,
                                   i32, vp]
        L.smoe_ctx_create.argtypes = [C.POINTER(Shape), i32, i64, vp, C.POINTER(vp)]
        L.smoe_ctx_destroy.argtypes = [vp]
        L.set_slot_table.argtypes = [vp, i32, vp, vp]
        L.smoe_workspace_bytes.argtypes = [vp, i32]
        L.smoe_workspace_bytes.restype = u64
        L.moe_route.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, u64, vp]
        L.moe_forward.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, u64, vp, vp, vp, vp, u64, vp, vp]
        L.moe_forward_noalloc.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, u64, vp, vp, vp, vp, vp]
        L.moe_decode_stack.argtypes = [vp, i32, i32, C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), vp, vp, vp, vp,
                                       vp, vp, u64, vp, u64, vp, vp]
        L.moe_forward_debug.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, u64, vp, vp, vp, vp, vp]
        L.smoe_cache_create.argtypes = [vp, vp, u64, vp, u64, vp, C.POINTER(vp)]
        L.smoe_cache_destroy.argtypes = [vp]
        L.smoe_cache_prepare.argtypes = [vp, i32, vp, i32, vp, C.POINTER(i32), C.POINTER(i32)]
        L.smoe_cache_stats.argtypes = [vp, C.POINTER(u64), C.POINTER(u64), C.POINTER(u64)]
        L.smoe_cache_simulate.argtypes = [i32, i32, i64, vp, i32, vp, C.POINTER(i64), C.POINTER(i64)]
        L.smoe_stack_workspace_bytes.argtypes = [vp, i32]
        L.smoe_stack_workspace_bytes.restype = u64
        L.smoe_check.argtypes = [vp, C.POINTER(C.c_int32), vp]
        L.smoe_ctx_describe.argtypes = [vp, C.c_char_p, i32]
        L.smoe_set_profile_events.argtypes = [vp, C.POINTER(vp), i32]
        L.smoe_set_stack_wait.argtypes = [vp, u64, i32]
        L.smoe_status_string.argtypes = [C.c_int]
        L.gdn_step.argtypes = [C.POINTER(GdnShape), i32, i32, vp, vp, vp, vp, vp, C.c_float, vp, vp, vp]
        L.smoe_quantize_mlx.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.smoe_status_string.restype = C.c_char_p
        for name in EXPORTS:
            if name not in ("smoe_workspace_bytes", "smoe_status_string"):
                getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().smoe_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise SmoeError(rc, what)


def _ptr(t) -> int | None:
    """Raw address of a torch tensor / numpy array (None stays NULL)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _dev(t, name: str, dtype=None, numel=None, min_bytes=None) -> int | None:
    """Address of a contiguous CUDA tensor, after checking its dtype and
    element count where given (None stays NULL). Anything else is refused
    here, so a kernel is never handed a host address or a short buffer."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s: expected a CUDA tensor, got %s" % (name, type(t).__name__ if not isinstance(
            t, torch.Tensor) else "a tensor on " + str(t.device)))
    if not t.is_contiguous():
        raise ValueError("%s: must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s: expected %s, got %s" % (name, dtype, t.dtype))
    if numel is not None and t.numel() != numel:
        raise ValueError("%s: expected %d elements, got %d" % (name, numel, t.numel()))
    if min_bytes is not None and t.numel() * t.element_size() < min_bytes:
        raise ValueError("%s: expected at least %d bytes, got %d" % (name, min_bytes, t.numel() * t.element_size()))
    return t.data_ptr()


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream) -> int | None:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except Exception:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_shape(H, E, k, I, I_shared=None, bits=4) -> Shape:
    """bits = 8: MLX's 8-bit format (two-plane atoms), taken by every call:
    layout, host and device packing, routing, moe_forward at any T,
    moe_forward_noalloc, moe_decode_stack and moe_forward_debug."""
    return Shape(H, E, k, I, I if I_shared is None else I_shared, 64, bits)


def layout_of(shape: Shape) -> Layout:
    out = Layout()
    _check(lib().smoe_layout_of(C.byref(shape), C.byref(out)), "smoe_layout_of")
    return out


def expert_src(arrays) -> ExpertSrc:
    """9 arrays/tensors in the order gate q,s,b, up q,s,b, down q,s,b."""
    st = ExpertSrc()
    for m in range(3):
        st.q[m] = _ptr(arrays[3 * m])
        st.s[m] = _ptr(arrays[3 * m + 1])
        st.b[m] = _ptr(arrays[3 * m + 2])
    return st


def quantize_mlx(w, bits: int = 4):
    """MLX-style affine triples of a float32 matrix [rows][cols] (host numpy,
    cols a multiple of 64): (q uint32 [rows][cols*bits/32], s, b fp16 bits
    [rows][cols/64]), by the library's smoe_quantize_mlx."""
    import numpy as np
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = w.shape
    q = np.zeros((rows, cols * bits // 32), np.uint32)
    s = np.zeros((rows, cols // 64), np.uint16)
    b = np.zeros((rows, cols // 64), np.uint16)
    _check(lib().smoe_quantize_mlx(w.ctypes.data, rows, cols, bits, q.ctypes.data, s.ctypes.data, b.ctypes.data),
           "smoe_quantize_mlx")
    return q, s, b


def pack_experts(shape: Shape, experts, slots, pool, pool_bytes: int, where: int, stream=None):
    """experts: list of 9-array lists (host numpy or device torch, per `where`)."""
    n = len(experts)
    srcs = (ExpertSrc * n)(*[expert_src(e) for e in experts])
    sl = (C.c_int64 * n)(*[int(s) for s in slots])
    st = None if where == HOST else _stream(stream)
    _check(lib().pack_experts(C.byref(shape), srcs, n, sl, _ptr(pool), int(pool_bytes), where, st),
           "pack_experts")


class Context:
    """Host-side context for one shape / layer stack / slot pool (smoe_ctx)."""

    def __init__(self, shape: Shape, n_layers: int, n_slots: int, table_dev):
        self.shape = shape
        self.n_layers = n_layers
        self.n_slots = n_slots
        self.table = table_dev          # keep the caller's tensor alive
        h = C.c_void_p()
        _check(lib().smoe_ctx_create(C.byref(shape), n_layers, n_slots, _ptr(table_dev), C.byref(h)),
               "smoe_ctx_create")
        self.handle = h.value
        self.layout = layout_of(shape)

    def close(self):
        if self.handle:
            lib().smoe_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def describe(self) -> str:
        buf = C.create_string_buffer(1024)
        _check(lib().smoe_ctx_describe(self.handle, buf, 1024), "smoe_ctx_describe")
        return buf.value.decode()

    def set_profile_events(self, events):
        """events: list of up to 4 torch.cuda.Event (already recorded once), or []."""
        n = len(events)
        arr = (C.c_void_p * max(n, 1))(*[e.cuda_event for e in events])
        _check(lib().smoe_set_profile_events(self.handle, arr, n), "smoe_set_profile_events")

    def set_stack_wait(self, grid_wait_ns: int = 0, stall_layer: int = -1):
        """Failure-detection hook of moe_decode_stack (smoe_set_stack_wait):
        the grid-wide wait limit (0: two seconds) and a layer whose first
        grid-wide wait is made to run out (-1: none)."""
        _check(lib().smoe_set_stack_wait(self.handle, int(grid_wait_ns), int(stall_layer)), "smoe_set_stack_wait")

    def stack_workspace_bytes(self, n_layers: int) -> int:
        """Workspace bytes of moe_decode_stack over n_layers layers (0: not available)."""
        return int(lib().smoe_stack_workspace_bytes(self.handle, int(n_layers)))

    def workspace_bytes(self, T: int) -> int:
        return int(lib().smoe_workspace_bytes(self.handle, int(T)))


def set_slot_table(ctx: Context, layer: int, host_table: np.ndarray, stream=None):
    tab = np.ascontiguousarray(host_table, np.int32)
    _check(lib().set_slot_table(ctx.handle, int(layer), tab.ctypes.data, _stream(stream)), "set_slot_table")


def moe_route(ctx: Context, W_r, w_s, x, ids, w, gate, workspace, logit_bias=None, stream=None):
    import torch
    sh = ctx.shape
    T = x.shape[0]
    _check(lib().moe_route(ctx.handle, _dev(W_r, "W_r", torch.bfloat16, sh.E * sh.H),
                           _dev(w_s, "w_s", torch.bfloat16, sh.H), _dev(x, "x", torch.bfloat16, T * sh.H), T,
                           _dev(logit_bias, "logit_bias", torch.float32, sh.E),
                           _dev(ids, "ids", torch.int32, T * sh.k), _dev(w, "w", torch.float32, T * sh.k),
                           _dev(gate, "gate", torch.float32, T), _dev(workspace, "workspace"), _nbytes(workspace),
                           _stream(stream)), "moe_route")


def _forward_args(ctx: Context, x, ids, w, gate, pool, shared_blob, out, residual):
    """Checked addresses of the arguments moe_forward and its variants share."""
    import torch
    sh = ctx.shape
    T = x.shape[0]
    return (_dev(x, "x", torch.bfloat16, T * sh.H), T, _dev(ids, "ids", torch.int32, T * sh.k),
            _dev(w, "w", torch.float32, T * sh.k), _dev(gate, "gate", torch.float32, T),
            _dev(pool, "pool"), _nbytes(pool),
            _dev(shared_blob, "shared_blob", min_bytes=ctx.layout.blob_bytes),
            _dev(residual, "residual", torch.bfloat16, T * sh.H), _dev(out, "out", torch.bfloat16, T * sh.H))


def moe_forward(ctx: Context, layer: int, x, ids, w, gate, pool, shared_blob, out, workspace, err,
                residual=None, stream=None):
    import torch
    a = _forward_args(ctx, x, ids, w, gate, pool, shared_blob, out, residual)
    _check(lib().moe_forward(ctx.handle, int(layer), *a, _dev(workspace, "workspace"), _nbytes(workspace),
                             _dev(err, "err", torch.int32, 1), _stream(stream)), "moe_forward")


def moe_forward_debug(ctx: Context, layer: int, x, ids, w, gate, pool, shared_blob, out, err, residual=None,
                      stream=None):
    """The plain per-token CUDA path (for checking the fast kernels)."""
    import torch
    a = _forward_args(ctx, x, ids, w, gate, pool, shared_blob, out, residual)
    _check(lib().moe_forward_debug(ctx.handle, int(layer), *a, _dev(err, "err", torch.int32, 1), _stream(stream)),
           "moe_forward_debug")


def moe_forward_noalloc(ctx: Context, layer: int, x, ids, w, gate, pool, shared_blob, out, err,
                        residual=None, stream=None):
    """moe_forward without a workspace (scratch inside the library); T <= 8."""
    import torch
    a = _forward_args(ctx, x, ids, w, gate, pool, shared_blob, out, residual)
    _check(lib().moe_forward_noalloc(ctx.handle, int(layer), *a, _dev(err, "err", torch.int32, 1), _stream(stream)),
           "moe_forward_noalloc")


def moe_decode_stack(ctx: Context, first_layer: int, Wr, ws, shared_blobs, xs, ids, w, gate, pool, workspace, err,
                     logit_bias=None, stream=None):
    """One token through len(Wr) layers in one launch. Wr, ws, shared_blobs:
    per-layer device tensors; xs bf16 [L + 1, H] (xs[0] the input); ids, w
    [L, k]; gate [L]."""
    import torch
    sh = ctx.shape
    n = len(Wr)
    if len(ws) != n or len(shared_blobs) != n:
        raise ValueError("Wr, ws and shared_blobs must have one entry per layer")
    arr = lambda ts: (C.c_void_p * n)(*ts)
    _check(lib().moe_decode_stack(ctx.handle, int(first_layer), n,
                                  arr([_dev(t, "Wr[%d]" % i, torch.bfloat16, sh.E * sh.H) for i, t in enumerate(Wr)]),
                                  arr([_dev(t, "ws[%d]" % i, torch.bfloat16, sh.H) for i, t in enumerate(ws)]),
                                  arr([_dev(t, "shared_blobs[%d]" % i, min_bytes=ctx.layout.blob_bytes)
                                       for i, t in enumerate(shared_blobs)]),
                                  _dev(logit_bias, "logit_bias", torch.float32, sh.E),
                                  _dev(xs, "xs", torch.bfloat16, (n + 1) * sh.H), _dev(ids, "ids", torch.int32, n * sh.k),
                                  _dev(w, "w", torch.float32, n * sh.k), _dev(gate, "gate", torch.float32, n),
                                  _dev(pool, "pool"), _nbytes(pool), _dev(workspace, "workspace"), _nbytes(workspace),
                                  _dev(err, "err", torch.int32, 1), _stream(stream)),
           "moe_decode_stack")


class Cache:
    """Streaming slot pool (smoe_cache): the context's device slots as a cache
    over every expert's packed blob in host memory. host_store: a host uint8
    tensor [n_layers * E * stride] (pinned for full-rate copies); pool: the
    context's device pool. Both must outlive the cache."""

    def __init__(self, ctx: Context, host_store, pool, stream=None):
        self.ctx, self.host_store, self.pool = ctx, host_store, pool
        h = C.c_void_p()
        _check(lib().smoe_cache_create(ctx.handle, C.c_void_p(host_store.data_ptr()),
                                       host_store.numel() * host_store.element_size(), _ptr(pool),
                                       pool.numel() * pool.element_size(), _stream(stream), C.byref(h)),
               "smoe_cache_create")
        self.handle = h.value

    def prepare(self, layer: int, ids: np.ndarray, stream=None) -> tuple[int, int]:
        """Makes the experts in ids (host int array) of `layer` resident; returns (hits, misses)."""
        a = np.ascontiguousarray(ids, np.int32).ravel()
        hits, misses = C.c_int32(0), C.c_int32(0)
        _check(lib().smoe_cache_prepare(self.handle, int(layer), a.ctypes.data, a.size, _stream(stream),
                                        C.byref(hits), C.byref(misses)), "smoe_cache_prepare")
        return int(hits.value), int(misses.value)

    def stats(self) -> tuple[int, int, int]:
        """(hits, misses, bytes copied) since creation."""
        h, m, b = C.c_uint64(0), C.c_uint64(0), C.c_uint64(0)
        _check(lib().smoe_cache_stats(self.handle, C.byref(h), C.byref(m), C.byref(b)), "smoe_cache_stats")
        return int(h.value), int(m.value), int(b.value)

    def close(self):
        if self.handle:
            lib().smoe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def cache_simulate(n_layers: int, E: int, n_slots: int, requests) -> tuple[np.ndarray, int, int]:
    """The replacement policy alone on the host. requests: list of (layer, ids).
    Returns (slot of every requested id in order, hits, misses)."""
    flat = []
    for layer, ids in requests:
        ids = list(map(int, ids))
        flat += [int(layer), len(ids)] + ids
    req = np.asarray(flat, np.int32)
    out = np.zeros(sum(len(ids) for _, ids in requests), np.int32)
    h, m = C.c_int64(0), C.c_int64(0)
    _check(lib().smoe_cache_simulate(int(n_layers), int(E), int(n_slots), req.ctypes.data, len(requests),
                                     out.ctypes.data, C.byref(h), C.byref(m)), "smoe_cache_simulate")
    return out, int(h.value), int(m.value)


def gdn_step(nk: int, nv: int, q, k, v, g, beta, state, out, scale: float = 0.0, stream=None):
    """T Gated DeltaNet recurrence steps on `state` in place. q, k bf16
    [T, B, nk, dk]; v, out bf16 [T, B, nv, dv]; g, beta fp32 [T, B, nv];
    state fp32 [B, nv, dv, dk]. scale <= 0 means 1 / sqrt(dk)."""
    import torch
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v: expected [T, B, heads, width]")
    T, B, _, dk = q.shape
    dv = v.shape[3]
    sh = GdnShape(int(nk), int(nv), int(dk), int(dv))
    _check(lib().gdn_step(C.byref(sh), int(B), int(T), _dev(q, "q", torch.bfloat16, T * B * nk * dk),
                          _dev(k, "k", torch.bfloat16, T * B * nk * dk), _dev(v, "v", torch.bfloat16, T * B * nv * dv),
                          _dev(g, "g", torch.float32, T * B * nv), _dev(beta, "beta", torch.float32, T * B * nv),
                          float(scale), _dev(state, "state", torch.float32, B * nv * dv * dk),
                          _dev(out, "out", torch.bfloat16, T * B * nv * dv), _stream(stream)), "gdn_step")


def check(err, stream=None) -> int:
    """Synchronises, returns the device error code (0 if none) and clears it."""
    code = C.c_int32(0)
    rc = lib().smoe_check(_ptr(err), C.byref(code), _stream(stream))
    if rc not in (OK, EDEVICE):
        raise SmoeError(rc, "smoe_check")
    return int(code.value)
