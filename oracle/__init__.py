"""Python front of the CPU oracle (``oracle/smoe_oracle.c``).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. The
CUDA library never imports, links or calls it, and it never imports the CUDA
library. All arithmetic lives in the C file; this wrapper only marshals numpy
arrays (inputs come from ``synthetic``).

Functions and the passages they follow are documented in ``smoe_oracle.c``
and ``gdn_oracle.c`` (the Gated DeltaNet recurrence step).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None

_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")


class OrcExpert(C.Structure):
    _fields_ = [("q", C.c_void_p * 3), ("s", C.c_void_p * 3), ("b", C.c_void_p * 3)]


def lib():
    global _lib
    if _lib is None:
        # a test may point this at a deliberately broken build of the oracle
        path = os.environ.get("SMOE_ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        L.orc_bf16_to_f64.argtypes = [C.c_uint16]
        L.orc_bf16_to_f64.restype = C.c_double
        L.orc_f16_to_f64.argtypes = [C.c_uint16]
        L.orc_f16_to_f64.restype = C.c_double
        L.orc_f64_to_bf16.argtypes = [C.c_double]
        L.orc_f64_to_bf16.restype = C.c_uint16
        L.orc_f64_to_f16.argtypes = [C.c_double]
        L.orc_f64_to_f16.restype = C.c_uint16
        L.orc_dequant_mlx.argtypes = [_u32p, _u16p, _u16p, C.c_int, C.c_int, _f64p]
        L.orc_dequant_mlx.restype = None
        L.orc_quantize_mlx.argtypes = [_f64p, C.c_int, C.c_int, _u32p, _u16p, _u16p]
        L.orc_quantize_mlx.restype = None
        L.orc_route.argtypes = [_u16p, C.c_int, C.c_int, _u16p, _u16p, C.c_int, C.c_void_p,
                                C.c_int, _i32p, _f64p, _f64p, C.c_void_p]
        L.orc_route.restype = None
        L.orc_moe_combine.argtypes = [C.c_int] * 5 + [_u16p, _i32p, _f64p, _f64p, C.c_void_p,
                                                      C.c_int, C.c_void_p, _f64p, _u16p]
        L.orc_moe_combine.restype = C.c_int
        L.orc_residual_bf16.argtypes = [_u16p, _f64p, C.c_size_t, _u16p]
        L.orc_residual_bf16.restype = None
        L.orc_blob_bytes.argtypes = [C.c_int, C.c_int]
        L.orc_blob_bytes.restype = C.c_uint64
        L.orc_blob_to_mlx.argtypes = [_u8p, C.c_int, C.c_int] + [_u32p, _u16p, _u16p] * 3
        L.orc_blob_to_mlx.restype = None
        L.orc_moe_combine_pool.argtypes = [C.c_int] * 5 + [_u16p, _i32p, _f64p, _f64p,
                                                           C.c_void_p, C.c_uint64, C.c_int64,
                                                           _i32p, C.c_void_p, _f64p, _u16p]
        L.orc_moe_combine_pool.restype = C.c_int
        L.orc_dequant_mlx8.argtypes = [_u32p, _u16p, _u16p, C.c_int, C.c_int, _f64p]
        L.orc_dequant_mlx8.restype = None
        L.orc_quantize_mlx8.argtypes = [_f64p, C.c_int, C.c_int, _u32p, _u16p, _u16p]
        L.orc_quantize_mlx8.restype = None
        L.orc_moe_combine_dense.argtypes = [C.c_int] * 5 + [_u16p, _i32p, _f64p, _f64p] + [C.c_void_p] * 3 + \
            [C.c_int] + [_f64p] * 3 + [_f64p, _u16p]
        L.orc_moe_combine_dense.restype = C.c_int
        L.orc_blob_bytes8.argtypes = [C.c_int, C.c_int]
        L.orc_blob_bytes8.restype = C.c_uint64
        L.orc_blob_to_mlx8.argtypes = [_u8p, C.c_int, C.c_int] + [_u32p, _u16p, _u16p] * 3
        L.orc_blob_to_mlx8.restype = None
        L.orc_gdn_step.argtypes = [C.c_int] * 6 + [_u16p, _u16p, _u16p, _f64p, _f64p, C.c_double, _f64p, _f64p]
        L.orc_gdn_step.restype = C.c_int
        _lib = L
    return _lib


# ------------------------------------------------------------------ helpers

def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).ravel()
    f = lib().orc_bf16_to_f64
    return np.array([f(int(v)) for v in b], dtype=np.float64).reshape(np.shape(bits))


def f16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).ravel()
    f = lib().orc_f16_to_f64
    return np.array([f(int(v)) for v in b], dtype=np.float64).reshape(np.shape(bits))


def f64_to_bf16(vals) -> np.ndarray:
    v = np.asarray(vals, dtype=np.float64).ravel()
    f = lib().orc_f64_to_bf16
    return np.array([f(float(a)) for a in v], dtype=np.uint16).reshape(np.shape(vals))


def f64_to_f16(vals) -> np.ndarray:
    v = np.asarray(vals, dtype=np.float64).ravel()
    f = lib().orc_f64_to_f16
    return np.array([f(float(a)) for a in v], dtype=np.uint16).reshape(np.shape(vals))


def dequant(q, s, b) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint32)
    rows, cols = q.shape[0], q.shape[1] * 8
    W = np.empty((rows, cols), np.float64)
    lib().orc_dequant_mlx(q, np.ascontiguousarray(s, np.uint16),
                          np.ascontiguousarray(b, np.uint16), rows, cols, W)
    return W


def quantize(W):
    W = np.ascontiguousarray(W, np.float64)
    rows, cols = W.shape
    q = np.empty((rows, cols // 8), np.uint32)
    s = np.empty((rows, cols // 64), np.uint16)
    b = np.empty((rows, cols // 64), np.uint16)
    lib().orc_quantize_mlx(W, rows, cols, q, s, b)
    return q, s, b


def route(x, Wr, ws, k, bias=None, want_probs=False):
    """Returns ids [T,k] int32, w [T,k] f64, gate [T] f64 (, probs [T,E])."""
    x = np.ascontiguousarray(x, np.uint16)
    Wr = np.ascontiguousarray(Wr, np.uint16)
    ws = np.ascontiguousarray(ws, np.uint16)
    T, H = x.shape
    E = Wr.shape[0]
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    gate = np.empty((T,), np.float64)
    probs = np.empty((T, E), np.float64) if want_probs else None
    bias_arr = None if bias is None else np.ascontiguousarray(bias, np.float32)
    lib().orc_route(x, T, H, Wr, ws, E,
                    None if bias_arr is None else bias_arr.ctypes.data, k, ids, w, gate,
                    None if probs is None else probs.ctypes.data)
    return (ids, w, gate, probs) if want_probs else (ids, w, gate)


def _expert_struct(tr):
    arrs = [np.ascontiguousarray(a) for a in tr.arrays()]
    st = OrcExpert()
    for m in range(3):
        st.q[m] = arrs[3 * m].ctypes.data
        st.s[m] = arrs[3 * m + 1].ctypes.data
        st.b[m] = arrs[3 * m + 2].ctypes.data
    return st, arrs


def combine(x, ids, w, gate, experts: dict, shared, E: int, I: int, I_shared: int):
    """Layer output given routing. experts: {e: ExpertTriples} for every e in ids.

    Returns (out64 [T,H] float64, out_bf16 [T,H] uint16 bits)."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    k = ids.shape[1]
    keep = []
    table = (OrcExpert * E)()
    for e, tr in experts.items():
        st, arrs = _expert_struct(tr)
        table[e] = st
        keep.append(arrs)
    sh, sharrs = _expert_struct(shared)
    keep.append(sharrs)
    out64 = np.empty((T, H), np.float64)
    outb = np.empty((T, H), np.uint16)
    rc = lib().orc_moe_combine(T, H, k, I, I_shared, x, np.ascontiguousarray(ids, np.int32),
                               np.ascontiguousarray(w, np.float64),
                               np.ascontiguousarray(gate, np.float64),
                               C.addressof(table), E, C.addressof(sh), out64, outb)
    if rc != 0:
        raise ValueError("oracle: a routed expert was not provided")
    return out64, outb


def combine_pool(x, ids, w, gate, pool: np.ndarray, stride: int, n_slots: int,
                 table_row: np.ndarray, shared_blob: np.ndarray, E: int, I: int):
    """Layer output with experts read from blob bytes through a slot table."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    k = ids.shape[1]
    out64 = np.empty((T, H), np.float64)
    outb = np.empty((T, H), np.uint16)
    pool = np.ascontiguousarray(pool, np.uint8)
    shared_blob = np.ascontiguousarray(shared_blob, np.uint8)
    rc = lib().orc_moe_combine_pool(T, H, k, I, E, x, np.ascontiguousarray(ids, np.int32),
                                    np.ascontiguousarray(w, np.float64),
                                    np.ascontiguousarray(gate, np.float64),
                                    pool.ctypes.data, stride, n_slots,
                                    np.ascontiguousarray(table_row, np.int32),
                                    shared_blob.ctypes.data, out64, outb)
    if rc != 0:
        raise ValueError("oracle: invalid slot or expert id")
    return out64, outb


def blob_bytes(H: int, I: int) -> int:
    return int(lib().orc_blob_bytes(H, I))


def blob_to_mlx(blob: np.ndarray, H: int, I: int):
    """Parse one expert blob -> list of 9 arrays in ExpertTriples order."""
    gq = np.empty((I, H // 8), np.uint32); uq = np.empty_like(gq)
    dq = np.empty((H, I // 8), np.uint32)
    gs = np.empty((I, H // 64), np.uint16); gb = np.empty_like(gs)
    us = np.empty_like(gs); ub = np.empty_like(gs)
    ds = np.empty((H, I // 64), np.uint16); db = np.empty_like(ds)
    lib().orc_blob_to_mlx(np.ascontiguousarray(blob, np.uint8), H, I,
                          gq, gs, gb, uq, us, ub, dq, ds, db)
    return [gq, gs, gb, uq, us, ub, dq, ds, db]


# ------------------------------------------------------------ 8-bit experts

def dequant8(q, s, b) -> np.ndarray:
    """8-bit MLX triple (4 values per word) -> fp64 weights [rows, cols]."""
    q = np.ascontiguousarray(q, np.uint32)
    rows, cols = q.shape[0], q.shape[1] * 4
    W = np.empty((rows, cols), np.float64)
    lib().orc_dequant_mlx8(q, np.ascontiguousarray(s, np.uint16), np.ascontiguousarray(b, np.uint16), rows, cols, W)
    return W


def quantize8(W):
    W = np.ascontiguousarray(W, np.float64)
    rows, cols = W.shape
    q = np.empty((rows, cols // 4), np.uint32)
    s = np.empty((rows, cols // 64), np.uint16)
    b = np.empty((rows, cols // 64), np.uint16)
    lib().orc_quantize_mlx8(W, rows, cols, q, s, b)
    return q, s, b


def combine_dense(x, ids, w, gate, dense: dict, shared_dense, E: int, I: int, I_shared: int):
    """Layer output given routing, for experts given as dense fp64 (G, U, D)
    {e: (G [I,H], U [I,H], D [H,I])} and the shared expert's (G, U, D).

    Returns (out64 [T,H] float64, out_bf16 [T,H] uint16 bits)."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    k = ids.shape[1]
    keep = {e: tuple(np.ascontiguousarray(m, np.float64) for m in gud) for e, gud in dense.items()}
    ptrs = [(C.c_void_p * E)() for _ in range(3)]
    for e, gud in keep.items():
        for m in range(3):
            ptrs[m][e] = gud[m].ctypes.data
    Gs, Us, Ds = (np.ascontiguousarray(m, np.float64) for m in shared_dense)
    out64 = np.empty((T, H), np.float64)
    outb = np.empty((T, H), np.uint16)
    rc = lib().orc_moe_combine_dense(T, H, k, I, I_shared, x, np.ascontiguousarray(ids, np.int32),
                                     np.ascontiguousarray(w, np.float64), np.ascontiguousarray(gate, np.float64),
                                     C.addressof(ptrs[0]), C.addressof(ptrs[1]), C.addressof(ptrs[2]), E,
                                     Gs, Us, Ds, out64, outb)
    if rc != 0:
        raise ValueError("oracle: a routed expert was not provided")
    return out64, outb


def dense_of8(tr):
    """(G, U, D) of an 8-bit ExpertTriples."""
    return (dequant8(tr.gate_q, tr.gate_s, tr.gate_b), dequant8(tr.up_q, tr.up_s, tr.up_b),
            dequant8(tr.down_q, tr.down_s, tr.down_b))


def combine8(x, ids, w, gate, experts: dict, shared, E: int, I: int, I_shared: int):
    """combine() for 8-bit experts: each one dequantised, then combine_dense."""
    return combine_dense(x, ids, w, gate, {e: dense_of8(tr) for e, tr in experts.items()}, dense_of8(shared),
                         E, I, I_shared)


def combine_pool8(x, ids, w, gate, pool: np.ndarray, stride: int, n_slots: int, table_row: np.ndarray,
                  shared_blob: np.ndarray, E: int, I: int):
    """combine_pool() for 8-bit blobs: each named expert read from its slot's
    blob bytes by the oracle's 8-bit reader, dequantised, then combine_dense."""
    x = np.ascontiguousarray(x, np.uint16)
    H = x.shape[1]

    def dense_at(blob):
        q = blob_to_mlx8(blob, H, I)
        return dequant8(q[0], q[1], q[2]), dequant8(q[3], q[4], q[5]), dequant8(q[6], q[7], q[8])
    dense = {}
    for e in np.unique(ids):
        slot = int(table_row[int(e)])
        if not 0 <= slot < n_slots:
            raise ValueError("oracle: invalid slot or expert id")
        dense[int(e)] = dense_at(pool[slot * stride:(slot + 1) * stride])
    return combine_dense(x, ids, w, gate, dense, dense_at(shared_blob), E, I, I)


def blob_bytes8(H: int, I: int) -> int:
    return int(lib().orc_blob_bytes8(H, I))


def blob_to_mlx8(blob: np.ndarray, H: int, I: int):
    """Parse one 8-bit expert blob -> list of 9 arrays in ExpertTriples order."""
    gq = np.empty((I, H // 4), np.uint32); uq = np.empty_like(gq)
    dq = np.empty((H, I // 4), np.uint32)
    gs = np.empty((I, H // 64), np.uint16); gb = np.empty_like(gs)
    us = np.empty_like(gs); ub = np.empty_like(gs)
    ds = np.empty((H, I // 64), np.uint16); db = np.empty_like(ds)
    lib().orc_blob_to_mlx8(np.ascontiguousarray(blob, np.uint8), H, I, gq, gs, gb, uq, us, ub, dq, ds, db)
    return [gq, gs, gb, uq, us, ub, dq, ds, db]


def residual(x, y64):
    x = np.ascontiguousarray(x, np.uint16)
    out = np.empty_like(x)
    lib().orc_residual_bf16(x, np.ascontiguousarray(y64, np.float64), x.size, out)
    return out


# --------------------------------------------------------- whole-layer helper

def layer(wl, seed_layer: int, x, Wr, ws, bias=None, want_probs=False):
    """Route then combine one layer of workload ``wl`` (synthetic.Workload),
    regenerating only the experts that the routing selects."""
    import synthetic
    r = route(x, Wr, ws, wl.k, bias=bias, want_probs=want_probs)
    ids, w, gate = r[0], r[1], r[2]
    experts = {int(e): synthetic.expert_triples(wl.seed, seed_layer, int(e), wl.H, wl.I)
               for e in np.unique(ids)}
    shared = synthetic.expert_triples(wl.seed, seed_layer, None, wl.H, wl.I_shared)
    out64, outb = combine(x, ids, w, gate, experts, shared, wl.E, wl.I, wl.I_shared)
    return dict(ids=ids, w=w, gate=gate, out64=out64, out_bf16=outb,
                probs=(r[3] if want_probs else None))


# ------------------------------------------------------- Gated DeltaNet step

def gdn_step(q, k, v, g, beta, state, scale=None):
    """One Gated DeltaNet recurrence step per token (gdn_oracle.c): q, k bf16
    bits [T][B][n_k][d_k], v [T][B][n_v][d_v], g, beta [T][B][n_v] (float),
    state [B][n_v][d_v][d_k] float64 (not modified). scale defaults to
    d_k ** -0.5. Returns (new state, out [T][B][n_v][d_v] float64)."""
    q = np.ascontiguousarray(q, np.uint16)
    k = np.ascontiguousarray(k, np.uint16)
    v = np.ascontiguousarray(v, np.uint16)
    T, B, nk, dk = q.shape
    nv, dv = v.shape[2], v.shape[3]
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    out = np.empty((T, B, nv, dv), np.float64)
    sc = dk ** -0.5 if scale is None else float(scale)
    rc = lib().orc_gdn_step(T, B, nk, nv, dk, dv, q, k, v, np.ascontiguousarray(g, np.float64),
                            np.ascontiguousarray(beta, np.float64), sc, S, out)
    if rc != 0:
        raise ValueError("oracle: bad Gated DeltaNet shape")
    return S, out
