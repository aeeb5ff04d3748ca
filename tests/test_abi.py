"""C-ABI library checks that need no GPU: it loads, exports every declared
symbol, reports the blob layout, and its host packer writes blobs that the
oracle's independently written reader parses back to the source triples."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import int4_routed_expert_router_gb300 as smoe
import oracle
import synthetic
from int4_routed_expert_router_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "smoe.h")).read()
    return re.findall(r"SMOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) >= {"pack_experts", "set_slot_table", "moe_route", "moe_forward"}
    L = smoe.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(smoe.EXPORTS)


def test_layout_sizes():
    lay = smoe.layout_of(smoe.make_shape(2048, 512, 10, 512))
    assert lay.blob_bytes == 1769472 == 432 * 4096
    assert lay.gu_bytes == 2 * 589824 and lay.down_offset == lay.gu_bytes and lay.down_bytes == 589824
    assert (lay.atom_bytes, lay.atom_rows, lay.group) == (576, 16, 64)
    tiny = smoe.layout_of(smoe.make_shape(256, 16, 4, 64))
    assert tiny.blob_bytes == 27648 == oracle.blob_bytes(256, 64)


@pytest.mark.parametrize("shape,status", [
    ((2048, 512, 10, 512, 256), smoe.ENOTSUP),     # I_shared != I
    ((2000, 512, 10, 512, 512), smoe.ENOTSUP),     # H not a multiple of 256
    ((4096, 512, 10, 512, 512), smoe.ENOTSUP),     # H above what the decode kernel stages
    ((2048, 512, 10, 1024, 1024), smoe.ENOTSUP),   # I too large for the kernels
    ((2048, 8, 10, 512, 512), smoe.ENOTSUP),       # k > E
    ((2048, 512, 0, 512, 512), smoe.EINVAL),
])
def test_layout_rejects_bad_shapes(shape, status):
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.layout_of(smoe.make_shape(*shape))
    assert ei.value.status == status


def _triples(wl, layer, e):
    return synthetic.expert_triples(wl.seed, layer, e, wl.H, wl.I).arrays()


@pytest.mark.parametrize("name", ["tiny", "decode80b"])
def test_host_pack_round_trips_through_oracle_reader(name):
    wl = synthetic.WORKLOADS[name]
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I)
    stride = smoe.layout_of(shape).blob_bytes
    srcs = [_triples(wl, 0, e) for e in (3, 7)]
    pool = np.zeros(3 * stride, np.uint8)
    smoe.pack_experts(shape, srcs, [2, 0], pool, pool.size, smoe.HOST)
    for src, slot in zip(srcs, [2, 0]):
        back = oracle.blob_to_mlx(pool[slot * stride:(slot + 1) * stride], wl.H, wl.I)
        for a, b in zip(src, back):
            assert np.array_equal(a, b)
    assert not pool[stride:2 * stride].any()        # slot 1 untouched


def test_host_pack_beyond_4GiB_offsets():
    wl = synthetic.WORKLOADS["decode80b"]
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I)
    stride = smoe.layout_of(shape).blob_bytes
    slot = (1 << 32) // stride + 5                  # offset past 4 GiB
    pool = np.empty((slot + 1) * stride, np.uint8)  # untouched pages cost no memory
    src = _triples(wl, 1, 42)
    smoe.pack_experts(shape, [src], [slot], pool, pool.size, smoe.HOST)
    back = oracle.blob_to_mlx(pool[slot * stride:], wl.H, wl.I)
    for a, b in zip(src, back):
        assert np.array_equal(a, b)
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.pack_experts(shape, [src], [slot + 1], pool, pool.size, smoe.HOST)
    assert ei.value.status == smoe.ENOMEM
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.pack_experts(shape, [src], [-1], pool, pool.size, smoe.HOST)
    assert ei.value.status == smoe.ERANGE


def test_oracle_pool_path_is_slot_permutation_invariant():
    """Cache or disk, same answer: the oracle reading experts through any slot
    permutation of the pool gives bit-identical output, equal to reading the
    triples directly."""
    wl = synthetic.WORKLOADS["tiny"]
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I)
    stride = smoe.layout_of(shape).blob_bytes
    x = synthetic.activations(wl.seed, wl.T, wl.H)
    Wr = synthetic.router_weights(wl.seed, 0, wl.E, wl.H)
    ws = synthetic.shared_gate_weights(wl.seed, 0, wl.H)
    ids, w, gate = oracle.route(x, Wr, ws, wl.k)
    direct = oracle.layer(wl, 0, x, Wr, ws)
    shared = np.zeros(stride, np.uint8)
    smoe.pack_experts(shape, [synthetic.expert_triples(wl.seed, 0, None, wl.H, wl.I).arrays()], [0],
                      shared, stride, smoe.HOST)
    outs = []
    for seed in range(3):
        table = np.random.default_rng(seed).permutation(2 * wl.E)[:wl.E].astype(np.int32)
        pool = np.zeros(2 * wl.E * stride, np.uint8)
        smoe.pack_experts(shape, [_triples(wl, 0, e) for e in range(wl.E)], table.tolist(), pool, pool.size,
                          smoe.HOST)
        o64, ob = oracle.combine_pool(x, ids, w, gate, pool, stride, 2 * wl.E, table, shared, wl.E, wl.I)
        outs.append(o64)
        assert np.array_equal(ob, direct["out_bf16"])
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    assert np.array_equal(outs[0], direct["out64"])


def test_binding_refuses_host_tensors_before_any_call():
    """Device arguments must be CUDA tensors: a host tensor (or a numpy array)
    is refused by the binding, so no kernel is ever handed a host address."""
    import types

    import torch
    shape = smoe.make_shape(256, 16, 4, 64)
    ctx = types.SimpleNamespace(handle=None, shape=shape, layout=smoe.layout_of(shape))
    T, H, k = 2, 256, 4
    x = torch.zeros((T, H), dtype=torch.bfloat16)
    ids = torch.zeros((T, k), dtype=torch.int32)
    w = torch.zeros((T, k), dtype=torch.float32)
    gate = torch.zeros(T, dtype=torch.float32)
    blob = torch.zeros(int(ctx.layout.blob_bytes), dtype=torch.uint8)
    err = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="x: expected a CUDA tensor"):
        smoe.moe_forward(ctx, 0, x, ids, w, gate, blob, blob, x, blob, err)
    with pytest.raises(ValueError, match="W_r: expected a CUDA tensor"):
        smoe.moe_route(ctx, np.zeros((16, H), np.uint16), x[0], x, ids, w, gate, blob)
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        smoe.moe_forward_noalloc(ctx, 0, x, ids, w, gate, blob, blob, x, err)


# --------------------------------------------------------------- 8-bit experts

def test_layout_8_bit():
    lay = smoe.layout_of(smoe.make_shape(2048, 512, 10, 512, bits=8))
    assert lay.atom_bytes == 1088 and lay.blob_bytes == 3342336 == oracle.blob_bytes8(2048, 512)
    assert lay.down_offset == lay.gu_bytes == 64 * 32 * 1088 and lay.down_bytes == 128 * 8 * 1088
    assert smoe.layout_of(smoe.make_shape(256, 16, 4, 64, bits=8)).blob_bytes == oracle.blob_bytes8(256, 64)
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.layout_of(smoe.make_shape(2048, 512, 10, 512, bits=6))
    assert ei.value.status == smoe.ENOTSUP


@pytest.mark.parametrize("name", ["tiny", "decode80b"])
def test_host_pack_8_bit_round_trips_through_oracle_reader(name):
    """The library's 8-bit packer and the oracle's independently written
    8-bit reader agree on every byte of the two-plane atoms."""
    wl = synthetic.WORKLOADS[name]
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I, bits=8)
    stride = smoe.layout_of(shape).blob_bytes
    srcs = [synthetic.expert_triples(wl.seed, 0, e, wl.H, wl.I, bits=8).arrays() for e in (3, 7)]
    pool = np.zeros(3 * stride, np.uint8)
    smoe.pack_experts(shape, srcs, [2, 0], pool, pool.size, smoe.HOST)
    for src, slot in zip(srcs, [2, 0]):
        back = oracle.blob_to_mlx8(pool[slot * stride:(slot + 1) * stride], wl.H, wl.I)
        for a, b in zip(src, back):
            assert np.array_equal(a, b)
    assert not pool[stride:2 * stride].any()
    # the low-nibble plane of an 8-bit blob is the 4-bit blob of the low nibbles
    lo = [a & np.uint32(0x0F0F0F0F) if i % 3 == 0 else a for i, a in enumerate(srcs[0])]
    lo4 = [_mlx8_to_4(a) if i % 3 == 0 else a for i, a in enumerate(lo)]
    s4 = smoe.make_shape(wl.H, wl.E, wl.k, wl.I)
    blob4 = np.zeros(smoe.layout_of(s4).blob_bytes, np.uint8)
    smoe.pack_experts(s4, [lo4], [0], blob4, blob4.size, smoe.HOST)
    atoms8 = pool[2 * stride:3 * stride].reshape(-1, 1088)
    atoms4 = blob4.reshape(-1, 576)
    assert np.array_equal(atoms8[:, :512], atoms4[:, :512]) and np.array_equal(atoms8[:, 1024:], atoms4[:, 512:])


def _mlx8_to_4(q8):
    """8-bit MLX words holding values 0..15 -> 4-bit MLX words (8 per word)."""
    v = np.stack([(q8 >> np.uint32(8 * j)) & np.uint32(15) for j in range(4)], axis=-1).reshape(q8.shape[0], -1)
    v = v.reshape(v.shape[0], -1, 8).astype(np.uint32)
    return sum(v[:, :, j] << np.uint32(4 * j) for j in range(8)).astype(np.uint32)


def test_oracle_pool_path_8_bit_is_slot_permutation_invariant():
    """Cache or disk, same answer, for 8-bit experts: read through any slot
    permutation of an 8-bit pool (the library's packer, the oracle's reader),
    the layer is bit-identical, and equal to the layer on the triples."""
    wl = synthetic.WORKLOADS["tiny"]
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I, bits=8)
    stride = smoe.layout_of(shape).blob_bytes
    x = synthetic.activations(wl.seed, wl.T, wl.H)
    ids, w, gate = oracle.route(x, synthetic.router_weights(wl.seed, 0, wl.E, wl.H),
                                synthetic.shared_gate_weights(wl.seed, 0, wl.H), wl.k)
    trip = {e: synthetic.expert_triples(wl.seed, 0, e, wl.H, wl.I, bits=8) for e in range(wl.E)}
    sh_t = synthetic.expert_triples(wl.seed, 0, None, wl.H, wl.I, bits=8)
    direct, _ = oracle.combine8(x, ids, w, gate, trip, sh_t, wl.E, wl.I, wl.I)
    shared = np.zeros(stride, np.uint8)
    smoe.pack_experts(shape, [sh_t.arrays()], [0], shared, stride, smoe.HOST)
    for seed in range(3):
        table = np.random.default_rng(seed).permutation(2 * wl.E)[:wl.E].astype(np.int32)
        pool = np.zeros(2 * wl.E * stride, np.uint8)
        smoe.pack_experts(shape, [trip[e].arrays() for e in range(wl.E)], table.tolist(), pool, pool.size,
                          smoe.HOST)
        o64, _ = oracle.combine_pool8(x, ids, w, gate, pool, stride, 2 * wl.E, table, shared, wl.E, wl.I)
        assert np.array_equal(o64, direct)


def test_pack_refuses_misaligned_buffers_before_any_work():
    """A device pool that does not start on a 16-byte boundary (say an offset
    view of a buffer) is refused with EINVAL before any copy or launch, as
    are q words not on a 4-byte and s/b not on a 2-byte boundary (host or
    device). The addresses are never dereferenced: the check comes first."""
    wl = synthetic.WORKLOADS["tiny"]
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I)
    stride = smoe.layout_of(shape).blob_bytes
    L = smoe.lib()

    def call(pool_addr, q_off=0, s_off=0, where=smoe.DEVICE):
        src = smoe.ExpertSrc()
        for m in range(3):
            src.q[m] = 0x100000 + 0x1000 * m + q_off
            src.s[m] = 0x200000 + 0x1000 * m + s_off
            src.b[m] = 0x300000 + 0x1000 * m
        slots = (C.c_int64 * 1)(0)
        return L.pack_experts(C.byref(shape), C.byref(src), 1, slots, pool_addr, 4 * stride, where, None)

    assert call(0x400008) == smoe.EINVAL                    # device pool 8 bytes past a boundary
    assert call(0x400010, q_off=2) == smoe.EINVAL           # q words not 4-byte aligned
    assert call(0x400010, s_off=1) == smoe.EINVAL           # fp16 scales at an odd address
    assert call(0x400010, q_off=2, where=smoe.HOST) == smoe.EINVAL


def test_gdn_step_checks_shapes_before_any_work():
    """gdn_step refuses bad shapes and null buffers without touching memory or
    the device (the checks come before any launch), and does nothing for B = 0
    or T = 0."""
    L = smoe.lib()

    def call(nk, nv, dk, dv, B=1, T=1, ptr=None):
        sh = smoe.GdnShape(nk, nv, dk, dv)
        return L.gdn_step(C.byref(sh), B, T, ptr, ptr, ptr, ptr, ptr, 0.0, ptr, ptr, None)

    assert call(2, 3, 128, 128) == smoe.EINVAL          # n_v not a multiple of n_k
    assert call(0, 4, 128, 128) == smoe.EINVAL
    assert call(2, 4, 96, 128) == smoe.ENOTSUP          # d_k outside {32, 64, 128}
    assert call(2, 4, 128, 130) == smoe.ENOTSUP         # d_v not a multiple of 4
    assert call(2, 4, 128, 2048) == smoe.ENOTSUP        # d_v above 1024
    assert call(2, 4, 128, 128, B=-1) == smoe.EINVAL
    assert call(2, 4, 128, 128) == smoe.EINVAL          # null buffers
    assert call(2, 4, 128, 128, ptr=0x100008) == smoe.EINVAL   # not 16-byte aligned
    assert call(2, 4, 128, 128, B=0) == smoe.OK
    assert call(2, 4, 128, 128, T=0) == smoe.OK
