"""GPU: moe_forward over the streaming slot pool (smoe_cache). The device slots
hold a changing subset of the experts, filled from a host copy of every
packed blob as the routing asks for them. Outputs are bit-identical to the
fully resident pool and, element by element, within the layer tolerance of
the CPU oracle's layer on the same routing; the
hit and miss counts equal the host policy's on the same request stream; an
expert that is not resident makes moe_forward raise the bad-slot error word
instead of reading another expert's weights."""
import types

import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import synthetic
import workload as W
import oracle_shards
from test_gpu_parity import assert_output_close, assert_residual_close, gpu_forward, gpu_route, routing_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


def host_store_of(full):
    """Every expert's packed blob in [layer][expert] order, in pinned host memory."""
    idx = torch.from_numpy(full.table.astype(np.int64)).cuda().reshape(-1)
    blobs = full.pool.view(-1, full.stride).index_select(0, idx)
    return blobs.reshape(-1).cpu().pin_memory()


def cached(full, n_slots):
    wl = full.wl
    pool = torch.empty(n_slots * full.stride, dtype=torch.uint8, device="cuda")
    table = torch.zeros((full.n_layers, wl.E), dtype=torch.int32, device="cuda")
    ctx = smoe.Context(full.shape, full.n_layers, n_slots, table)
    store = host_store_of(full)
    cache = smoe.Cache(ctx, store, pool)
    torch.cuda.synchronize()
    return types.SimpleNamespace(wl=wl, ctx=ctx, pool=pool, shared=full.shared, table=table, cache=cache, store=store)


@pytest.fixture(scope="module")
def two_layers():
    wl = synthetic.WORKLOADS["decode35b"]
    full = W.DevicePool(wl, n_layers=2)
    return full, W.LayerInputs(wl, 2)


def test_cached_pool_is_bit_identical_and_counts_match_the_policy(two_layers):
    full, inp = two_layers
    wl = full.wl
    c = cached(full, n_slots=72)
    reqs, pieces, got = [], [], []
    for t in range(10):
        T = 1 if t < 6 else 8                                     # the decode kernel, then T = 8
        x = synthetic.activations(wl.seed, T, wl.H, tag=600 + t)
        for layer in range(full.n_layers):
            ids, w, gate = gpu_route(full, inp, layer, x)
            h, m = c.cache.prepare(layer, ids)
            assert h + m == ids.size
            reqs.append((layer, ids.ravel().tolist()))
            a = gpu_forward(full, layer, x, ids, w, gate, residual=True)
            b = gpu_forward(c, layer, x, ids, w, gate, residual=True)
            assert np.array_equal(a, b)
            pieces.append((wl.name, layer, x, ids, inp.Wr_bits[layer], inp.ws_bits[layer], None))
            got.append((ids, w, gate, x, b))
    for ref, (ids, w, gate, x, b) in zip(oracle_shards.run_pieces(pieces), got):
        routing_ok(ids, w, gate, ref, wl.k)
        assert_residual_close(b, x, ref["out64"])
    _, sh, sm = smoe.cache_simulate(full.n_layers, wl.E, 72, reqs)
    hits, misses, nbytes = c.cache.stats()
    assert (hits, misses) == (sh, sm)
    assert nbytes == misses * full.stride
    assert misses >= 72                                          # the pool has been cycled through


def test_bucketed_path_through_the_cache(two_layers):
    full, inp = two_layers
    wl = full.wl
    c = cached(full, n_slots=wl.E)                                # one layer's worth of slots
    x = synthetic.activations(wl.seed, 48, wl.H, tag=611)
    for layer in range(full.n_layers):
        ids, w, gate = gpu_route(full, inp, layer, x)
        c.cache.prepare(layer, ids)
        b = gpu_forward(c, layer, x, ids, w, gate)
        assert np.array_equal(gpu_forward(full, layer, x, ids, w, gate), b)
        ref = oracle_shards.tokens_sharded(wl.name, layer, x, ids, inp.Wr_bits[layer], inp.ws_bits[layer])
        routing_ok(ids, w, gate, ref, wl.k)
        assert_output_close(b, ref["out64"])


def test_expert_not_resident_sets_bad_slot(two_layers):
    full, inp = two_layers
    wl = full.wl
    c = cached(full, n_slots=16)
    x = synthetic.activations(wl.seed, 1, wl.H, tag=620)
    ids, w, gate = gpu_route(full, inp, 0, x)
    c.cache.prepare(0, ids)
    other = np.array([[e for e in range(wl.E) if e not in set(ids.ravel().tolist())][:wl.k]], np.int32)
    out = torch.zeros((1, wl.H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    smoe.moe_forward(c.ctx, 0, W.bf16_tensor(x), torch.from_numpy(other).cuda(), torch.from_numpy(w).cuda(),
                     torch.from_numpy(gate).cuda(), c.pool, c.shared[0], out, W.workspace(c.ctx, 1), err)
    assert smoe.check(err) == smoe.DEV_BAD_SLOT
    assert torch.isfinite(out.float()).all()


def test_cache_arguments():
    wl = synthetic.WORKLOADS["tiny"]
    full = W.DevicePool(wl)
    c = cached(full, n_slots=4)
    with pytest.raises(smoe.SmoeError) as ei:
        c.cache.prepare(0, np.arange(5))                          # five distinct experts, four slots
    assert ei.value.status == smoe.ENOMEM
    with pytest.raises(smoe.SmoeError) as ei:
        c.cache.prepare(1, np.arange(2))                          # a one-layer context
    assert ei.value.status == smoe.EINVAL
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.Cache(c.ctx, c.store[:100], c.pool)                 # host store too small
    assert ei.value.status == smoe.ENOMEM
