"""GPU: the plain per-token CUDA path (moe_forward_debug) against the oracle,
and the fast kernels (the decode kernel for T <= 8, the bucketed tensor-core
path above) against it, each within the layer tolerance; bad slots set the
error word."""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import oracle
import synthetic
import workload as W
from test_gpu_parity import assert_output_close, gpu_forward, oracle_layer, routing_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


def debug_forward(pool, layer, x_bits, ids, w, gate, residual=False):
    wl = pool.wl
    T = x_bits.shape[0]
    x = W.bf16_tensor(x_bits)
    out = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    smoe.moe_forward_debug(pool.ctx, layer, x, torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda(),
                           torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda(),
                           torch.from_numpy(np.ascontiguousarray(gate, np.float32)).cuda(), pool.pool,
                           pool.shared[layer], out, err, residual=x if residual else None)
    code = smoe.check(err)
    return W.bits_of(out), code


@pytest.mark.parametrize("name,Ts", [("tiny", (1, 4, 20)), ("decode35b", (2, 16))])
def test_debug_path_matches_oracle_and_fast_kernels(name, Ts):
    wl = synthetic.WORKLOADS[name]
    pool, inp = W.DevicePool(wl, n_layers=1), W.LayerInputs(wl, 1)
    for T in Ts:
        x = synthetic.activations(wl.seed, T, wl.H, tag=900 + T)
        ref = oracle_layer(wl, 0, x, inp)
        dbg, code = debug_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"])
        assert code == 0
        assert_output_close(dbg, ref["out64"])
        fast = gpu_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"])
        assert_output_close(fast, ref["out64"])
        # fast against debug: two approximations of the oracle, so twice the layer bounds
        f = synthetic.bf16_bits_to_f32(fast).astype(np.float64)
        d = synthetic.bf16_bits_to_f32(dbg).astype(np.float64)
        rms = np.sqrt(np.mean(ref["out64"] ** 2))
        assert np.linalg.norm(f - d) <= 2 * 5e-3 * np.linalg.norm(ref["out64"])
        assert np.abs(f - d).max() <= 2 * 2e-2 * rms
        dres, _ = debug_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"], residual=True)
        xr = synthetic.bf16_bits_to_f32(x).astype(np.float64)
        assert_output_close(dres, xr + ref["out64"])


def test_debug_path_8_bit_experts_match_oracle():
    """8-bit experts (two-plane atoms, packed on the host) through the plain
    CUDA path, the fused decode kernel (moe_forward and moe_forward_noalloc)
    and the one-launch stack, against the oracle's 8-bit layer."""
    wl = synthetic.WORKLOADS["tiny"]
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I, bits=8)
    stride = smoe.layout_of(shape).blob_bytes
    trip = {e: synthetic.expert_triples(wl.seed, 0, e, wl.H, wl.I, bits=8) for e in range(wl.E)}
    shared_t = synthetic.expert_triples(wl.seed, 0, None, wl.H, wl.I, bits=8)
    host = np.zeros(wl.E * stride, np.uint8)
    smoe.pack_experts(shape, [trip[e].arrays() for e in range(wl.E)], list(range(wl.E)), host, host.size, smoe.HOST)
    sh = np.zeros(stride, np.uint8)
    smoe.pack_experts(shape, [shared_t.arrays()], [0], sh, sh.size, smoe.HOST)
    pool, shared = torch.from_numpy(host).cuda(), torch.from_numpy(sh).cuda()
    table = torch.zeros((1, wl.E), dtype=torch.int32, device="cuda")
    ctx = smoe.Context(shape, 1, wl.E, table)
    smoe.set_slot_table(ctx, 0, np.arange(wl.E, dtype=np.int32))
    inp = W.LayerInputs(wl, 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T in (1, 5):
        x = synthetic.activations(wl.seed, T, wl.H, tag=990 + T)
        ids, w, gate = oracle.route(x, inp.Wr_bits[0], inp.ws_bits[0], wl.k)
        ref, _ = oracle.combine8(x, ids, w, gate, {int(e): trip[int(e)] for e in np.unique(ids)}, shared_t,
                                 wl.E, wl.I, wl.I)
        dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).cuda()
        out = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
        smoe.moe_forward_debug(ctx, 0, W.bf16_tensor(x), dev(ids, np.int32), dev(w, np.float32),
                               dev(gate, np.float32), pool, shared, out, err)
        assert smoe.check(err) == 0
        assert_output_close(W.bits_of(out), ref)
    # the fused decode kernel reads 8-bit atoms too (T <= 8): the same layer
    fast = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
    smoe.moe_forward(ctx, 0, W.bf16_tensor(x), dev(ids, np.int32), dev(w, np.float32), dev(gate, np.float32),
                     pool, shared, fast, W.workspace(ctx, T), err)
    assert smoe.check(err) == 0
    assert_output_close(W.bits_of(fast), ref)
    # moe_forward_noalloc runs the same kernel: the same bits
    na = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
    smoe.moe_forward_noalloc(ctx, 0, W.bf16_tensor(x), dev(ids, np.int32), dev(w, np.float32),
                             dev(gate, np.float32), pool, shared, na, err)
    assert smoe.check(err) == 0
    assert torch.equal(na, fast)
    # the stack on the same layer: its own routing (moe_route's rule) and x + the layer
    nb = ctx.stack_workspace_bytes(1)
    assert nb > 0
    x1 = synthetic.activations(wl.seed, 1, wl.H, tag=997)
    xs = torch.zeros((2, wl.H), dtype=torch.bfloat16, device="cuda")
    xs[0].copy_(W.bf16_tensor(x1)[0])
    sid = torch.zeros((1, wl.k), dtype=torch.int32, device="cuda")
    sw = torch.zeros((1, wl.k), dtype=torch.float32, device="cuda")
    sg = torch.zeros((1,), dtype=torch.float32, device="cuda")
    ws = torch.zeros((nb + 15) // 16 * 16, dtype=torch.uint8, device="cuda")
    smoe.moe_decode_stack(ctx, 0, [inp.Wr[0]], [inp.ws[0]], [shared], xs, sid, sw, sg, pool, ws, err)
    torch.cuda.synchronize()
    assert smoe.check(err) == 0
    r = oracle.route(x1, inp.Wr_bits[0], inp.ws_bits[0], wl.k, want_probs=True)
    gids = sid.cpu().numpy()
    w_own = routing_ok(gids, sw.cpu().numpy(), sg.cpu().numpy(), dict(ids=r[0], probs=r[3], gate=r[2]), wl.k)
    ref1, _ = oracle.combine8(x1, gids, w_own, r[2], {int(e): trip[int(e)] for e in np.unique(gids)}, shared_t,
                              wl.E, wl.I, wl.I)
    xr = synthetic.bf16_bits_to_f32(x1).astype(np.float64)
    assert_output_close(W.bits_of(xs[1:2]), xr + ref1)


def test_debug_path_bad_slot_sets_error_word():
    wl = synthetic.WORKLOADS["tiny"]
    pool, inp = W.DevicePool(wl), W.LayerInputs(wl, 1)
    x = synthetic.activations(wl.seed, 2, wl.H, tag=950)
    ref = oracle_layer(wl, 0, x, inp)
    e = int(ref["ids"][0, 0])
    saved = pool.table_dev[0, e].item()
    try:
        pool.table_dev[0, e] = -1
        out, code = debug_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"])
        assert code == smoe.DEV_BAD_SLOT
        assert np.isfinite(synthetic.bf16_bits_to_f32(out)).all()
    finally:
        pool.table_dev[0, e] = saved
        torch.cuda.synchronize()


def test_misaligned_buffers_are_refused_without_a_launch():
    """An offset view (pool[8:], a shared blob or output 2 bytes in) is
    contiguous and passes the binding, but the library refuses it with
    EINVAL: the kernels read 16-byte lanes and 4-byte words. Checked through
    the raw C ABI for moe_forward_debug and for device packing."""
    wl = synthetic.WORKLOADS["tiny"]
    pool, inp = W.DevicePool(wl, n_layers=1), W.LayerInputs(wl, 1)
    T = 2
    x = W.bf16_tensor(synthetic.activations(wl.seed, T, wl.H, tag=5))
    ids = torch.zeros((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros((T,), dtype=torch.float32, device="cuda")
    out = torch.zeros((T * wl.H + 8,), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L, p = smoe.lib(), smoe._ptr
    nbytes = pool.pool.numel()

    def dbg(pool_p, shared_p, out_p):
        return L.moe_forward_debug(pool.ctx.handle, 0, p(x), T, p(ids), p(w), p(gate), pool_p, nbytes, shared_p,
                                   None, out_p, p(err), None)
    assert dbg(p(pool.pool) + 8, p(pool.shared[0]), p(out)) == smoe.EINVAL
    assert dbg(p(pool.pool), p(pool.shared[0]) + 4, p(out)) == smoe.EINVAL
    assert dbg(p(pool.pool), p(pool.shared[0]), p(out) + 2) == smoe.EINVAL
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I)
    dev = [t[0] for t in W.device_triples(wl.seed, 0, 1, 1, wl.H, wl.I)]
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.pack_experts(shape, [dev], [0], pool.pool[8:], nbytes - 8, smoe.DEVICE)
    assert ei.value.status == smoe.EINVAL
    torch.cuda.synchronize()
    assert smoe.check(err) == 0
