"""GPU: shapes at the boundary's limits against the oracle, through the C ABI.
The largest router the kernels take (E = 1024 experts, k = 16 chosen, with
H = 2048 and I = 512 at their maxima) and top-1 routing (k = 1: the
renormalised weight is exactly 1), through moe_route + moe_forward at T = 1
and 8 (the fused decode kernel) and T = 9 and 64 (the token-bucketed path),
every token checked; and moe_decode_stack over two layers of each shape where
the GPU runs it (otherwise it must refuse with ENOTSUP)."""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import oracle_shards
import synthetic
import workload as W
from test_gpu_parity import assert_output_close, check_chain_layers_on_own_input, gpu_forward, gpu_route, routing_ok

pytestmark = pytest.mark.gpu

SHAPES = ["limits_e1024_k16", "limits_k1"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


@pytest.fixture(scope="module", params=SHAPES)
def limit_pool(request):
    wl = synthetic.WORKLOADS[request.param]
    return W.DevicePool(wl, n_layers=2), W.LayerInputs(wl, 2)


@pytest.mark.parametrize("T", [1, 8, 9, 64])
def test_limit_shapes_against_oracle(limit_pool, T):
    pool, inp = limit_pool
    wl = pool.wl
    for layer in (0, 1):
        x = synthetic.activations(wl.seed, T, wl.H, tag=600 + 10 * layer + T)
        ids, w, gate = gpu_route(pool, inp, layer, x)
        assert np.all((ids >= 0) & (ids < wl.E))
        assert all(len(set(r)) == wl.k for r in ids.tolist())          # k distinct experts per token
        if wl.k == 1:
            assert np.all(w == 1.0)
        ref = oracle_shards.tokens_sharded(wl.name, layer, x, ids, inp.Wr_bits[layer], inp.ws_bits[layer])
        routing_ok(ids, w, gate, ref, wl.k)
        out = gpu_forward(pool, layer, x, ids, w, gate)
        assert_output_close(out, ref["out64"])


def test_limit_shapes_decode_stack(limit_pool):
    pool, inp = limit_pool
    wl = pool.wl
    nb = pool.ctx.stack_workspace_bytes(2)
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=6060)
    xs = torch.zeros((3, wl.H), dtype=torch.bfloat16, device="cuda")
    xs[0].copy_(W.bf16_tensor(x0)[0])
    ids = torch.zeros((2, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((2, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros((2,), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, (nb + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
    if nb == 0:
        # the shape's stack does not fit one CTA per SM: refused at the boundary
        with pytest.raises(smoe.SmoeError) as e:
            smoe.moe_decode_stack(pool.ctx, 0, inp.Wr[:2], inp.ws[:2], [pool.shared[l] for l in range(2)], xs, ids, w,
                                  gate, pool.pool, ws, err, logit_bias=inp.bias)
        assert e.value.status == smoe.ENOTSUP
        return
    smoe.moe_decode_stack(pool.ctx, 0, inp.Wr[:2], inp.ws[:2], [pool.shared[l] for l in range(2)], xs, ids, w, gate,
                          pool.pool, ws, err, logit_bias=inp.bias)
    torch.cuda.synchronize()
    assert smoe.check(err) == 0
    xb = W.bits_of(xs)
    idn, wn, gn = ids.cpu().numpy(), w.cpu().numpy(), gate.cpu().numpy()
    check_chain_layers_on_own_input(wl, [0, 1], [xb[l:l + 1] for l in range(2)], [xb[l + 1:l + 2] for l in range(2)],
                                    [idn[l:l + 1] for l in range(2)], [wn[l:l + 1] for l in range(2)],
                                    [gn[l:l + 1] for l in range(2)], inp)
    for l in range(2):                        # the stack's routing is moe_route's, bit for bit
        ids_r, w_r, gate_r = gpu_route(pool, inp, l, xb[l:l + 1])
        assert np.array_equal(idn[l], ids_r[0]) and np.array_equal(wn[l], w_r[0])
        assert np.array_equal(gn[l:l + 1], gate_r)
