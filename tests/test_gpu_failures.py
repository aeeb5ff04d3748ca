"""GPU: failure detection without a fault. A bounded wait that runs out
returns an error status that the host reads, and the context stays usable;
an input outside the fp16 range of the token-bucketed path sets its error
word instead of trapping.

The timeout is made on purpose through smoe_set_stack_wait: a short limit
for the grid-wide waits of moe_decode_stack, and one wait that asks for an
arrival that never comes. The kernel's waits for its own bulk copies keep
their normal limit, so no CTA leaves with a copy in flight."""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import synthetic
import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


def _stack_call(pool, inp, x0, n):
    wl = pool.wl
    xs = torch.zeros((n + 1, wl.H), dtype=torch.bfloat16, device="cuda")
    xs[0].copy_(W.bf16_tensor(x0)[0])
    ids = torch.zeros((n, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((n, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros((n,), dtype=torch.float32, device="cuda")
    nb = pool.ctx.stack_workspace_bytes(n)
    ws = torch.zeros((nb + 15) // 16 * 16, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    smoe.moe_decode_stack(pool.ctx, 0, inp.Wr[:n], inp.ws[:n], [pool.shared[l] for l in range(n)], xs, ids, w,
                          gate, pool.pool, ws, err)
    torch.cuda.synchronize()
    return xs, err


def test_stack_wait_that_runs_out_reports_timeout_and_returns():
    wl = synthetic.WORKLOADS["tiny"]
    pool, inp = W.DevicePool(wl, n_layers=2), W.LayerInputs(wl, 2)
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=12)
    good, err = _stack_call(pool, inp, x0, 2)
    assert smoe.check(err) == 0
    try:
        pool.ctx.set_stack_wait(grid_wait_ns=1_000_000, stall_layer=1)   # 1 ms; layer 1 never completes
        _, err = _stack_call(pool, inp, x0, 2)
        assert smoe.check(err) == smoe.DEV_TIMEOUT
    finally:
        pool.ctx.set_stack_wait(0, -1)
    # the context and the GPU are still usable: the same step gives the same bits
    again, err = _stack_call(pool, inp, x0, 2)
    assert smoe.check(err) == 0
    assert torch.equal(again, good)


def test_bucketed_path_flags_values_outside_fp16():
    """T = 16 (the tensor-core path, fp16 operands) with one token at
    |x| = 1e5: the call returns, the error word reads SMOE_DEV_RANGE, and a
    call with in-range x afterwards is clean."""
    wl = synthetic.WORKLOADS["tiny"]
    pool, inp = W.DevicePool(wl, n_layers=1), W.LayerInputs(wl, 1)
    T = 16
    xb = synthetic.activations(wl.seed, T, wl.H, tag=44)
    big = xb.copy()
    big[3, :] = synthetic.f32_to_bf16_bits(np.full(wl.H, 1e5, np.float32))
    for bits, want in ((big, smoe.DEV_RANGE), (xb, 0)):
        x = W.bf16_tensor(bits)
        ids = torch.zeros((T, wl.k), dtype=torch.int32, device="cuda")
        w = torch.zeros((T, wl.k), dtype=torch.float32, device="cuda")
        gate = torch.zeros((T,), dtype=torch.float32, device="cuda")
        ws = W.workspace(pool.ctx, T)
        smoe.moe_route(pool.ctx, inp.Wr[0], inp.ws[0], x, ids, w, gate, ws)
        out = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        smoe.moe_forward(pool.ctx, 0, x, ids, w, gate, pool.pool, pool.shared[0], out, ws, err)
        torch.cuda.synchronize()
        assert smoe.check(err) == want
