"""moe_forward_noalloc: the decode path for callers that cannot allocate
device memory (they are handed only input and output buffers, or must not
let an allocation synchronise the device). It must give what moe_forward
gives, call after call, with its scratch held inside the library.

Kept in its own file, collected last, so a run that stops at the first
failure has run every other test before this one; it needs nothing that the
other tests set up.
"""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import oracle
import synthetic
import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


def _inputs(pool, inp, T, tag):
    wl = pool.wl
    x_bits = synthetic.activations(wl.seed, T, wl.H, tag=tag)
    r = oracle.route(x_bits, inp.Wr_bits[0], inp.ws_bits[0], wl.k)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).cuda()
    return W.bf16_tensor(x_bits), dev(r[0], np.int32), dev(r[1], np.float32), dev(r[2], np.float32)


@pytest.mark.parametrize("name,T", [("tiny", 4), ("decode80b", 1), ("decode80b", 8), ("decode80b_int8", 1),
                                    ("decode80b_int8", 8)])
def test_noalloc_matches_moe_forward_twice(name, T):
    wl = synthetic.WORKLOADS[name]
    pool = W.DevicePool(wl, n_layers=1)
    inp = W.LayerInputs(wl, 1)
    ref_out = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        x, ids, w, gate = _inputs(pool, inp, T, tag=900 + 10 * call + T)
        smoe.moe_forward(pool.ctx, 0, x, ids, w, gate, pool.pool, pool.shared[0], ref_out,
                         W.workspace(pool.ctx, T), err)
        out = torch.full((T, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        smoe.moe_forward_noalloc(pool.ctx, 0, x, ids, w, gate, pool.pool, pool.shared[0], out, err)
        assert smoe.check(err) == 0
        a = ref_out.double().cpu().numpy()
        b = out.double().cpu().numpy()
        # the layer tolerance (relative L2 <= 5e-3, max abs <= 2e-2 rms); the
        # same kernel runs on both sides, so in practice the bits agree
        assert np.linalg.norm(b - a) <= 5e-3 * np.linalg.norm(a)
        assert np.abs(b - a).max() <= 2e-2 * np.sqrt(np.mean(a ** 2))
        assert torch.equal(out, ref_out)


def test_noalloc_rejects_calls_larger_than_its_scratch():
    wl = synthetic.Workload("many", 2048, 1024, 16, 512, 512, 8, 1, False, False, 77, "many experts")
    shape = smoe.make_shape(wl.H, wl.E, wl.k, wl.I)
    table = torch.zeros((1, wl.E), dtype=torch.int32, device="cuda")
    ctx = smoe.Context(shape, 1, 1, table)
    pool = torch.zeros(int(ctx.layout.blob_bytes), dtype=torch.uint8, device="cuda")
    T = 8                                  # (min(1024, 128) + 1) * 8 * 2048 * 4 B > 8 MiB
    x = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros((T,), dtype=torch.float32, device="cuda")
    out = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.moe_forward_noalloc(ctx, 0, x, ids, w, gate, pool, pool, out, err)
    assert ei.value.status == smoe.ENOMEM
    T9 = 9                                 # above the decode path's 8 tokens
    x9 = torch.zeros((T9, wl.H), dtype=torch.bfloat16, device="cuda")
    ids9 = torch.zeros((T9, wl.k), dtype=torch.int32, device="cuda")
    w9 = torch.zeros((T9, wl.k), dtype=torch.float32, device="cuda")
    gate9 = torch.zeros((T9,), dtype=torch.float32, device="cuda")
    out9 = torch.zeros((T9, wl.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.moe_forward_noalloc(ctx, 0, x9, ids9, w9, gate9, pool, pool, out9, err)
    assert ei.value.status == smoe.ENOTSUP


def test_noalloc_refuses_misaligned_output_or_residual():
    """Like moe_forward, the output and the residual must start on a 16-byte
    boundary; an offset view is refused with EINVAL before any launch."""
    wl = synthetic.WORKLOADS["tiny"]
    pool = W.DevicePool(wl, n_layers=1)
    inp = W.LayerInputs(wl, 1)
    T = 2
    x, ids, w, gate = _inputs(pool, inp, T, tag=990)
    out = torch.zeros((T * wl.H + 8,), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L, p = smoe.lib(), smoe._ptr
    n = pool.pool.numel()
    rc = L.moe_forward_noalloc(pool.ctx.handle, 0, p(x), T, p(ids), p(w), p(gate), p(pool.pool), n,
                               p(pool.shared[0]), None, p(out) + 2, p(err), None)
    assert rc == smoe.EINVAL
    rc = L.moe_forward_noalloc(pool.ctx.handle, 0, p(x), T, p(ids), p(w), p(gate), p(pool.pool), n,
                               p(pool.shared[0]), p(out) + 2, p(out), p(err), None)
    assert rc == smoe.EINVAL
    torch.cuda.synchronize()
    assert smoe.check(err) == 0
