"""GPU parity of moe_decode_stack (one token through a stack of layers in one
persistent launch), through the C ABI: against the CPU oracle's residual
chain, against moe_route (routing bit-identical) and moe_forward (outputs
within the layer tolerance) on the same layer inputs, determinism, slot
placement, graph capture and the error word."""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import oracle
import synthetic
import workload as W
from test_gpu_parity import assert_output_close, check_chain, gpu_forward, gpu_route

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


def make(name, n_layers, table=None):
    wl = synthetic.WORKLOADS[name]
    pool = W.DevicePool(wl, n_layers=n_layers, table=table)
    inp = W.LayerInputs(wl, n_layers)
    return pool, inp


def run_stack(pool, inp, x0_bits, first=0, n=None, err=None):
    wl = pool.wl
    n = pool.n_layers - first if n is None else n
    xs = torch.zeros((n + 1, wl.H), dtype=torch.bfloat16, device="cuda")
    xs[0].copy_(W.bf16_tensor(x0_bits)[0])
    ids = torch.zeros((n, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((n, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros((n,), dtype=torch.float32, device="cuda")
    nb = pool.ctx.stack_workspace_bytes(n)
    assert nb > 0
    ws = torch.zeros((nb + 15) // 16 * 16, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda") if err is None else err
    smoe.moe_decode_stack(pool.ctx, first, inp.Wr[first:first + n], inp.ws[first:first + n],
                          [pool.shared[l] for l in range(first, first + n)], xs, ids, w, gate, pool.pool, ws, err,
                          logit_bias=inp.bias)
    torch.cuda.synchronize()
    return xs, ids, w, gate, err


@pytest.mark.parametrize("name,n_layers,first", [("tiny", 3, 0), ("decode35b", 6, 0), ("decode80b", 6, 2)])
def test_stack_against_oracle_chain(name, n_layers, first):
    pool, inp = make(name, n_layers)
    wl = pool.wl
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=4242 + first)
    xs, ids, w, gate, err = run_stack(pool, inp, x0, first=first)
    assert smoe.check(err) == 0
    check_chain(wl, inp, x0, W.bits_of(xs), ids.cpu().numpy(), w.cpu().numpy(), gate.cpu().numpy(), first=first)


@pytest.mark.parametrize("name", ["tiny", "decode80b"])
def test_stack_routing_equals_moe_route_and_layers_match_moe_forward(name):
    """Each layer's routing is moe_route's bit for bit on that layer's input
    x_l (the stack's own xs[l]); its output matches moe_forward's on the same
    x_l and routing within the layer tolerance (the two kernels sum the expert
    partials in different orders)."""
    pool, inp = make(name, 3)
    wl = pool.wl
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=99)
    xs, ids, w, gate, err = run_stack(pool, inp, x0)
    assert smoe.check(err) == 0
    for l in range(3):
        xl = W.bits_of(xs[l:l + 1])
        ids_r, w_r, gate_r = gpu_route(pool, inp, l, xl)
        assert np.array_equal(ids[l].cpu().numpy(), ids_r[0])
        assert np.array_equal(w[l].cpu().numpy(), w_r[0])
        assert np.array_equal(gate[l:l + 1].cpu().numpy(), gate_r)
        ref_fwd = gpu_forward(pool, l, xl, ids_r, w_r, gate_r, residual=True)
        got = W.bits_of(xs[l + 1:l + 2])
        assert_output_close(got, synthetic.bf16_bits_to_f32(ref_fwd).astype(np.float64))


def test_stack_top_k_of_equal_logits():
    """A layer whose router rows are all zero: every logit is 0, so the top-k
    is decided by the tie rule alone (the lowest ids first) and the candidate
    set is far wider than one warp (the slow ranking path). The ids and
    weights equal moe_route's and the rule's: experts 0 .. k-1, each 1/k."""
    pool, inp = make("decode80b", 2)
    wl = pool.wl
    inp.Wr[1].zero_()
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=31)
    xs, ids, w, gate, err = run_stack(pool, inp, x0)
    assert smoe.check(err) == 0
    xl = W.bits_of(xs[1:2])
    ids_r, w_r, gate_r = gpu_route(pool, inp, 1, xl)
    assert np.array_equal(ids[1].cpu().numpy(), ids_r[0])
    assert np.array_equal(w[1].cpu().numpy(), w_r[0])
    assert np.array_equal(ids_r[0], np.arange(wl.k))
    assert np.allclose(w_r[0], 1.0 / wl.k, rtol=0, atol=1e-7)


def test_stack_bit_identical_across_runs_slot_permutations_and_graph_replay():
    wl = synthetic.WORKLOADS["decode80b"]
    L = 3
    a_pool, inp = make("decode80b", L)
    perm = np.random.default_rng(11).permutation(L * wl.E).astype(np.int32).reshape(L, wl.E)
    b_pool, _ = make("decode80b", L, table=perm)
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=7)
    r1 = run_stack(a_pool, inp, x0)
    r2 = run_stack(a_pool, inp, x0)
    r3 = run_stack(b_pool, inp, x0)
    for t1, t2, t3 in zip(r1[:4], r2[:4], r3[:4]):
        assert torch.equal(t1, t2)
        assert torch.equal(t1, t3)
    # captured in a CUDA graph and replayed: the same step
    xs = torch.zeros_like(r1[0])
    xs[0].copy_(r1[0][0])
    ids, w, gate = torch.zeros_like(r1[1]), torch.zeros_like(r1[2]), torch.zeros_like(r1[3])
    nb = a_pool.ctx.stack_workspace_bytes(L)
    ws = torch.zeros((nb + 15) // 16 * 16, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        smoe.moe_decode_stack(a_pool.ctx, 0, inp.Wr, inp.ws, [a_pool.shared[l] for l in range(L)], xs, ids, w, gate,
                              a_pool.pool, ws, err, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert smoe.check(err) == 0
    assert torch.equal(xs, r1[0]) and torch.equal(ids, r1[1]) and torch.equal(w, r1[2])


def test_stack_bad_slot_sets_error_word_and_finishes():
    pool, inp = make("tiny", 2)
    wl = pool.wl
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=3)
    xs, ids, w, gate, err = run_stack(pool, inp, x0)
    assert smoe.check(err) == 0
    e = int(ids[1, 0].item())
    saved = pool.table_dev[1, e].item()
    try:
        pool.table_dev[1, e] = -7
        xs2, ids2, w2, gate2, err2 = run_stack(pool, inp, x0)
        assert smoe.check(err2) == smoe.DEV_BAD_SLOT
        assert torch.equal(xs2[:2], xs[:2])                  # layer 0 untouched
        assert torch.isfinite(xs2.float()).all()
    finally:
        pool.table_dev[1, e] = saved
        torch.cuda.synchronize()


def test_stack_argument_checks():
    pool, inp = make("tiny", 2)
    wl = pool.wl
    assert pool.ctx.stack_workspace_bytes(65) == 0
    xs = torch.zeros((3, wl.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((2, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((2, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros((2,), dtype=torch.float32, device="cuda")
    ws = torch.zeros(pool.ctx.stack_workspace_bytes(2), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    two = lambda a: [a[1], a[1]]
    with pytest.raises(smoe.SmoeError) as ei:               # layers 1 and 2 of a 2-layer context
        smoe.moe_decode_stack(pool.ctx, 1, two(inp.Wr), two(inp.ws), two(pool.shared), xs, ids, w, gate, pool.pool,
                              ws, err)
    assert ei.value.status == smoe.EINVAL
    with pytest.raises(smoe.SmoeError) as ei:               # workspace too small
        smoe.moe_decode_stack(pool.ctx, 0, inp.Wr, inp.ws, [pool.shared[0], pool.shared[1]], xs, ids, w, gate,
                              pool.pool, ws[:64], err)
    assert ei.value.status == smoe.ENOMEM
