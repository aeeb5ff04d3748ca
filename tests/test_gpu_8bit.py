"""GPU: MLX 8-bit experts through moe_forward, against the oracle's 8-bit
layer, element by element: the fused decode kernel (T <= 8) at T = 1 and 8
and the token-bucketed grouped GEMMs (T > 8) at T = 9 and 64 on the GPU's
own routing, and at T = 600 with every token routed among 12 experts (three
tiles per expert, the last one ragged); bit-identity across reruns and slot
permutations, agreement with the plain CUDA path, and the one-launch decode
stack (moe_decode_stack) on 8-bit experts (moe_forward_noalloc on 8-bit
experts: test_zz_no_alloc.py)."""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import oracle_shards
import synthetic
import workload as W
from test_gpu_parity import assert_output_close, check_chain_layers_on_own_input, gpu_forward, gpu_route, routing_ok
from test_gpu_stack import run_stack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


@pytest.fixture(scope="module")
def p80_8():
    wl = synthetic.WORKLOADS["decode80b_int8"]
    return W.DevicePool(wl, n_layers=2), W.LayerInputs(wl, 2)


@pytest.mark.parametrize("T", [1, 8, 9, 64])
def test_8bit_decode_against_oracle(p80_8, T):
    pool, inp = p80_8
    wl = pool.wl
    for layer in (0, 1):
        x = synthetic.activations(wl.seed, T, wl.H, tag=300 + 10 * layer + T)
        ids, w, gate = gpu_route(pool, inp, layer, x)
        ref = oracle_shards.tokens_sharded(wl.name, layer, x, ids, inp.Wr_bits[layer], inp.ws_bits[layer])
        routing_ok(ids, w, gate, ref, wl.k)
        out = gpu_forward(pool, layer, x, ids, w, gate)
        assert_output_close(out, ref["out64"])
        res = gpu_forward(pool, layer, x, ids, w, gate, residual=True)
        xr = synthetic.bf16_bits_to_f32(x).astype(np.float64)
        assert_output_close(res, xr + ref["out64"])


def test_8bit_bit_identical_across_runs_and_slot_permutations(p80_8):
    pool, inp = p80_8
    wl = pool.wl
    perm = np.random.default_rng(21).permutation(2 * wl.E).astype(np.int32).reshape(2, wl.E)
    other = W.DevicePool(wl, n_layers=2, table=perm)
    for T in (1, 4, 40):
        x = synthetic.activations(wl.seed, T, wl.H, tag=700 + T)
        ids, w, gate = gpu_route(pool, inp, 1, x)
        a = gpu_forward(pool, 1, x, ids, w, gate)
        assert np.array_equal(a, gpu_forward(pool, 1, x, ids, w, gate))
        assert np.array_equal(a, gpu_forward(other, 1, x, ids, w, gate))


def test_8bit_fast_and_plain_paths_agree(p80_8):
    """Two approximations of the oracle's layer: within twice the layer bounds
    of each other, and each within the bounds of the oracle."""
    pool, inp = p80_8
    wl = pool.wl
    T = 3
    x = synthetic.activations(wl.seed, T, wl.H, tag=777)
    ids, w, gate = gpu_route(pool, inp, 0, x)
    fast = gpu_forward(pool, 0, x, ids, w, gate)
    out = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).cuda()
    smoe.moe_forward_debug(pool.ctx, 0, W.bf16_tensor(x), dev(ids, np.int32), dev(w, np.float32),
                           dev(gate, np.float32), pool.pool, pool.shared[0], out, err)
    assert smoe.check(err) == 0
    ref = oracle_shards.tokens_sharded(wl.name, 0, x, ids, inp.Wr_bits[0], inp.ws_bits[0])
    f = synthetic.bf16_bits_to_f32(fast).astype(np.float64)
    d = synthetic.bf16_bits_to_f32(W.bits_of(out)).astype(np.float64)
    assert_output_close(W.bits_of(out), ref["out64"])
    assert np.linalg.norm(f - d) <= 2 * 5e-3 * np.linalg.norm(ref["out64"])


def test_8bit_bucketed_multi_tile_experts(p80_8):
    """600 tokens, each routed to 10 of the same 12 experts (about 500 pairs
    per expert: three tiles of at most 192 tokens, the last one ragged),
    through the large-T bucketing; weights are the oracle's probabilities
    renormalised over that choice. A rerun is bit-identical."""
    pool, inp = p80_8
    wl = pool.wl
    T = 600
    x = synthetic.activations(wl.seed, T, wl.H, tag=901)
    rng = np.random.default_rng(33)
    hot = rng.choice(wl.E, 12, replace=False)
    ids = np.stack([rng.choice(hot, wl.k, replace=False) for _ in range(T)]).astype(np.int32)
    ref = oracle_shards.tokens_sharded(wl.name, 1, x, ids, inp.Wr_bits[1], inp.ws_bits[1])
    out = gpu_forward(pool, 1, x, ids, ref["w_used"], ref["gate"])
    assert_output_close(out, ref["out64"])
    assert np.array_equal(out, gpu_forward(pool, 1, x, ids, ref["w_used"], ref["gate"]))


def test_8bit_stack_against_oracle_and_per_layer_path(p80_8):
    """moe_decode_stack on 8-bit experts (two layers of the 80B shape): each
    layer on its own input against the oracle's 8-bit combine of the GPU's
    choice (the flat per-layer rule), routing bit-identical to moe_route on
    that input, output within the layer tolerance of moe_forward's; a rerun
    and a permuted slot placement give the same bits."""
    pool, inp = p80_8
    wl = pool.wl
    x0 = synthetic.activations(wl.seed, 1, wl.H, tag=808)
    xs, ids, w, gate, err = run_stack(pool, inp, x0)
    assert smoe.check(err) == 0
    xb = W.bits_of(xs)
    idn, wn, gn = ids.cpu().numpy(), w.cpu().numpy(), gate.cpu().numpy()
    check_chain_layers_on_own_input(wl, [0, 1], [xb[l:l + 1] for l in range(2)], [xb[l + 1:l + 2] for l in range(2)],
                                    [idn[l:l + 1] for l in range(2)], [wn[l:l + 1] for l in range(2)],
                                    [gn[l:l + 1] for l in range(2)], inp)
    for l in range(2):
        ids_r, w_r, gate_r = gpu_route(pool, inp, l, xb[l:l + 1])
        assert np.array_equal(idn[l], ids_r[0]) and np.array_equal(wn[l], w_r[0])
        assert np.array_equal(gn[l:l + 1], gate_r)
        ref_fwd = gpu_forward(pool, l, xb[l:l + 1], ids_r, w_r, gate_r, residual=True)
        assert_output_close(xb[l + 1:l + 2], synthetic.bf16_bits_to_f32(ref_fwd).astype(np.float64))
    again = run_stack(pool, inp, x0)
    perm = np.random.default_rng(23).permutation(2 * wl.E).astype(np.int32).reshape(2, wl.E)
    other = run_stack(W.DevicePool(wl, n_layers=2, table=perm), inp, x0)
    for a, b, c in zip((xs, ids, w, gate), again[:4], other[:4]):
        assert torch.equal(a, b) and torch.equal(a, c)
