"""GPU parity of the token-bucketed path (T > 8): bucketing, tcgen05 grouped
gate/up and down GEMMs, ordered combine, and the tensor-core router.

Weights are dequantised to fp16 tiles (one rounding of s q + b), x and h
are fp16, products accumulate in fp32 and each pair's expert output is
stored as fp16 before the fp32 weighted combine, so only the layer tolerance applies (relative L2 <= 5e-3,
max abs <= 2e-2 rms against the oracle's fp64 output)."""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import oracle
import synthetic
import workload as W
import oracle_shards
from test_gpu_parity import assert_output_close, gpu_forward, gpu_route, oracle_layer, routing_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    from synthetic import _build as sb
    _build.build()
    sb.build()


@pytest.fixture(scope="module")
def tiny():
    wl = synthetic.WORKLOADS["tiny"]
    return W.DevicePool(wl), W.LayerInputs(wl, 1)


@pytest.mark.parametrize("T", [9, 64, 200, 600])
def test_prefill_tiny_against_oracle(tiny, T):
    pool, inp = tiny
    x = synthetic.activations(pool.wl.seed, T, pool.wl.H, tag=5000 + T)
    ref = oracle_layer(pool.wl, 0, x, inp)
    out = gpu_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"])
    assert_output_close(out, ref["out64"])
    out2 = gpu_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"], residual=True)
    xr = synthetic.bf16_bits_to_f32(x).astype(np.float64)
    assert_output_close(out2, xr + ref["out64"])


@pytest.mark.parametrize("name", ["tiny", "zipf80b_t64"])
def test_prefill_t64_full_width_tiles(name):
    """T = 64 with every token routed to the same k experts: each of them gets
    a full 64-token tile, the widest the T <= 64 ring shape takes (the
    weights are the oracle's probabilities renormalised over that choice)."""
    wl = synthetic.WORKLOADS[name]
    pool, inp = W.DevicePool(wl, n_layers=1), W.LayerInputs(wl, 1)
    T = 64
    x = synthetic.activations(wl.seed, T, wl.H, tag=6464)
    hot = np.random.default_rng(64).choice(wl.E, wl.k, replace=False).astype(np.int32)
    ids = np.stack([np.random.default_rng(t).permutation(hot) for t in range(T)]).astype(np.int32)
    ref = oracle_shards.tokens_sharded(wl.name, 0, x, ids, inp.Wr_bits[0], inp.ws_bits[0])
    out = gpu_forward(pool, 0, x, ids, ref["w_used"], ref["gate"])
    assert_output_close(out, ref["out64"])


def test_prefill_zipf_t64_full_layer():
    """The skewed T = 64 layer through moe_route and moe_forward on the GPU's
    own routing: every token's routing and output against the oracle's
    combine of that choice; a rerun is bit-identical."""
    wl = synthetic.WORKLOADS["zipf80b_t64"]
    pool = W.DevicePool(wl)
    inp = W.LayerInputs(wl, 1)
    x = synthetic.activations(wl.seed, wl.T, wl.H)
    ids, w, gate = gpu_route(pool, inp, 0, x)
    ref = oracle_shards.tokens_sharded(wl.name, 0, x, ids, inp.Wr_bits[0], inp.ws_bits[0], inp.bias_np)
    routing_ok(ids, w, gate, ref, wl.k)
    out = gpu_forward(pool, 0, x, ids, w, gate)
    assert_output_close(out, ref["out64"])
    again = gpu_forward(pool, 0, x, ids, w, gate)
    assert np.array_equal(out, again)


def covering_sample(ids, n, E, seed=7):
    """A seeded sample of n tokens, plus, for every expert that none of them
    routes to, the first token that does: the sample's pairs cover every
    expert the batch uses."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(ids.shape[0], n, replace=False).tolist())
    seen = np.zeros(E, bool)
    seen[ids[sorted(pick)].ravel()] = True
    for e in np.flatnonzero(~seen):
        t = int(np.flatnonzero((ids == e).any(axis=1))[0])
        pick.add(t)
        seen[ids[t]] = True
    return np.array(sorted(pick))


@pytest.mark.parametrize("name", ["prefill80b", "prefill35b"])
def test_prefill_8192_tokens_sampled(name):
    """A full prefill workload (80B shape: ~160 pairs per expert; 35B shape:
    ~256, two tiles per expert) through moe_route + moe_forward on the GPU.
    The oracle checks a seeded sample of at least 512 tokens whose pairs
    cover every expert: each sampled token's routing by the rule and its
    output against the oracle's combine of the GPU's own choice. Every output
    is finite, a rerun is bit-identical, and the load per expert is near
    uniform."""
    wl = synthetic.WORKLOADS[name]
    pool, inp = W.DevicePool(wl, n_layers=1), W.LayerInputs(wl, 1)
    x = synthetic.activations(wl.seed, wl.T, wl.H)
    ids, w, gate = gpu_route(pool, inp, 0, x)
    out = gpu_forward(pool, 0, x, ids, w, gate)
    assert np.isfinite(synthetic.bf16_bits_to_f32(out)).all()
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    mean = wl.T * wl.k / wl.E                                 # 160 (80B), 256 (35B) tokens per expert
    assert counts.min() > 0.3 * mean and counts.max() < 2 * mean
    sample = covering_sample(ids, 512, wl.E)
    assert len(sample) >= 512
    assert len(np.unique(ids[sample])) == wl.E                # every expert's weights are checked
    ref = oracle_shards.tokens_sharded(wl.name, 0, x[sample], ids[sample], inp.Wr_bits[0], inp.ws_bits[0])
    routing_ok(ids[sample], w[sample], gate[sample], ref, wl.k)
    assert_output_close(out[sample], ref["out64"])
    assert np.array_equal(out, gpu_forward(pool, 0, x, ids, w, gate))


def test_prefill_at_the_token_limit():
    """T = SMOE_MAX_TOKENS (2^20 tokens, the largest call the boundary takes)
    on the tiny shape: about 262,000 pairs per expert (some 1,400 tiles each),
    the bucketed path's row offsets and the gather's byte offsets near their
    32-bit bounds. x is 16 seeded blocks of 65,536 tokens. The routing and
    outputs of a seeded sample that holds the first and last tokens, a token of
    every block and a token of every expert, against the oracle; every output
    finite."""
    wl = synthetic.WORKLOADS["tiny"]
    pool, inp = W.DevicePool(wl, n_layers=1), W.LayerInputs(wl, 1)
    T, blk = smoe.MAX_TOKENS, 1 << 16
    x = np.concatenate([synthetic.activations(wl.seed, blk, wl.H, tag=5000 + j) for j in range(T // blk)])
    ids, w, gate = gpu_route(pool, inp, 0, x)
    out = gpu_forward(pool, 0, x, ids, w, gate)
    assert np.isfinite(synthetic.bf16_bits_to_f32(out)).all()
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert counts.sum() == T * wl.k and counts.min() > 0
    edges = [0, 1, T - 2, T - 1] + [j * blk + 7 for j in range(T // blk)]
    sample = np.union1d(covering_sample(ids, 48, wl.E), edges)
    ref = oracle_shards.tokens_sharded(wl.name, 0, x[sample], ids[sample], inp.Wr_bits[0], inp.ws_bits[0])
    routing_ok(ids[sample], w[sample], gate[sample], ref, wl.k)
    assert_output_close(out[sample], ref["out64"])


def test_decode_and_prefill_agree(tiny):
    """Each token decoded alone (T = 1) equals the same tokens run as one
    batch through the bucketed path, within the layer tolerance."""
    pool, inp = tiny
    wl = pool.wl
    T = 24
    x = synthetic.activations(wl.seed, T, wl.H, tag=77)
    ref = oracle_layer(wl, 0, x, inp)
    batch = gpu_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"])
    single = np.concatenate([gpu_forward(pool, 0, x[t:t + 1], ref["ids"][t:t + 1], ref["w"][t:t + 1],
                                         ref["gate"][t:t + 1]) for t in range(T)])
    b = synthetic.bf16_bits_to_f32(batch).astype(np.float64)
    assert_output_close(single, b)


def test_prefill_slot_permutation_bit_identical():
    wl = synthetic.WORKLOADS["tiny"]
    a = W.DevicePool(wl)
    perm = np.random.default_rng(3).permutation(wl.E).astype(np.int32).reshape(1, wl.E)
    b = W.DevicePool(wl, table=perm)
    inp = W.LayerInputs(wl, 1)
    x = synthetic.activations(wl.seed, 100, wl.H, tag=1)
    ref = oracle_layer(wl, 0, x, inp)
    oa = gpu_forward(a, 0, x, ref["ids"], ref["w"], ref["gate"])
    ob = gpu_forward(b, 0, x, ref["ids"], ref["w"], ref["gate"])
    assert np.array_equal(oa, ob)


def test_prefill_bad_slot_sets_error_word(tiny):
    pool, inp = tiny
    wl = pool.wl
    T = 32
    x = synthetic.activations(wl.seed, T, wl.H, tag=31)
    ref = oracle_layer(wl, 0, x, inp)
    e = int(ref["ids"][0, 0])
    saved = pool.table_dev[0, e].item()
    try:
        pool.table_dev[0, e] = -5
        out = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        smoe.moe_forward(pool.ctx, 0, W.bf16_tensor(x), torch.from_numpy(ref["ids"]).cuda(),
                         torch.from_numpy(ref["w"].astype(np.float32)).cuda(),
                         torch.from_numpy(ref["gate"].astype(np.float32)).cuda(), pool.pool, pool.shared[0], out,
                         W.workspace(pool.ctx, T), err)
        assert smoe.check(err) == smoe.DEV_BAD_SLOT
        assert torch.isfinite(out.float()).all()
    finally:
        pool.table_dev[0, e] = saved
        torch.cuda.synchronize()


def test_token_limit_is_rejected_before_any_work(tiny):
    """T above SMOE_MAX_TOKENS (the limit that keeps every row offset of the
    bucketed path inside 32 bits) is refused at the boundary: no workspace
    size, and EINVAL from moe_route and moe_forward without touching memory."""
    pool, inp = tiny
    wl = pool.wl
    T = smoe.MAX_TOKENS + 1
    assert pool.ctx.workspace_bytes(smoe.MAX_TOKENS) > 0
    assert pool.ctx.workspace_bytes(T) == 0
    x = torch.zeros((8, wl.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((8, wl.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((8, wl.k), dtype=torch.float32, device="cuda")
    gate = torch.zeros(8, dtype=torch.float32, device="cuda")
    out = torch.zeros_like(x)
    ws = W.workspace(pool.ctx, 8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = smoe.lib()
    p = smoe._ptr
    st = L.moe_forward(pool.ctx.handle, 0, p(x), T, p(ids), p(w), p(gate), p(pool.pool),
                       pool.pool.numel() * pool.pool.element_size(), p(pool.shared[0]), None, p(out), p(ws),
                       ws.numel() * ws.element_size(), p(err), None)
    assert st == smoe.EINVAL
    st = L.moe_route(pool.ctx.handle, p(inp.Wr[0]), p(inp.ws[0]), p(x), T, None, p(ids), p(w), p(gate), p(ws),
                     ws.numel() * ws.element_size(), None)
    assert st == smoe.EINVAL
    torch.cuda.synchronize()
    assert smoe.check(err) == 0


@pytest.mark.parametrize("name,lengths", [("tiny", (37, 9, 120, 300, 12)), ("decode35b", (9, 64, 200, 31))])
def test_mixed_length_batch_equals_each_request(name, lengths):
    """Requests of different lengths concatenated into one call: every token's
    output is bit-identical to its own request's call (the same routing; all
    calls on the token-bucketed path, T > 8). A token's rows meet the same
    weights in the same K order whatever other tokens share its tiles."""
    wl = synthetic.WORKLOADS[name]
    pool, inp = W.DevicePool(wl, n_layers=1), W.LayerInputs(wl, 1)
    xs = [synthetic.activations(wl.seed, T, wl.H, tag=7000 + i) for i, T in enumerate(lengths)]
    x = np.concatenate(xs, 0)
    ids, w, gate = gpu_route(pool, inp, 0, x)
    full = gpu_forward(pool, 0, x, ids, w, gate)
    o = 0
    for T, xr in zip(lengths, xs):
        part = gpu_forward(pool, 0, xr, ids[o:o + T], w[o:o + T], gate[o:o + T])
        assert np.array_equal(part, full[o:o + T]), (T, o)
        o += T
    if name == "tiny":                                   # the whole batch against the oracle
        ref = oracle_layer(wl, 0, x, inp)
        assert_output_close(gpu_forward(pool, 0, x, ref["ids"], ref["w"], ref["gate"]), ref["out64"])
