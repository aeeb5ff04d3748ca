"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a closed form, a special case that reduces
to a library routine (torch CPU fp64), brute force, or an invariant the pages
state (Swiftlet pages: cache/disk give the same answer; incremental decode
matches the full sequence). Chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synthetic

TINY = synthetic.WORKLOADS["tiny"]


def tiny_inputs(seed=TINY.seed, T=TINY.T, layer=0):
    x = synthetic.activations(seed, T, TINY.H)
    Wr = synthetic.router_weights(seed, layer, TINY.E, TINY.H)
    ws = synthetic.shared_gate_weights(seed, layer, TINY.H)
    return x, Wr, ws


def torch_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


def torch_f16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.float16)


# ---------------------------------------------------------------- conversions

def test_bf16_and_f16_decode_match_torch_on_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref_b = torch_bf16(pats).to(torch.float64).numpy()
    ref_h = torch_f16(pats).to(torch.float64).numpy()
    got_b = oracle.bf16_to_f64(pats)
    got_h = oracle.f16_to_f64(pats)
    fin = np.isfinite(ref_b)
    assert np.array_equal(got_b[fin], ref_b[fin])
    assert np.array_equal(np.isnan(got_b), np.isnan(ref_b))
    fin = np.isfinite(ref_h)
    assert np.array_equal(got_h[fin], ref_h[fin])
    assert np.array_equal(np.isinf(got_h), np.isinf(ref_h))


def test_rounding_to_bf16_and_f16_matches_torch_rne():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 8, 20000),
        # exact halfway cases between neighbours exercise ties-to-even
        (torch_bf16(np.arange(0x3f00, 0x3f40, dtype=np.uint16)).float().numpy() + 2.0 ** -9).astype(np.float64),
        np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 65519.0, 65520.0, 1e-8, -6e-8]),
    ]).astype(np.float32).astype(np.float64)   # fp32 inputs: torch rounds from fp32
    ref_b = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref_h = torch.from_numpy(v.astype(np.float32)).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(v), ref_b)
    assert np.array_equal(oracle.f64_to_f16(v), ref_h)


# ------------------------------------------------------------- dequantisation

def test_dequant_matches_byte_table_unpack():
    """A second unpack: a 256-entry byte table, byte j of a word = columns 2j, 2j+1."""
    rng = np.random.default_rng(11)
    rows, cols = 24, 192
    q = rng.integers(0, 2 ** 32, size=(rows, cols // 8), dtype=np.uint64).astype(np.uint32)
    s = oracle.f64_to_f16(rng.uniform(1e-3, 1e-1, size=(rows, cols // 64)))
    b = oracle.f64_to_f16(rng.uniform(-1, 1, size=(rows, cols // 64)))
    table = np.array([[byte & 15, byte >> 4] for byte in range(256)], dtype=np.int64)
    nib = table[q.view(np.uint8).reshape(rows, cols // 2)].reshape(rows, cols)   # little-endian bytes
    sc = torch_f16(s).double().numpy().repeat(64, axis=1)
    bi = torch_f16(b).double().numpy().repeat(64, axis=1)
    assert np.array_equal(oracle.dequant(q, s, b), sc * nib + bi)


@pytest.mark.parametrize("lo,hi", [(-0.05, 0.05), (0.0, 1.0), (-3.0, -2.5), (1e-4, 2e-4)])
def test_quantize_dequantize_error_at_most_half_scale(lo, hi):
    rng = np.random.default_rng(int(1e4 * (hi - lo)))
    W = rng.uniform(lo, hi, size=(16, 256))
    W[3, 64:128] = W[3, 64]          # a constant group
    q, s, b = oracle.quantize(W)
    Wd = oracle.dequant(q, s, b)
    sc = oracle.f16_to_f64(s).repeat(64, axis=1)
    err = np.abs(Wd - W)
    assert np.all(err <= sc / 2 * (1 + 1e-12) + 1e-300)


# ------------------------------------------------------------------- routing

def test_zero_input_closed_form():
    """x = 0: all logits 0, uniform p, ties go to the lowest ids, w = 1/k,
    gate = sigmoid(0) = 1/2, every expert sees g = u = 0 so out = 0."""
    x = np.zeros((2, TINY.H), np.uint16)
    _, Wr, ws = tiny_inputs()
    r = oracle.layer(TINY, 0, x, Wr, ws)
    assert np.array_equal(r["ids"], np.tile(np.arange(TINY.k, dtype=np.int32), (2, 1)))
    assert np.all(r["w"] == 1.0 / TINY.k)
    assert np.all(r["gate"] == 0.5)
    assert np.all(r["out64"] == 0.0)


def test_topk_brute_force_over_all_subsets():
    x, Wr, ws = tiny_inputs()
    ids, w, gate, p = oracle.route(x, Wr, ws, TINY.k, want_probs=True)
    for t in range(TINY.T):
        best = max(itertools.combinations(range(TINY.E), TINY.k), key=lambda c: sum(p[t, list(c)]))
        assert set(best) == set(ids[t].tolist())
        assert all(p[t, ids[t, j]] >= p[t, ids[t, j + 1]] for j in range(TINY.k - 1))


def test_renormalised_weights_equal_softmax_over_chosen_logits():
    """softmax -> top-k -> renormalise equals a softmax over the k chosen logits."""
    x, Wr, ws = tiny_inputs()
    bias = synthetic.zipf_bias(3, TINY.E)
    ids, w, gate = oracle.route(x, Wr, ws, TINY.k, bias=bias)
    z = torch_bf16(x).double() @ torch_bf16(Wr).double().T + torch.from_numpy(bias).double()
    for t in range(TINY.T):
        ref = torch.softmax(z[t, torch.from_numpy(ids[t]).long()], dim=0).numpy()
        assert np.allclose(w[t], ref, rtol=1e-13, atol=0)
        assert math.isclose(gate[t], torch.sigmoid(torch_bf16(x[t]).double() @ torch_bf16(ws).double()).item(),
                            rel_tol=1e-14)


def _torch_expert(tr, x64):
    G = torch.from_numpy(oracle.dequant(tr.gate_q, tr.gate_s, tr.gate_b))
    U = torch.from_numpy(oracle.dequant(tr.up_q, tr.up_s, tr.up_b))
    D = torch.from_numpy(oracle.dequant(tr.down_q, tr.down_s, tr.down_b))
    return F.linear(F.silu(F.linear(x64, G)) * F.linear(x64, U), D)


def test_k_equals_E_is_dense_softmax_mixture():
    """With k = E the layer is sum_e softmax(z)_e f_e(x) + sigmoid(w_s.x) f_s(x),
    evaluated here with torch fp64 (no sort, no renormalisation)."""
    wl = TINY
    x, Wr, ws = tiny_inputs()
    ids, w, gate = oracle.route(x, Wr, ws, wl.E)
    experts = {e: synthetic.expert_triples(wl.seed, 0, e, wl.H, wl.I) for e in range(wl.E)}
    shared = synthetic.expert_triples(wl.seed, 0, None, wl.H, wl.I_shared)
    out64, _ = oracle.combine(x, ids, w, gate, experts, shared, wl.E, wl.I, wl.I_shared)
    x64 = torch_bf16(x).double()
    p = torch.softmax(x64 @ torch_bf16(Wr).double().T, dim=1)
    ref = sum(p[:, e:e + 1] * _torch_expert(experts[e], x64) for e in range(wl.E))
    ref = ref + torch.sigmoid(x64 @ torch_bf16(ws).double())[:, None] * _torch_expert(shared, x64)
    assert np.allclose(out64, ref.numpy(), rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("k", [1, 3])
def test_one_hot_router_is_one_dense_swiglu_mlp(k):
    wl = TINY
    x, Wr, ws = tiny_inputs()
    star = 5
    bias = np.full(wl.E, -np.inf, np.float32)
    bias[star] = 0.0
    ids, w, gate = oracle.route(x, Wr, ws, k, bias=bias)
    assert np.all(ids[:, 0] == star)
    assert np.all(w[:, 0] == 1.0) and np.all(w[:, 1:] == 0.0)
    experts = {e: synthetic.expert_triples(wl.seed, 0, e, wl.H, wl.I) for e in np.unique(ids)}
    shared = synthetic.expert_triples(wl.seed, 0, None, wl.H, wl.I_shared)
    out64, outb = oracle.combine(x, ids, w, gate, experts, shared, wl.E, wl.I, wl.I_shared)
    x64 = torch_bf16(x).double()
    ref = _torch_expert(experts[star], x64) + \
        torch.sigmoid(x64 @ torch_bf16(ws).double())[:, None] * _torch_expert(shared, x64)
    assert np.allclose(out64, ref.numpy(), rtol=1e-12, atol=1e-15)


def test_constant_expert_closed_form():
    """Hand-built expert: gate weights 0.5, up 1.0, down 0.25 (q = 8 and
    power-of-two scales, zero bias). With x = e_c (one-hot, value 1) every
    intermediate is silu(0.5) * 1 and every output is I * 0.25 * silu(0.5)."""
    H, I = 128, 64

    def const(rows, cols, s):
        q = np.full((rows, cols // 8), 0x88888888, np.uint32)
        sb = np.full((rows, cols // 64), oracle.f64_to_f16([s])[0], np.uint16)
        return q, sb, np.zeros((rows, cols // 64), np.uint16)

    gq, gs, gb = const(I, H, 1 / 16)
    uq, us, ub = const(I, H, 1 / 8)
    dq, ds, db = const(H, I, 1 / 32)
    ex = synthetic.ExpertTriples(gq, gs, gb, uq, us, ub, dq, ds, db)
    x = np.zeros((1, H), np.uint16)
    x[0, 17] = 0x3f80                                   # bf16 1.0
    ids = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1))
    gate = np.array([0.25])
    out64, _ = oracle.combine(x, ids, w, gate, {0: ex}, ex, 1, I, I)
    silu = 0.5 / (1 + math.exp(-0.5))
    assert np.allclose(out64, (1 + 0.25) * I * 0.25 * silu, rtol=1e-15)


# --------------------------------------------------------------- invariants

def test_token_by_token_equals_full_sequence():
    x, Wr, ws = tiny_inputs(T=6)
    full = oracle.layer(TINY, 0, x, Wr, ws)
    for t in range(6):
        one = oracle.layer(TINY, 0, x[t:t + 1], Wr, ws)
        assert np.array_equal(one["ids"][0], full["ids"][t])
        assert np.array_equal(one["out64"][0], full["out64"][t])
        assert np.array_equal(one["out_bf16"][0], full["out_bf16"][t])


def test_residual_chain_rounds_once():
    x = synthetic.activations(5, 2, 64)
    y = np.random.default_rng(0).standard_normal((2, 64)) * 0.1
    got = oracle.residual(x, y)
    ref = oracle.f64_to_bf16(oracle.bf16_to_f64(x) + y)
    assert np.array_equal(got, ref)


def test_oracle_reproduces_stored_tiny_fixture():
    """Regression guard (see tests/golden/README.md): bit-identical on this host."""
    import os
    import importlib.util
    path = os.path.join(os.path.dirname(__file__), "golden", "make_golden.py")
    spec = importlib.util.spec_from_file_location("make_golden", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    ref = np.load(os.path.join(os.path.dirname(__file__), "golden", "tiny_layer.npz"))
    got = mod.compute()
    for key in ref.files:
        assert np.array_equal(got[key], ref[key]), key


# --------------------------------------------------------------- 8-bit experts

def test_dequant8_matches_byte_view_unpack():
    """8-bit MLX words: a second unpack that reads the words as little-endian
    bytes (byte j of a word = column 4 w + j)."""
    rng = np.random.default_rng(12)
    rows, cols = 24, 192
    q = rng.integers(0, 2 ** 32, size=(rows, cols // 4), dtype=np.uint64).astype(np.uint32)
    s = oracle.f64_to_f16(rng.uniform(1e-4, 1e-2, size=(rows, cols // 64)))
    b = oracle.f64_to_f16(rng.uniform(-1, 1, size=(rows, cols // 64)))
    byte = q.view(np.uint8).reshape(rows, cols).astype(np.int64)
    sc = torch_f16(s).double().numpy().repeat(64, axis=1)
    bi = torch_f16(b).double().numpy().repeat(64, axis=1)
    assert np.array_equal(oracle.dequant8(q, s, b), sc * byte + bi)


@pytest.mark.parametrize("lo,hi", [(-0.05, 0.05), (0.0, 1.0), (-3.0, -2.5), (1e-4, 2e-4)])
def test_quantize8_dequantize_error_at_most_half_scale(lo, hi):
    rng = np.random.default_rng(int(1e4 * (hi - lo)) + 1)
    W = rng.uniform(lo, hi, size=(16, 256))
    W[3, 64:128] = W[3, 64]          # a constant group
    q, s, b = oracle.quantize8(W)
    Wd = oracle.dequant8(q, s, b)
    sc = oracle.f16_to_f64(s).repeat(64, axis=1)
    assert np.all(np.abs(Wd - W) <= sc / 2 * (1 + 1e-12) + 1e-300)
    # 255 steps: about 17 times finer than the 4-bit quantiser on the same groups
    s4 = oracle.f16_to_f64(oracle.quantize(W)[1])
    assert np.median(s4 / np.maximum(oracle.f16_to_f64(s), 1e-300)) > 15


def test_dense_combine_equals_the_4_bit_combine():
    """combine_dense (experts given as fp64 weights) is the same definition as
    the pinned 4-bit combine: fed the 4-bit experts' exact dequantisation, its
    output is bit-identical, including a repeated expert within a token."""
    x, Wr, ws = tiny_inputs(T=5)
    ids, w, gate = oracle.route(x, Wr, ws, TINY.k)
    ids[2, 1] = ids[2, 0]
    experts = {int(e): synthetic.expert_triples(TINY.seed, 0, int(e), TINY.H, TINY.I) for e in np.unique(ids)}
    shared = synthetic.expert_triples(TINY.seed, 0, None, TINY.H, TINY.I)
    want, want_b = oracle.combine(x, ids, w, gate, experts, shared, TINY.E, TINY.I, TINY.I)
    dq = lambda t: (oracle.dequant(t.gate_q, t.gate_s, t.gate_b), oracle.dequant(t.up_q, t.up_s, t.up_b),
                    oracle.dequant(t.down_q, t.down_s, t.down_b))
    got, got_b = oracle.combine_dense(x, ids, w, gate, {e: dq(t) for e, t in experts.items()}, dq(shared),
                                      TINY.E, TINY.I, TINY.I)
    assert np.array_equal(got, want) and np.array_equal(got_b, want_b)
    with pytest.raises(ValueError):
        oracle.combine_dense(x, ids, w, gate, {}, dq(shared), TINY.E, TINY.I, TINY.I)


def test_8_bit_layer_one_hot_router_is_one_dense_swiglu_mlp():
    """An 8-bit layer with k = 1 and the shared gate at 0 is one expert's
    SwiGLU MLP on its dequantised weights (torch CPU fp64)."""
    x, Wr, ws = tiny_inputs(T=3)
    ids = np.full((3, 1), 5, np.int32)
    w = np.ones((3, 1))
    gate = np.zeros(3)
    tr = synthetic.expert_triples(TINY.seed, 0, 5, TINY.H, TINY.I, bits=8)
    sh = synthetic.expert_triples(TINY.seed, 0, None, TINY.H, TINY.I, bits=8)
    out, _ = oracle.combine8(x, ids, w, gate, {5: tr}, sh, TINY.E, TINY.I, TINY.I)
    G, U, D = (torch.from_numpy(m) for m in oracle.dense_of8(tr))
    xt = torch_bf16(x).double()
    ref = (F.silu(xt @ G.T) * (xt @ U.T)) @ D.T
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
