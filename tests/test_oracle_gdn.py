"""Pins of the oracle's Gated DeltaNet step (no GPU): closed forms that the
gated delta rule fixes, an independent algebraic form of the update, and
token-by-token equal to a multi-token call. Each is written from the rule's
definition, not from the oracle's code path."""
import numpy as np
import pytest

import oracle
import synthetic


def f64(bits):
    return synthetic.bf16_bits_to_f32(bits).astype(np.float64)


def unit(a, mul=1.0):
    return a * (mul / np.sqrt(np.sum(a * a, axis=-1, keepdims=True) + 1e-6))


def inputs(T=1, B=2, nk=2, nv=4, dk=32, dv=24, tag=0):
    return synthetic.gdn_inputs(77, T, B, nk, nv, dk, dv, tag=tag)


def test_no_write_is_pure_decay():
    """beta = 0: S' = alpha S and o = S' q^."""
    q, k, v, g, beta, S0 = inputs()
    beta = np.zeros_like(beta)
    S, o = oracle.gdn_step(q, k, v, g, beta, S0)
    alpha = np.exp(g.astype(np.float64))[0]
    want = S0.astype(np.float64) * alpha[:, :, None, None]
    assert np.allclose(S, want, rtol=1e-14, atol=1e-15)
    qn = unit(f64(q)[0], 32 ** -0.5)
    qh = np.repeat(qn, 2, axis=1)                        # value heads 2h, 2h + 1 use key head h
    assert np.allclose(o[0], np.einsum("bhij,bhj->bhi", want, qh), rtol=1e-12, atol=1e-14)


def test_empty_state_takes_the_outer_product():
    """S = 0: S' = beta v k^T and o = beta v (k^ . q^)."""
    q, k, v, g, beta, S0 = inputs(tag=1)
    S, o = oracle.gdn_step(q, k, v, g, beta, np.zeros_like(S0))
    kn = np.repeat(unit(f64(k)[0]), 2, axis=1)
    qn = np.repeat(unit(f64(q)[0], 32 ** -0.5), 2, axis=1)
    b = beta.astype(np.float64)[0][:, :, None]
    vv = f64(v)[0]
    assert np.allclose(S, (b * vv)[..., None] * kn[:, :, None, :], rtol=1e-14, atol=1e-16)
    assert np.allclose(o[0], b * vv * np.sum(kn * qn, -1, keepdims=True), rtol=1e-12, atol=1e-14)


def test_full_write_maps_the_key_to_the_value():
    """beta = 1: whatever alpha, the new state reads v back for k^ (the delta
    rule's defining property), up to the 1e-6 in k^'s norm."""
    q, k, v, g, beta, S0 = inputs(tag=2)
    S, _ = oracle.gdn_step(q, k, v, g, np.ones_like(beta), S0)
    kn = np.repeat(unit(f64(k)[0]), 2, axis=1)
    assert np.allclose(np.einsum("bhij,bhj->bhi", S, kn), f64(v)[0], rtol=0, atol=1e-6)


def test_transition_matrix_form():
    """S' = alpha S (I - beta k^ k^T) + beta v k^T, o = S' q^, built with
    numpy matrix products (another form of the update than the oracle's
    rank-one correction), over grouped heads."""
    q, k, v, g, beta, S0 = inputs(B=2, nk=2, nv=4, dk=32, dv=24, tag=3)
    S, o = oracle.gdn_step(q, k, v, g, beta, S0)
    for b in range(2):
        for h in range(4):
            kn = unit(f64(k)[0, b, h // 2])
            qn = unit(f64(q)[0, b, h // 2], 32 ** -0.5)
            a, bt = np.exp(float(g[0, b, h])), float(beta[0, b, h])
            M = np.eye(32) - bt * np.outer(kn, kn)
            want = a * S0[b, h].astype(np.float64) @ M + bt * np.outer(f64(v)[0, b, h], kn)
            assert np.allclose(S[b, h], want, rtol=1e-12, atol=1e-14)
            assert np.allclose(o[0, b, h], want @ qn, rtol=1e-12, atol=1e-13)


def test_token_by_token_equals_one_call():
    q, k, v, g, beta, S0 = inputs(T=5, tag=4)
    S_all, o_all = oracle.gdn_step(q, k, v, g, beta, S0)
    S = S0.astype(np.float64)
    for t in range(5):
        S, o = oracle.gdn_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S)
        assert np.array_equal(o[0], o_all[t])
    assert np.array_equal(S, S_all)


def test_bad_shape_is_refused():
    q, k, v, g, beta, S0 = inputs(nk=3, nv=4)
    with pytest.raises(ValueError):
        oracle.gdn_step(q, k, v, g, beta, S0)
