"""CPU checks of the parity checker itself (no GPU): the routing rule accepts
exactly the valid top-k choices, and the sharded oracle helper returns what
one plain oracle call returns."""
import numpy as np
import pytest

import oracle
import oracle_shards
import synthetic
from test_gpu_parity import assert_output_close, assert_residual_close, routing_ok


@pytest.fixture(scope="module")
def tiny_ref():
    wl = synthetic.WORKLOADS["tiny"]
    x = synthetic.activations(wl.seed, 200, wl.H, tag=31)
    Wr = synthetic.router_weights(wl.seed, 0, wl.E, wl.H)
    ws = synthetic.shared_gate_weights(wl.seed, 0, wl.H)
    ids, w, gate, probs = oracle.route(x, Wr, ws, wl.k, want_probs=True)
    return wl, x, Wr, ws, dict(ids=ids, w=w, gate=gate, probs=probs)


def test_oracle_routing_passes(tiny_ref):
    wl, _, _, _, ref = tiny_ref
    w_own = routing_ok(ref["ids"], ref["w"].astype(np.float32), ref["gate"].astype(np.float32), ref, wl.k)
    assert np.allclose(w_own, ref["w"], rtol=0, atol=1e-15)


def test_wrong_expert_outside_the_tie_band_fails(tiny_ref):
    wl, _, _, _, ref = tiny_ref
    p = ref["probs"]
    ps = -np.sort(-p, axis=1)
    t = int(np.argmax(ps[:, wl.k - 1] - ps[:, wl.k]))          # the clearest cut
    bad = ref["ids"].copy()
    outside = [e for e in np.argsort(-p[t]) if e not in bad[t]][-1]   # the least likely expert
    bad[t, wl.k - 1] = outside
    with pytest.raises(AssertionError):
        routing_ok(bad[t:t + 1], ref["w"][t:t + 1], ref["gate"][t:t + 1], {k: v[t:t + 1] for k, v in ref.items()},
                   wl.k)


def test_swap_inside_a_near_tie_is_valid():
    """A made-up token whose k-th and (k+1)-th probabilities differ by 1e-6:
    choosing either is valid, and the weights checked are those of the choice."""
    k, E = 2, 4
    p = np.array([[0.5, 0.25 + 5e-7, 0.25 - 5e-7, 0.0]])
    ref = dict(probs=p, ids=np.array([[0, 1]], np.int32), gate=np.array([0.5]))
    for choice in ([0, 1], [0, 2]):
        ids = np.array([choice], np.int32)
        w = p[0, choice] / p[0, choice].sum()
        w_own = routing_ok(ids, w[None].astype(np.float32), np.array([0.5], np.float32), ref, k)
        assert np.allclose(w_own[0], w)
    with pytest.raises(AssertionError):                       # outside the band
        routing_ok(np.array([[0, 3]], np.int32), np.array([[1.0, 0.0]], np.float32), np.array([0.5], np.float32),
                   ref, k)
    with pytest.raises(AssertionError):                       # wrong weights for the choice
        routing_ok(np.array([[0, 2]], np.int32), np.array([[0.5, 0.5]], np.float32), np.array([0.5], np.float32),
                   ref, k)


def test_sharded_oracle_equals_one_call(tiny_ref):
    wl, x, Wr, ws, ref = tiny_ref
    x = x[:24]
    one = oracle.layer(wl, 0, x, Wr, ws, want_probs=True)
    par = oracle_shards.tokens_sharded(wl.name, 0, x, None, Wr, ws, shards=3)
    for key in ("ids", "w", "gate", "probs", "out64", "out_bf16"):
        assert np.array_equal(par[key], one[key]), key
    # the GPU's own choice equal to the oracle's gives the oracle's result
    own = oracle_shards.tokens_sharded(wl.name, 0, x, one["ids"], Wr, ws, shards=2)
    assert np.array_equal(own["out64"], one["out64"])


def test_residual_rule_allows_the_output_rounding_only(tiny_ref):
    wl, x, Wr, ws, _ = tiny_ref
    one = oracle.layer(wl, 0, x[:4], Wr, ws)
    exact = oracle.residual(x[:4], one["out64"])
    assert_residual_close(exact, x[:4], one["out64"])
    off = exact.copy()
    off[0, 0] += 3                                            # three bf16 units away
    with pytest.raises(AssertionError):
        assert_residual_close(off, x[:4], one["out64"])


def test_exactly_rounded_output_passes_the_output_rule():
    """The oracle's own round-to-nearest bf16 output must pass the output rule:
    on this input its rounding alone is 1.15e-4 while 2e-2 rms is 1.11e-4 (an
    element of 6.3 rms just above a power of two), which is why the rule adds
    half a bf16 unit. Two units off still fails."""
    wl = synthetic.WORKLOADS["tiny"]
    x = synthetic.activations(wl.seed, 64, wl.H, tag=64)
    one = oracle.layer(wl, 0, x, synthetic.router_weights(wl.seed, 0, wl.E, wl.H),
                       synthetic.shared_gate_weights(wl.seed, 0, wl.H))
    y, yb = one["out64"], one["out_bf16"]
    rounding = np.abs(synthetic.bf16_bits_to_f32(yb).astype(np.float64) - y).max()
    assert rounding > 2e-2 * np.sqrt(np.mean(y ** 2))
    assert_output_close(yb, y)
    i = np.unravel_index(np.abs(y).argmax(), y.shape)
    off = yb.copy()
    off[i] += 2
    with pytest.raises(AssertionError):
        assert_output_close(off, y)
