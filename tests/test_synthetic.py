"""Host side of the seeded input generator: recipe and determinism (no GPU)."""
import numpy as np

import synthetic


def test_splitmix64_known_values():
    # SplitMix64 seeded with 0 yields these first outputs (state advances by GOLDEN).
    z = synthetic.GOLDEN * np.arange(1, 4, dtype=np.uint64)
    out = synthetic.splitmix64(z)
    assert [hex(int(v)) for v in out] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4", "0x6c45d188009454f"]


def test_expert_recipe_ranges_and_determinism():
    t1 = synthetic.expert_triples(7, 3, 11, 512, 128)
    t2 = synthetic.expert_triples(7, 3, 11, 512, 128)
    t3 = synthetic.expert_triples(7, 3, 12, 512, 128)
    for a, b in zip(t1.arrays(), t2.arrays()):
        assert np.array_equal(a, b)
    assert not np.array_equal(t1.gate_q, t3.gate_q)
    assert not np.array_equal(t1.gate_q, t1.up_q)
    nib = np.stack([(t1.gate_q >> np.uint32(4 * i)) & np.uint32(15) for i in range(8)]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16
    s = t1.gate_s.view(np.float16).astype(np.float64)
    b = t1.gate_b.view(np.float16).astype(np.float64)
    assert s.min() >= 0.0019 and s.max() <= 0.00601
    assert np.array_equal(b, (-7.5 * s).astype(np.float16).astype(np.float64))
    assert t1.gate_q.shape == (128, 64) and t1.down_q.shape == (512, 16) and t1.down_s.shape == (512, 2)


def test_dense_tensors():
    x = synthetic.activations(1, 64, 2048)
    xf = synthetic.bf16_bits_to_f32(x)
    assert abs(xf.mean()) < 0.02 and abs(xf.std() - 1) < 0.02
    Wr = synthetic.bf16_bits_to_f32(synthetic.router_weights(1, 0, 256, 2048))
    assert abs(Wr.std() - 0.02) < 0.001
    tab = synthetic.slot_table(3, 4, 16, permuted=True)
    assert sorted(tab.ravel().tolist()) == list(range(64))
    z = synthetic.zipf_bias(3, 16)
    assert np.isclose(np.sort(z)[::-1][0], 0.0) and np.isclose(z.min(), -1.1 * np.log(16))


def test_expert_recipe_8_bit():
    """8-bit triples: 4 values per word, every byte value equally likely,
    s = the 4-bit recipe's / 17 and b = -127.5 s, so the weight range is the
    4-bit recipe's; the 4-bit draw is unchanged by the option."""
    t = synthetic.expert_triples(7, 3, 11, 512, 128, bits=8)
    assert t.gate_q.shape == (128, 128) and t.down_q.shape == (512, 32) and t.down_s.shape == (512, 2)
    q = np.stack([(t.gate_q >> np.uint32(8 * i)) & np.uint32(255) for i in range(4)]).ravel()
    counts = np.bincount(q, minlength=256)
    assert counts.min() > 0.75 * q.size / 256 and counts.max() < 1.25 * q.size / 256
    s = t.gate_s.view(np.float16).astype(np.float64)
    b = t.gate_b.view(np.float16).astype(np.float64)
    assert s.min() >= 0.0019 / 17 and s.max() <= 0.00601 / 17
    assert np.array_equal(b, (-127.5 * s).astype(np.float16).astype(np.float64))
    t4 = synthetic.expert_triples(7, 3, 11, 512, 128)
    assert np.array_equal(t4.gate_s, synthetic.expert_triples(7, 3, 11, 512, 128, bits=4).gate_s)
    s4 = t4.gate_s.view(np.float16).astype(np.float64)
    # both are one fp16 rounding of the same draw (divided by 17 for s): two half-ulps apart at most
    assert np.all(np.abs(s - s4 / 17) <= 2 ** -10 * s4 / 17)
