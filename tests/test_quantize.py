"""smoe_quantize_mlx (the library's host quantiser, float32 -> MLX affine
triples) against the oracle's independently written quantiser: the same bits
on random, constant, one-signed, tiny and near-fp16-limit groups, 4- and
8-bit; the dequantisation error bound |w - (s q + b)| <= s / 2; the calls it
refuses; and triples it produces packed by pack_experts into the blob the
oracle's reader parses back."""
import numpy as np
import pytest

import int4_routed_expert_router_gb300 as smoe
import oracle


def cases(rng):
    yield rng.standard_normal((8, 256)).astype(np.float32) * 0.02
    yield np.full((2, 128), 0.37, np.float32)                               # constant groups: s = 0
    yield -np.abs(rng.standard_normal((4, 64)).astype(np.float32))          # one sign
    yield (rng.standard_normal((4, 192)) * 1e-6).astype(np.float32)         # fp16 subnormal range
    yield (rng.uniform(-6.0e4, 6.0e4, (2, 64))).astype(np.float32)          # near the fp16 limit
    w = rng.standard_normal((3, 128)).astype(np.float32)
    w[:, ::7] = 0.0                                                         # exact zeros, ties
    yield w


@pytest.mark.parametrize("bits", [4, 8])
def test_quantize_matches_oracle(bits):
    rng = np.random.default_rng(41 + bits)
    for w in cases(rng):
        q, s, b = smoe.quantize_mlx(w, bits)
        qo, so, bo = (oracle.quantize if bits == 4 else oracle.quantize8)(w.astype(np.float64))
        assert np.array_equal(q, qo) and np.array_equal(s, so) and np.array_equal(b, bo)


@pytest.mark.parametrize("bits", [4, 8])
def test_quantize_error_bound(bits):
    rng = np.random.default_rng(7 + bits)
    for w in cases(rng):
        q, s, b = smoe.quantize_mlx(w, bits)
        deq = (oracle.dequant if bits == 4 else oracle.dequant8)(q, s, b)
        sv = np.repeat(s.view(np.float16).astype(np.float64), 64, axis=1)
        assert np.all(np.abs(w.astype(np.float64) - deq) <= sv / 2 * (1 + 1e-12) + 1e-300)


def test_quantize_refusals():
    w = np.zeros((2, 64), np.float32)
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.quantize_mlx(np.zeros((2, 96), np.float32), 4)                 # cols % 64
    assert ei.value.status == smoe.ENOTSUP
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.quantize_mlx(w, 6)
    assert ei.value.status == smoe.ENOTSUP
    bad = w.copy()
    bad[1, 3] = np.inf
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.quantize_mlx(bad, 4)
    assert ei.value.status == smoe.ERANGE
    big = w.copy()
    big[0, 0] = 1e6
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.quantize_mlx(big, 8)
    assert ei.value.status == smoe.ERANGE


def test_quantized_expert_packs_and_reads_back():
    """Float weights of one tiny expert -> smoe_quantize_mlx -> pack_experts
    (host) -> the oracle's blob reader gives back the same triples."""
    H, I = 256, 64
    rng = np.random.default_rng(5)
    mats = [rng.standard_normal((I, H)).astype(np.float32) * 0.05, rng.standard_normal((I, H)).astype(np.float32) * 0.05,
            rng.standard_normal((H, I)).astype(np.float32) * 0.05]
    trip = [smoe.quantize_mlx(m, 4) for m in mats]
    arrays = [a for t in trip for a in t]                  # gate q, s, b, up q, s, b, down q, s, b
    shape = smoe.make_shape(H, 16, 4, I)
    stride = smoe.layout_of(shape).blob_bytes
    blob = np.zeros(stride, np.uint8)
    smoe.pack_experts(shape, [arrays], [0], blob, blob.size, smoe.HOST)
    back = oracle.blob_to_mlx(blob, H, I)
    for want, got in zip(arrays, back):
        assert np.array_equal(np.asarray(want).ravel(), np.asarray(got).ravel())
