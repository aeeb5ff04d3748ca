"""Seeded synthetic inputs for the int4 routed-expert MoE layer.

This module only draws numbers. It holds none of the layer's arithmetic (no
dequantisation, routing, MLP or combine). Both the CPU oracle (``oracle/``) and
the CUDA library receive the arrays it returns, so they see identical inputs.

Two generators are used:

* Expert weights (the big expert pool, tens of GB at the 80B shape) come from a
  counter-based generator: ``value(key, i) = splitmix64(key + GOLDEN*(i+1))``
  where ``splitmix64`` is the output mix of Steele, Lea and Flood's SplitMix64
  ("Fast splittable pseudorandom number generators", OOPSLA 2014). Any word of
  any expert can be produced on its own, so the oracle regenerates only the
  experts it needs, and ``synthetic/csrc/synth.cu`` produces the same bytes on
  the device for the full pool.
* Dense tensors (activations, router rows, shared-gate vector) are drawn on the
  host with numpy's Philox4x32 counter-based generator (Salmon et al., SC'11)
  and copied to the device.

Distributions (the workloads of the Swiftlet pages, shapes of Qwen3.6-35B-A3B
and Qwen3-Next-80B-A3B):
  q ~ U{0..15} (every bit of a q word is uniform, 8 nibbles per uint32)
  s ~ U[0.002, 0.006] rounded to fp16; b = fp16(-7.5 * s)
  8-bit experts (MLX's 8-bit affine format, 4 values per uint32): q ~ U{0..255},
  s ~ U[0.002, 0.006] / 17 rounded to fp16, b = fp16(-127.5 * s), so the
  weights span the same range as the 4-bit recipe's
  router rows, shared-gate vector ~ N(0, 0.02) -> fp32 -> bf16 (RNE)
  activations ~ N(0, 1) -> fp32 -> bf16 (RNE)
"""
from __future__ import annotations

import dataclasses
import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids inside one expert
TID_GATE_Q, TID_GATE_S, TID_UP_Q, TID_UP_S, TID_DOWN_Q, TID_DOWN_S = 1, 2, 3, 4, 5, 6
SHARED_EXPERT_CODE = (1 << 26) - 1   # expert code of the shared expert of a layer
GROUP = 64


def splitmix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output mix on uint64 arrays (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int, layer: int, expert_code: int) -> np.uint64:
    """Key of one tensor of one expert: mixes (seed, tensor id, layer, expert)."""
    assert 0 <= tid < (1 << 12) and 0 <= layer < (1 << 26) and 0 <= expert_code < (1 << 26)
    s = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    tag = np.uint64((tid << 52) | (layer << 26) | expert_code)
    with np.errstate(over="ignore"):
        return splitmix64((s * GOLDEN) ^ tag)[0]


def stream_values(key: np.uint64, index: np.ndarray) -> np.ndarray:
    """value(key, i) = splitmix64(key + GOLDEN * (i + 1)) for uint64 indices i."""
    i = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return splitmix64(key + GOLDEN * (i + np.uint64(1)))


def q_words(key: np.uint64, rows: int, cols: int) -> np.ndarray:
    """uint32 [rows, cols/8]: word w is half (w & 1) of value(key, w >> 1)."""
    n = rows * (cols // 8)
    w = np.arange(n, dtype=np.uint64)
    v = stream_values(key, w >> np.uint64(1))
    out = (v >> (np.uint64(32) * (w & np.uint64(1)))) & np.uint64(0xFFFFFFFF)
    return out.astype(np.uint32).reshape(rows, cols // 8)


def q_words8(key: np.uint64, rows: int, cols: int) -> np.ndarray:
    """uint32 [rows, cols/4] of 8-bit values (column c of a row in bits
    8*(c % 4) .. of word c/4): word w is half (w & 1) of value(key, w >> 1)."""
    n = rows * (cols // 4)
    w = np.arange(n, dtype=np.uint64)
    v = stream_values(key, w >> np.uint64(1))
    out = (v >> (np.uint64(32) * (w & np.uint64(1)))) & np.uint64(0xFFFFFFFF)
    return out.astype(np.uint32).reshape(rows, cols // 4)


def scale_bias(key: np.uint64, rows: int, cols: int, bits: int = 4):
    """fp16 bits [rows, cols/64] of s ~ U[0.002, 0.006] and b = fp16(-7.5 s)
    (bits = 8: s ~ U[0.002, 0.006] / 17 and b = fp16(-127.5 s)).

    u = value >> 40 (24 uniform bits); s = fp16_rne(0.002 + 0.004 * (u / 2^24))
    (divided by 17 for 8 bits), with the double operations rounded separately
    (no fused multiply-add).
    """
    n = rows * (cols // GROUP)
    v = stream_values(key, np.arange(n, dtype=np.uint64))
    u = (v >> np.uint64(40)).astype(np.float64) / 16777216.0
    t = np.multiply(0.004, u)
    s64 = np.add(0.002, t)
    if bits == 8:
        s64 = np.divide(s64, 17.0)
    s16 = s64.astype(np.float16)
    b16 = np.multiply(-7.5 if bits == 4 else -127.5, s16.astype(np.float64)).astype(np.float16)
    return (s16.view(np.uint16).reshape(rows, cols // GROUP),
            b16.view(np.uint16).reshape(rows, cols // GROUP))


@dataclasses.dataclass
class ExpertTriples:
    """MLX affine triples of one expert (q uint32 words, s/b fp16 bits).

    4 bits: gate, up: q [I, H/8], s/b [I, H/64]; down: q [H, I/8], s/b [H, I/64];
    within a word, column c of the row sits in bits 4*(c % 8) .. 4*(c % 8)+3.
    8 bits: q [I, H/4] and [H, I/4], column c in bits 8*(c % 4) .. 8*(c % 4)+7.
    """
    gate_q: np.ndarray
    gate_s: np.ndarray
    gate_b: np.ndarray
    up_q: np.ndarray
    up_s: np.ndarray
    up_b: np.ndarray
    down_q: np.ndarray
    down_s: np.ndarray
    down_b: np.ndarray

    def arrays(self):
        return [self.gate_q, self.gate_s, self.gate_b, self.up_q, self.up_s,
                self.up_b, self.down_q, self.down_s, self.down_b]


def expert_triples(seed: int, layer: int, expert: int | None, H: int, I: int, bits: int = 4) -> ExpertTriples:
    """Triples of routed expert ``expert`` (or the shared expert if None), with
    4-bit (default) or 8-bit q."""
    assert bits in (4, 8)
    code = SHARED_EXPERT_CODE if expert is None else int(expert)
    k = lambda tid: stream_key(seed, tid, layer, code)
    qw = q_words if bits == 4 else q_words8
    gs, gb = scale_bias(k(TID_GATE_S), I, H, bits)
    us, ub = scale_bias(k(TID_UP_S), I, H, bits)
    ds, db = scale_bias(k(TID_DOWN_S), H, I, bits)
    return ExpertTriples(qw(k(TID_GATE_Q), I, H), gs, gb,
                         qw(k(TID_UP_Q), I, H), us, ub,
                         qw(k(TID_DOWN_Q), H, I), ds, db)


# ---------------------------------------------------------------- dense tensors

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _philox(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed & 0xFFFFFFFFFFFFFFFF, stream]))


_STREAM_X, _STREAM_WR, _STREAM_WS, _STREAM_PERM, _STREAM_ZIPF = 1, 2, 3, 4, 5


def normal_bf16(seed: int, stream: int, shape, std: float) -> np.ndarray:
    g = _philox(seed, stream)
    v = g.standard_normal(size=shape, dtype=np.float64) * std
    return f32_to_bf16_bits(v.astype(np.float32))


def activations(seed: int, T: int, H: int, tag: int = 0) -> np.ndarray:
    """x [T, H] bf16 bits, ~N(0, 1)."""
    return normal_bf16(seed, (_STREAM_X << 32) | tag, (T, H), 1.0)


def router_weights(seed: int, layer: int, E: int, H: int) -> np.ndarray:
    """W_r [E, H] bf16 bits, ~N(0, 0.02)."""
    return normal_bf16(seed, (_STREAM_WR << 32) | layer, (E, H), 0.02)


def shared_gate_weights(seed: int, layer: int, H: int) -> np.ndarray:
    """w_s [H] bf16 bits, ~N(0, 0.02)."""
    return normal_bf16(seed, (_STREAM_WS << 32) | layer, (H,), 0.02)


def slot_table(seed: int, n_layers: int, E: int, permuted: bool) -> np.ndarray:
    """int32 [n_layers, E] map (layer, expert) -> slot; a permutation of 0..L*E-1."""
    n = n_layers * E
    if permuted:
        perm = _philox(seed, _STREAM_PERM << 32).permutation(n)
    else:
        perm = np.arange(n)
    return perm.astype(np.int32).reshape(n_layers, E)


def zipf_bias(seed: int, E: int, s: float = 1.1) -> np.ndarray:
    """fp32 [E] logit offsets -s*ln(1 + pi(e)) for a seeded permutation pi.

    Adding ln of a Zipf(s) pmf to the logits multiplies the softmax by that pmf
    (its normaliser cancels), so a few hot experts are shared by many tokens.
    """
    perm = _philox(seed, _STREAM_ZIPF << 32).permutation(E)
    return (-s * np.log1p(perm.astype(np.float64))).astype(np.float32)


# -------------------------------------------------------------------- workloads

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    H: int
    E: int
    k: int
    I: int
    I_shared: int
    T: int
    n_layers: int
    permuted_slots: bool
    zipf: bool
    seed: int
    description: str
    bits: int = 4          # expert weights: MLX 4-bit or 8-bit affine


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 256, 16, 4, 64, 64, 4, 1, False, False, 1001,
                 "tiny MoE layer: H=256, E=16, k=4, I=64, T=4"),
        Workload("decode35b", 2048, 256, 8, 512, 512, 1, 40, False, False, 3501,
                 "35B-A3B-shaped decode: H=2048, E=256, k=8, I=512, T=1, 40-layer stack"),
        Workload("decode80b", 2048, 512, 10, 512, 512, 1, 48, True, False, 8001,
                 "80B-A3B-shaped decode: H=2048, E=512, k=10, I=512, T=1, 48-layer stack, permuted slots"),
        Workload("zipf80b_t64", 2048, 512, 10, 512, 512, 64, 1, False, True, 8064,
                 "80B-shaped batched decode: T=64, Zipf(1.1) router offsets"),
        Workload("prefill80b", 2048, 512, 10, 512, 512, 8192, 1, False, False, 8192,
                 "80B-shaped prefill: T=8192, uniform router"),
        Workload("prefill35b", 2048, 256, 8, 512, 512, 8192, 1, False, False, 3592,
                 "35B-shaped prefill: T=8192, uniform router"),
        Workload("decode80b_int8", 2048, 512, 10, 512, 512, 1, 48, True, False, 8008,
                 "80B-A3B-shaped decode with MLX 8-bit experts: H=2048, E=512, k=10, I=512, T=1, 48 layers, "
                 "permuted slots", bits=8),
        Workload("prefill80b_int8", 2048, 512, 10, 512, 512, 8192, 1, False, False, 8208,
                 "80B-shaped prefill with MLX 8-bit experts: T=8192, uniform router", bits=8),
        Workload("limits_e1024_k16", 2048, 1024, 16, 512, 512, 64, 2, False, False, 10016,
                 "the boundary's largest router: H=2048, E=1024, k=16, I=512, T=64"),
        Workload("limits_k1", 512, 8, 1, 128, 128, 64, 2, False, False, 1008,
                 "top-1 routing: H=512, E=8, k=1, I=128, T=64"),
    ]
}


# ------------------------------------------------- Gated DeltaNet step inputs

@dataclasses.dataclass(frozen=True)
class GdnShape:
    """One Gated DeltaNet layer's recurrence shape: n_k query/key heads, n_v
    value heads (n_v / n_k value heads share a query/key head), head dims
    d_k, d_v; B sequences; T tokens per call."""
    name: str
    nk: int
    nv: int
    dk: int
    dv: int
    B: int
    T: int
    seed: int
    description: str


GDN_WORKLOADS = {
    w.name: w for w in [
        GdnShape("gdn_tiny", 2, 4, 32, 32, 3, 2, 501, "tiny Gated DeltaNet: 2 key heads, 4 value heads, d=32"),
        GdnShape("gdn80b", 16, 32, 128, 128, 128, 1, 502,
                 "Qwen3-Next-80B-shaped Gated DeltaNet decode step: 16 key heads, 32 value heads, d_k = d_v = 128, "
                 "128 sequences, one token each"),
    ]
}


def gdn_inputs(seed: int, T: int, B: int, nk: int, nv: int, dk: int, dv: int, tag: int = 0):
    """Seeded inputs of T Gated DeltaNet steps: q, k bf16 bits [T][B][nk][dk]
    and v [T][B][nv][dv] ~ N(0, 1); the gate's log decay g ~ U[-2, -0.01] and
    the write strength beta ~ U[0.05, 0.95], fp32 [T][B][nv]; a starting
    state ~ N(0, 0.1), fp32 [B][nv][dv][dk] (a state in mid-sequence)."""
    q = normal_bf16(seed, 7000 + 16 * tag + 1, (T, B, nk, dk), 1.0)
    k = normal_bf16(seed, 7000 + 16 * tag + 2, (T, B, nk, dk), 1.0)
    v = normal_bf16(seed, 7000 + 16 * tag + 3, (T, B, nv, dv), 1.0)
    rng = _philox(seed, 7000 + 16 * tag + 4)
    g = rng.uniform(-2.0, -0.01, size=(T, B, nv)).astype(np.float32)
    beta = rng.uniform(0.05, 0.95, size=(T, B, nv)).astype(np.float32)
    state = (rng.standard_normal((B, nv, dv, dk)) * 0.1).astype(np.float32)
    return q, k, v, g, beta, state
