"""GPU: the Gated DeltaNet recurrence step (gdn_step) against the oracle's
fp64 recurrence, element by element: the tiny shape over several tokens, the
80B layer's decode step at full size (128 sequences x 32 value heads, every
state element and every output), a multi-token call, ragged value widths,
d_k = 64, one value head per key head, the empty calls and the shapes the
kernel refuses.

Tolerances, from the kernel's fp32 arithmetic (unit roundoff u = 2^-24):
each token's state update rounds a d_k-term dot product (u = S k^), the
normalisations and one fused multiply-add per element, so one step moves an
element by at most about (d_k + 16) u M, M the largest magnitude among the
state, the correction beta (v - alpha u) and 1; the update contracts (alpha
< 1, and I - beta k^ k^T has norm at most 1), so T steps add at most T times
that. The outputs are the state's rows dotted with q^ (norm = scale), so they
carry that error times sqrt(d_k) scale plus their own d_k-term dot product,
then one rounding to bf16 (half a bf16 unit of the exact value)."""
import numpy as np
import pytest
import torch

import int4_routed_expert_router_gb300 as smoe
import oracle
import synthetic
from workload import bf16_tensor, bits_of

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_routed_expert_router_gb300 import _build
    _build.build()


def run_gpu(nk, nv, q, k, v, g, beta, state, scale=0.0):
    T, B = q.shape[:2]
    dv = v.shape[3]
    S = torch.from_numpy(np.ascontiguousarray(state, np.float32)).cuda()
    out = torch.full((T, B, nv, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    smoe.gdn_step(nk, nv, bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), torch.from_numpy(g).cuda(),
                  torch.from_numpy(beta).cuda(), S, out, scale=scale)
    torch.cuda.synchronize()
    return S.cpu().numpy(), bits_of(out)


def half_bf16_unit(a):
    """Half the bf16 spacing at |a| (the largest error of one rounding)."""
    e = np.floor(np.log2(np.maximum(np.abs(a), 2.0 ** -126)))
    return 2.0 ** (e - 8)


def check(nk, nv, q, k, v, g, beta, state, scale=None):
    T, B, _, dk = q.shape
    S_gpu, out_gpu = run_gpu(nk, nv, q, k, v, g, beta, state, 0.0 if scale is None else scale)
    # the oracle reads the same fp32 gates and starting state, widened exactly
    S_ref, out_ref = oracle.gdn_step(q, k, v, g, beta, state.astype(np.float64), scale=scale)
    M = max(1.0, float(np.abs(S_ref).max()), float(np.abs(state).max()),
            float(np.abs(synthetic.bf16_bits_to_f32(v)).max()))
    tol_s = T * (dk + 16) * U32 * M
    err_s = np.abs(S_gpu.astype(np.float64) - S_ref)
    assert err_s.max() <= tol_s, (err_s.max(), tol_s)
    sc = dk ** -0.5 if scale is None else scale
    tol_o = (tol_s * np.sqrt(dk) + (dk + 16) * U32 * M * np.sqrt(dk)) * sc
    o = synthetic.bf16_bits_to_f32(out_gpu).astype(np.float64)
    assert np.isfinite(o).all()
    err_o = np.abs(o - out_ref)
    assert (err_o <= half_bf16_unit(out_ref) + tol_o).all(), float((err_o - half_bf16_unit(out_ref)).max())
    # almost every output is the correctly rounded bf16 of the exact value
    exact = synthetic.f32_to_bf16_bits(out_ref.astype(np.float32))
    assert np.mean(out_gpu == exact) > 0.98
    return S_gpu, out_gpu


def inputs(name_or_shape, T=None, B=None, tag=0):
    if isinstance(name_or_shape, str):
        s = synthetic.GDN_WORKLOADS[name_or_shape]
        nk, nv, dk, dv = s.nk, s.nv, s.dk, s.dv
        T = s.T if T is None else T
        B = s.B if B is None else B
        seed = s.seed
    else:
        nk, nv, dk, dv = name_or_shape
        seed = 509
    return (nk, nv) + synthetic.gdn_inputs(seed, T, B, nk, nv, dk, dv, tag=tag)


@pytest.mark.parametrize("T", [1, 2, 7])
def test_gdn_tiny(T):
    check(*inputs("gdn_tiny", T=T, tag=T))


def test_gdn_80b_decode_full_size():
    """The 80B layer's decode step as the benchmark runs it: every state
    element and every output of 128 sequences x 32 value heads."""
    check(*inputs("gdn80b"))


def test_gdn_80b_multi_token():
    check(*inputs("gdn80b", T=6, B=5, tag=3))


def test_gdn_tokens_one_call_equals_one_call_per_token():
    nk, nv, q, k, v, g, beta, state = inputs("gdn80b", T=4, B=3, tag=4)
    S_all, out_all = run_gpu(nk, nv, q, k, v, g, beta, state)
    S = state
    outs = []
    for t in range(4):
        S, o = run_gpu(nk, nv, q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S)
        outs.append(o)
    # the same fp32 operations in the same order: identical bits
    assert np.array_equal(S, S_all)
    assert np.array_equal(np.concatenate(outs), out_all)


@pytest.mark.parametrize("shape", [(2, 4, 128, 36), (1, 3, 64, 100), (4, 4, 32, 4), (3, 6, 128, 1024)])
def test_gdn_ragged_and_other_widths(shape):
    """Value widths that leave a partial row block (36, 100), a single row
    block of 4 rows, the widest supported rows, d_k = 64 and 32, one value head
    per key head."""
    check(*inputs(shape, T=3, B=2, tag=5))


def test_gdn_explicit_scale():
    check(*inputs("gdn_tiny", T=2, tag=6), scale=0.5)


def test_gdn_repeatable():
    a = run_gpu(*inputs("gdn80b", T=2, B=4, tag=7))
    b = run_gpu(*inputs("gdn80b", T=2, B=4, tag=7))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gdn_refusals_and_empty_calls():
    nk, nv, q, k, v, g, beta, state = inputs("gdn_tiny", T=1, B=1)
    S = torch.from_numpy(state).cuda()
    before = S.clone()
    out = torch.zeros((1, 1, nv, v.shape[3]), dtype=torch.bfloat16, device="cuda")
    qd, kd, vd = bf16_tensor(q), bf16_tensor(k), bf16_tensor(v)
    gd, bd = torch.from_numpy(g).cuda(), torch.from_numpy(beta).cuda()
    lib = smoe.lib()
    sh = smoe.GdnShape(nk, nv, q.shape[3], v.shape[3])
    args = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), gd.data_ptr(), bd.data_ptr(), 0.0)
    bad = smoe.GdnShape(3, nv, q.shape[3], v.shape[3])            # n_v not a multiple of n_k
    assert lib.gdn_step(smoe.C.byref(bad), 1, 1, *args, S.data_ptr(), out.data_ptr(), None) == smoe.EINVAL
    wide = smoe.GdnShape(nk, nv, 256, v.shape[3])                # d_k outside {32, 64, 128}
    assert lib.gdn_step(smoe.C.byref(wide), 1, 1, *args, S.data_ptr(), out.data_ptr(), None) == smoe.ENOTSUP
    # a misaligned state pointer is refused before any launch
    big = torch.zeros(state.size + 4, dtype=torch.float32, device="cuda")
    rc = lib.gdn_step(smoe.C.byref(sh), 1, 1, *args, big.data_ptr() + 4, out.data_ptr(), None)
    assert rc == smoe.EINVAL
    torch.cuda.synchronize()
    assert torch.equal(S, before) and not big.any()
    # T = 0 and B = 0 do nothing
    rc = lib.gdn_step(smoe.C.byref(sh), 1, 0, None, None, None, None, None, 0.0, None, None, None)
    assert rc == smoe.OK
