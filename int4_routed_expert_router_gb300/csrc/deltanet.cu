// deltanet.cu -- the Gated DeltaNet recurrence step: the fixed-size state
// update of the linear-attention layers that make up three quarters of the
// hybrid model (xix.ai article, paragraph on the forward pass; agentlenshq
// article, section on how expert streaming works). The pages name the layer
// but not its rule; this is the published gated delta rule, with
// L2-normalised queries and keys. Per sequence b, value head h (query/key
// head h / (n_v / n_k)) and token t, with state S (d_v rows x d_k columns):
//   k^ = k / sqrt(sum k^2 + 1e-6),  q^ = scale q / sqrt(sum q^2 + 1e-6)
//   u = S k^,  S <- exp(g) S + beta (v - exp(g) u) k^T,  o = S q^.
//
// The step is a stream over the state (d_v x d_k fp32 per head), so the
// kernel is laid out for HBM: a CTA of 8 warps takes 32 rows of one
// (sequence, value head); a warp keeps 4 rows in registers (lane l holds
// columns l * DKL .. l * DKL + DKL - 1 of each, so a row is one coalesced
// 4 * d_k-byte access) for all T tokens of the call, so the state is read
// and written once per call. Each token: the warp normalises k and q (warp
// sums), reads back u for its rows (warp sums), updates them, and forms o
// (warp sums); lanes 0-3 write the rows of o in bf16. All arithmetic is fp32.
#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

constexpr int kGdnWarps = 8;
constexpr int kGdnRowsPerWarp = 4;
constexpr int kGdnRowsPerCta = kGdnWarps * kGdnRowsPerWarp;

struct GdnParams {
    const uint16_t *q, *k, *v;   // [T][B][nk][dk], [T][B][nk][dk], [T][B][nv][dv] bf16
    const float *g, *beta;       // [T][B][nv]
    float *state;                // [B][nv][dv][dk]
    uint16_t *out;               // [T][B][nv][dv] bf16
    float scale;
    int T, B, nk, nv, dk, dv, row_blocks;
};

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// N consecutive fp32 values as one access (N = 1, 2, 4; the address is N * 4-byte aligned).
template <int N>
__device__ __forceinline__ void load_f32(const float *src, float (&d)[N])
{
    if constexpr (N == 4) {
        const float4 a = *reinterpret_cast<const float4 *>(src);
        d[0] = a.x, d[1] = a.y, d[2] = a.z, d[3] = a.w;
    } else if constexpr (N == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(src);
        d[0] = a.x, d[1] = a.y;
    } else {
        d[0] = src[0];
    }
}

template <int N>
__device__ __forceinline__ void store_f32(float *dst, const float (&d)[N])
{
    if constexpr (N == 4) *reinterpret_cast<float4 *>(dst) = make_float4(d[0], d[1], d[2], d[3]);
    else if constexpr (N == 2) *reinterpret_cast<float2 *>(dst) = make_float2(d[0], d[1]);
    else dst[0] = d[0];
}

// N consecutive bf16 values (N = 1, 2, 4; the address is N * 2-byte aligned), widened to fp32.
template <int N>
__device__ __forceinline__ void load_bf16(const uint16_t *src, float (&d)[N])
{
    if constexpr (N == 4) {
        const uint2 a = *reinterpret_cast<const uint2 *>(src);
        d[0] = bf16lo(a.x), d[1] = bf16hi(a.x), d[2] = bf16lo(a.y), d[3] = bf16hi(a.y);
    } else if constexpr (N == 2) {
        const uint32_t a = *reinterpret_cast<const uint32_t *>(src);
        d[0] = bf16lo(a), d[1] = bf16hi(a);
    } else {
        d[0] = bf16_to_f32(src[0]);
    }
}

// DKL = d_k / 32 columns per lane.
template <int DKL>
__global__ void __launch_bounds__(kGdnWarps * 32) gdn_step_kernel(const GdnParams p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x % p.row_blocks;
    const int bh = blockIdx.x / p.row_blocks;               // b * nv + h
    const int b = bh / p.nv, h = bh % p.nv;
    const int hk = h / (p.nv / p.nk);
    const int dk = p.dk, dv = p.dv;
    const int r0 = rb * kGdnRowsPerCta + warp * kGdnRowsPerWarp;

    float S[kGdnRowsPerWarp][DKL];
    float *base = p.state + (size_t(bh) * dv) * dk;
#pragma unroll
    for (int i = 0; i < kGdnRowsPerWarp; ++i) {
        if (r0 + i < dv) load_f32<DKL>(base + size_t(r0 + i) * dk + lane * DKL, S[i]);
        else
#pragma unroll
            for (int j = 0; j < DKL; ++j) S[i][j] = 0.f;
    }

    for (int t = 0; t < p.T; ++t) {
        const size_t qk = ((size_t(t) * p.B + b) * p.nk + hk) * dk + lane * DKL;
        float kn[DKL], qn[DKL];
        load_bf16<DKL>(p.k + qk, kn);
        load_bf16<DKL>(p.q + qk, qn);
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int j = 0; j < DKL; ++j) {
            sk = fmaf(kn[j], kn[j], sk);
            sq = fmaf(qn[j], qn[j], sq);
        }
        sk = warp_sum(sk);
        sq = warp_sum(sq);
        const float ik = 1.0f / sqrtf(sk + 1e-6f), iq = p.scale / sqrtf(sq + 1e-6f);
#pragma unroll
        for (int j = 0; j < DKL; ++j) {
            kn[j] *= ik;
            qn[j] *= iq;
        }
        const size_t gi = (size_t(t) * p.B + b) * p.nv + h;
        const float alpha = expf(p.g[gi]), bt = p.beta[gi];
        // u_i = S_i . k^ for the warp's rows (four independent warp sums)
        float u[kGdnRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kGdnRowsPerWarp; ++i) {
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < DKL; ++j) a = fmaf(S[i][j], kn[j], a);
            u[i] = a;
        }
#pragma unroll
        for (int i = 0; i < kGdnRowsPerWarp; ++i) u[i] = warp_sum(u[i]);
        float o[kGdnRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kGdnRowsPerWarp; ++i) {
            const float vi = r0 + i < dv ? bf16_to_f32(p.v[gi * dv + r0 + i]) : 0.f;
            const float c = bt * (vi - alpha * u[i]);
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < DKL; ++j) {
                S[i][j] = fmaf(alpha, S[i][j], c * kn[j]);
                a = fmaf(S[i][j], qn[j], a);
            }
            o[i] = a;
        }
#pragma unroll
        for (int i = 0; i < kGdnRowsPerWarp; ++i) o[i] = warp_sum(o[i]);
        if (lane < kGdnRowsPerWarp && r0 + lane < dv) {
            float oi = o[0];
#pragma unroll
            for (int i = 1; i < kGdnRowsPerWarp; ++i) oi = lane == i ? o[i] : oi;
            p.out[gi * dv + r0 + lane] = f32_to_bf16_bits(oi);
        }
    }
#pragma unroll
    for (int i = 0; i < kGdnRowsPerWarp; ++i)
        if (r0 + i < dv) store_f32<DKL>(base + size_t(r0 + i) * dk + lane * DKL, S[i]);
}

}  // namespace smoe

using namespace smoe;

extern "C" int gdn_step(const smoe_gdn_shape *shape, int32_t B, int32_t T, const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, const float *g, const float *beta, float scale, float *state,
                        uint16_t *out, void *stream)
{
    if (!shape || B < 0 || T < 0) return SMOE_EINVAL;
    const int nk = shape->nk, nv = shape->nv, dk = shape->dk, dv = shape->dv;
    if (nk <= 0 || nv <= 0 || dk <= 0 || dv <= 0 || nv % nk) return SMOE_EINVAL;
    if (!(dk == 32 || dk == 64 || dk == 128) || dv % kGdnRowsPerWarp || dv > 1024) return SMOE_ENOTSUP;
    if (B == 0 || T == 0) return SMOE_OK;                   // nothing to do; the buffers may be null
    if (!q || !k || !v || !g || !beta || !state || !out) return SMOE_EINVAL;
    auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(g) || !a16(beta) || !a16(state) || !a16(out)) return SMOE_EINVAL;
    if (uint64_t(B) * nv * ((dv + kGdnRowsPerCta - 1) / kGdnRowsPerCta) > 0x7fffffffull) return SMOE_ENOTSUP;
    GdnParams p = {};
    p.q = q;
    p.k = k;
    p.v = v;
    p.g = g;
    p.beta = beta;
    p.state = state;
    p.out = out;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf(float(dk));
    p.T = T;
    p.B = B;
    p.nk = nk;
    p.nv = nv;
    p.dk = dk;
    p.dv = dv;
    p.row_blocks = (dv + kGdnRowsPerCta - 1) / kGdnRowsPerCta;
    const dim3 grid(unsigned(B * nv * p.row_blocks)), block(kGdnWarps * 32);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dk == 32) gdn_step_kernel<1><<<grid, block, 0, st>>>(p);
    else if (dk == 64) gdn_step_kernel<2><<<grid, block, 0, st>>>(p);
    else gdn_step_kernel<4><<<grid, block, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? SMOE_OK : SMOE_ECUDA;
}
