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
// The step streams the fp32 state (d_v x d_k per head) from HBM and back, and
// the kernel is laid out for that: a CTA of 4 warps takes one tile of 32 rows
// of one (sequence, value head); a warp loads its 8 rows straight into
// registers with 16-byte streaming loads (lane l holds columns
// l * DKL .. l * DKL + DKL - 1 of each, so a row is one coalesced access),
// runs all T tokens of the call on them and writes them back with streaming
// stores. The grid is one CTA per tile; the block scheduler keeps the next
// tiles' loads in flight while earlier CTAs compute. (Persistent CTAs fed by
// bulk async copies through a shared-memory ring measured about 10% slower
// at the 80B decode shape: the copy-only form of that pipeline already
// topped out below a plain in-place elementwise kernel.) Per token and row
// the warp needs two dot products of the old row, a_i = S_i . k^ and
// b_i = S_i . q^, since
//   o_i = S'_i . q^ = alpha b_i + c_i (k^ . q^),  c_i = beta (v_i - alpha a_i),
// so the 16 sums of a warp's rows are reduced together by one transposing
// butterfly (16 shuffles in all), and the output needs no second pass over
// the updated rows. All arithmetic is fp32; o is rounded to bf16.
#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

constexpr int kGdnWarps = 4;
constexpr int kGdnRowsPerWarp = 8;
constexpr int kGdnTileRows = kGdnWarps * kGdnRowsPerWarp;   // 32

struct GdnParams {
    const uint16_t *q, *k, *v;   // [T][B][nk][dk], [T][B][nk][dk], [T][B][nv][dv] bf16
    const float *g, *beta;       // [T][B][nv]
    float *state;                // [B][nv][dv][dk]
    uint16_t *out;               // [T][B][nv][dv] bf16
    float scale;
    int T, B, nk, nv, dv;
    int group;                   // nv / nk: value heads per key head
    int tiles_per_head;
};

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// N consecutive fp32 values of global memory (N = 1, 2, 4; N * 4-byte
// aligned) as one streaming access: the state is touched once per launch.
template <int N>
__device__ __forceinline__ void ldg_f32(const float *src, float (&d)[N])
{
    if constexpr (N == 4) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(src));
        d[0] = a.x, d[1] = a.y, d[2] = a.z, d[3] = a.w;
    } else if constexpr (N == 2) {
        const float2 a = __ldcs(reinterpret_cast<const float2 *>(src));
        d[0] = a.x, d[1] = a.y;
    } else {
        d[0] = __ldcs(src);
    }
}

template <int N>
__device__ __forceinline__ void stg_f32(float *dst, const float (&d)[N])
{
    if constexpr (N == 4) __stcs(reinterpret_cast<float4 *>(dst), make_float4(d[0], d[1], d[2], d[3]));
    else if constexpr (N == 2) __stcs(reinterpret_cast<float2 *>(dst), make_float2(d[0], d[1]));
    else __stcs(dst, d[0]);
}

// N consecutive bf16 values of global memory (N * 2-byte aligned), widened.
template <int N>
__device__ __forceinline__ void ldg_bf16(const uint16_t *src, float (&d)[N])
{
    if constexpr (N == 4) {
        const uint2 a = __ldg(reinterpret_cast<const uint2 *>(src));
        d[0] = bf16lo(a.x), d[1] = bf16hi(a.x), d[2] = bf16lo(a.y), d[3] = bf16hi(a.y);
    } else if constexpr (N == 2) {
        const uint32_t a = __ldg(reinterpret_cast<const unsigned int *>(src));
        d[0] = bf16lo(a), d[1] = bf16hi(a);
    } else {
        d[0] = bf16lo(__ldg(src));
    }
}

// One step of the transposing butterfly: of 2M partial sums, the lanes whose
// bit `off` is clear keep the first M, the others the last M, each adding the
// partner lane's copy of the half it keeps.
template <int M>
__device__ __forceinline__ void fold(const float (&x)[2 * M], float (&y)[M], int off, bool upper)
{
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const float send = upper ? x[m] : x[m + M];
        const float keep = upper ? x[m + M] : x[m];
        y[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
}

// Sum over the warp of x[0..15] (per-lane partial sums): on return lane L
// holds the full sum of x[L >> 1].
__device__ __forceinline__ float reduce16(const float (&x)[16], int lane)
{
    float y8[8], y4[4], y2[2], y1[1];
    fold<8>(x, y8, 16, lane & 16);
    fold<4>(y8, y4, 8, lane & 8);
    fold<2>(y4, y2, 4, lane & 4);
    fold<1>(y2, y1, 2, lane & 2);
    return y1[0] + __shfl_xor_sync(0xffffffffu, y1[0], 1);
}

// DKL = d_k / 32 columns per lane; blockIdx.x = the tile (head-major, 32
// rows at a time).
template <int DKL>
__global__ void __launch_bounds__(kGdnWarps * 32) gdn_step_kernel(const GdnParams p)
{
    constexpr int kDk = 32 * DKL;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = int(blockIdx.x) / p.tiles_per_head;
    const int row0 = (int(blockIdx.x) - bh * p.tiles_per_head) * kGdnTileRows + warp * kGdnRowsPerWarp;
    const int b = bh / p.nv, h = bh - b * p.nv, hk = h / p.group;
    const int rows = min(kGdnRowsPerWarp, p.dv - row0);   // the warp's rows (may be <= 0 at a ragged end)
    if (rows <= 0) return;

    float *base = p.state + (size_t(bh) * p.dv + row0) * kDk + lane * DKL;
    float S[kGdnRowsPerWarp][DKL];
#pragma unroll
    for (int r = 0; r < kGdnRowsPerWarp; ++r) {
        if (r < rows) ldg_f32<DKL>(base + r * kDk, S[r]);
        else
#pragma unroll
            for (int j = 0; j < DKL; ++j) S[r][j] = 0.f;
    }

    for (int tok = 0; tok < p.T; ++tok) {
        const size_t qk = ((size_t(tok) * p.B + b) * p.nk + hk) * kDk + lane * DKL;
        float kn[DKL], qn[DKL];
        ldg_bf16<DKL>(p.k + qk, kn);
        ldg_bf16<DKL>(p.q + qk, qn);
        const size_t gi = (size_t(tok) * p.B + b) * p.nv + h;
        const float alpha = expf(__ldg(p.g + gi)), bt = __ldg(p.beta + gi);
        // lanes 2r and 2r + 1 (r < 8) hold v of the warp's row r
        const float vi = (lane < 16 && (lane >> 1) < rows) ? bf16lo(__ldg(p.v + gi * p.dv + row0 + (lane >> 1))) : 0.f;
        float sk = 0.f, sq = 0.f, skq = 0.f;
#pragma unroll
        for (int j = 0; j < DKL; ++j) {
            sk = fmaf(kn[j], kn[j], sk);
            sq = fmaf(qn[j], qn[j], sq);
            skq = fmaf(kn[j], qn[j], skq);
        }
        sk = warp_sum(sk);
        sq = warp_sum(sq);
        skq = warp_sum(skq);
        const float ik = 1.0f / sqrtf(sk + 1e-6f), iq = p.scale / sqrtf(sq + 1e-6f);
        const float kappa = skq * ik * iq;           // k^ . q^
#pragma unroll
        for (int j = 0; j < DKL; ++j) {
            kn[j] *= ik;
            qn[j] *= iq;
        }
        // x[r] = S_r . k^, x[8 + r] = S_r . q^, over the lane's columns
        float x[16];
#pragma unroll
        for (int r = 0; r < kGdnRowsPerWarp; ++r) {
            float a = 0.f, c = 0.f;
#pragma unroll
            for (int j = 0; j < DKL; ++j) {
                a = fmaf(S[r][j], kn[j], a);
                c = fmaf(S[r][j], qn[j], c);
            }
            x[r] = a;
            x[8 + r] = c;
        }
        const float sum = reduce16(x, lane);        // lanes < 16: a_{lane/2}; others: b_{lane/2 - 8}
        const float c = bt * (vi - alpha * sum);    // c_{lane/2} in lanes < 16
        const float c_hi = __shfl_xor_sync(0xffffffffu, c, 16);
        if (lane >= 16 && !(lane & 1)) {
            const int r = (lane - 16) >> 1;
            if (r < rows) p.out[gi * p.dv + row0 + r] = f32_to_bf16_bits(fmaf(alpha, sum, c_hi * kappa));
        }
#pragma unroll
        for (int r = 0; r < kGdnRowsPerWarp; ++r) {
            const float cr = __shfl_sync(0xffffffffu, c, 2 * r);
#pragma unroll
            for (int j = 0; j < DKL; ++j) S[r][j] = fmaf(alpha, S[r][j], cr * kn[j]);
        }
    }
#pragma unroll
    for (int r = 0; r < kGdnRowsPerWarp; ++r)
        if (r < rows) stg_f32<DKL>(base + r * kDk, S[r]);
}

template <int DKL>
int launch_gdn(const GdnParams &p, int n_tiles, cudaStream_t st)
{
    gdn_step_kernel<DKL><<<n_tiles, kGdnWarps * 32, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? SMOE_OK : SMOE_ECUDA;
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
    if (!(dk == 32 || dk == 64 || dk == 128) || dv % 4 || dv > 1024) return SMOE_ENOTSUP;
    if (B == 0 || T == 0) return SMOE_OK;                   // nothing to do; the buffers may be null
    if (!q || !k || !v || !g || !beta || !state || !out) return SMOE_EINVAL;
    auto a16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(g) || !a16(beta) || !a16(state) || !a16(out)) return SMOE_EINVAL;
    const int tiles_per_head = (dv + kGdnTileRows - 1) / kGdnTileRows;
    if (uint64_t(B) * nv * tiles_per_head > 0x7fffffffull) return SMOE_ENOTSUP;
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
    p.dv = dv;
    p.group = nv / nk;
    p.tiles_per_head = tiles_per_head;
    const int n_tiles = B * nv * tiles_per_head;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dk == 32) return launch_gdn<1>(p, n_tiles, st);
    if (dk == 64) return launch_gdn<2>(p, n_tiles, st);
    return launch_gdn<4>(p, n_tiles, st);
}
