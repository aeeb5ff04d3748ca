// route.cu -- router: logits, softmax, top-k (ties to the lower id),
// renormalised weights, and the sigmoid shared-expert gate.
//
// Routing counts (10 of 512 experts for the 80B model, 8 of 256 for the 35B)
// and the resident router follow the xix.ai article, paragraph on how it
// works. Since exp is increasing, the k largest probabilities are the k
// largest logits, and the renormalised weight of a chosen expert is
//   w_j = exp(z_j - z_max) / sum_{chosen i} exp(z_i - z_max),
// the full softmax denominator cancelling; the kernel computes exactly that.
//
// route_logits_kernel: CTA (row block, token block) of 8 rows x 8 tokens; the
// rows (router rows, plus the shared-gate vector as row E) and the tokens are
// bulk-copied into shared memory, one warp per row forms the fp32 dot products.
// With fused_topk the last CTA to finish (arrival ticket) then runs the top-k
// for every token, so a decode step costs one launch; otherwise topk_kernel
// runs one warp per token.
#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

constexpr int kRouteRows = 8;
constexpr int kRouteToks = 8;
constexpr int kTopkMaxPerLane = 32;   // E <= 1024

__device__ __forceinline__ void bulk_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Top-k of one token by one warp: logits row z[0..E) (+bias), gate logit zg.
__device__ void topk_warp(const float *z, const float *bias, float zg, int E, int k, int32_t *ids_out,
                          float *w_out, float *gate_out, int lane)
{
    float v[kTopkMaxPerLane];
    const int per = (E + 31) / 32;
#pragma unroll
    for (int j = 0; j < kTopkMaxPerLane; ++j) {
        const int e = lane + 32 * j;
        float val = -INFINITY;
        if (j < per && e < E) val = __ldcg(z + e) + (bias ? bias[e] : 0.f);
        v[j] = val;
    }
    uint32_t taken = 0;
    float zsel[16];
    int isel[16];
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kTopkMaxPerLane; ++j) {
            const int e = lane + 32 * j;
            if (j < per && e < E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < bi))) {
                bv = v[j];
                bi = e;
            }
        }
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        zsel[s] = bv;
        isel[s] = bi;
    }
    if (lane == 0) {
        const float zmax = zsel[0];
        float den = 0.f;
        float ex[16];
        for (int s = 0; s < k; ++s) {
            ex[s] = expf(zsel[s] - zmax);
            den += ex[s];
        }
        for (int s = 0; s < k; ++s) {
            ids_out[s] = isel[s];
            w_out[s] = ex[s] / den;
        }
        *gate_out = 1.0f / (1.0f + expf(-zg));
    }
}

__global__ void __launch_bounds__(256) route_logits_kernel(const RouteParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = p.H, E = p.E, T = p.T;
    uint16_t *wrow = reinterpret_cast<uint16_t *>(smem);                 // [8][H]
    uint16_t *xs = wrow + kRouteRows * H;                                 // [8][H]
    uint64_t *bars = reinterpret_cast<uint64_t *>(xs + kRouteToks * H);  // [2]
    __shared__ int last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = blockIdx.x * kRouteRows, tok0 = blockIdx.y * kRouteToks;
    const int nrows = min(kRouteRows, E + 1 - row0);
    const int ntok = min(kRouteToks, T - tok0);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // router rows do not depend on the previous kernel: fetch them first
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], uint32_t(nrows * H * 2));
        for (int r = 0; r < nrows; ++r) {
            const uint16_t *src = (row0 + r < E) ? p.Wr + size_t(row0 + r) * H : p.ws;
            bulk_plain(wrow + r * H, src, uint32_t(H * 2), &bars[0]);
        }
    }
    pdl_wait();
    pdl_trigger();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[1], uint32_t(ntok * H * 2));
        for (int t = 0; t < ntok; ++t)
            bulk_plain(xs + t * H, p.x + size_t(tok0 + t) * H, uint32_t(H * 2), &bars[1]);
    }
    bool ok = mbar_wait(&bars[0], 0, p.err);
    ok = mbar_wait(&bars[1], 0, p.err) && ok;

    if (warp < nrows && ok) {
        const int row = row0 + warp;
        for (int t = 0; t < ntok; ++t) {
            float acc = 0.f;
            for (int c = 8 * lane; c < H; c += 256) {
                const uint4 wv = *reinterpret_cast<const uint4 *>(wrow + warp * H + c);
                const uint4 xv = *reinterpret_cast<const uint4 *>(xs + t * H + c);
                acc = fmaf(bf16lo(wv.x), bf16lo(xv.x), acc);
                acc = fmaf(bf16hi(wv.x), bf16hi(xv.x), acc);
                acc = fmaf(bf16lo(wv.y), bf16lo(xv.y), acc);
                acc = fmaf(bf16hi(wv.y), bf16hi(xv.y), acc);
                acc = fmaf(bf16lo(wv.z), bf16lo(xv.z), acc);
                acc = fmaf(bf16hi(wv.z), bf16hi(xv.z), acc);
                acc = fmaf(bf16lo(wv.w), bf16lo(xv.w), acc);
                acc = fmaf(bf16hi(wv.w), bf16hi(xv.w), acc);
            }
            for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) p.logits[size_t(tok0 + t) * (E + 1) + row] = acc;
        }
    }
    if (!p.fused_topk) return;

    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t n = gridDim.x * gridDim.y;
        last = (atomicAdd(p.counter, 1u) == n - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int t = warp; t < T; t += 8) {
        const float *z = p.logits + size_t(t) * (E + 1);
        topk_warp(z, p.bias, __ldcg(z + E), E, p.k, p.ids + size_t(t) * p.k, p.w + size_t(t) * p.k,
                  p.gate + t, lane);
    }
    if (tid == 0) atomicExch(p.counter, 0u);
}

__global__ void __launch_bounds__(256) topk_kernel(const RouteParams p)
{
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.T) return;
    const float *z = p.logits + size_t(t) * (p.E + 1);
    topk_warp(z, p.bias, __ldcg(z + p.E), p.E, p.k, p.ids + size_t(t) * p.k, p.w + size_t(t) * p.k,
              p.gate + t, lane);
}

cudaError_t route_config()
{
    return cudaFuncSetAttribute(route_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (kRouteRows + kRouteToks) * 4096 * 2 + 16);
}

cudaError_t launch_route(const RouteParams &p0, cudaStream_t st)
{
    RouteParams p = p0;
    p.fused_topk = p.T <= kDecodeMaxT ? 1 : 0;
    const int smem = (kRouteRows + kRouteToks) * p.H * 2 + 16;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((p.E + 1 + kRouteRows - 1) / kRouteRows, (p.T + kRouteToks - 1) / kRouteToks);
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&lc, route_logits_kernel, p);
    if (e != cudaSuccess || p.fused_topk) return e;
    lc.gridDim = dim3((p.T + 7) / 8);
    lc.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&lc, topk_kernel, p);
}

}  // namespace smoe
