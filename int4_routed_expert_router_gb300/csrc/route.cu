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
// With fused_topk (T <= 8) the last CTA to finish (arrival ticket) then runs
// the top-k for every token with all its warps (two levels of warp
// max-reductions over order-preserving integer keys), so a decode step costs
// one launch; up to kRouteGemvMaxT tokens topk_cta_kernel then ranks each
// token with a CTA the same way; above it the logits come from the
// tensor-core kernel and topk_kernel runs one warp per token.
#include "route_common.cuh"

namespace smoe {

constexpr int kRouteRows = 8;
constexpr int kRouteToks = 8;

// Bytes of the route kernel's main shared-memory region: the staged rows and
// tokens, reused for the T x (E + 1) logits of the top-k.
__host__ __device__ inline int route_region_bytes(int H, int E, int T)
{
    const int a = (kRouteRows + kRouteToks) * H * 2, b = T * (E + 1) * 4;
    return ((a > b ? a : b) + 15) & ~15;
}

__device__ __forceinline__ void bulk_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Final outputs of one token from its k chosen keys (descending), one lane
// per choice (k <= 16); zs: the token's shared-gate logit.
__device__ void write_choice(const RouteParams &p, int t, const uint32_t *fk, const int32_t *fi, float zs, int lane)
{
    const float wl = choice_weight(fk, p.k, lane);
    if (lane < p.k) {
        p.ids[size_t(t) * p.k + lane] = fi[lane];
        p.w[size_t(t) * p.k + lane] = wl;
    }
    if (lane == 0) p.gate[t] = shared_gate(zs);
}

// Top-k of tokens tok0 .. tok0 + T - 1 (T <= 8) by the 8 warps of a CTA. The
// T x (E + 1) logits are first copied to shared memory by all threads (one
// round trip to L2). Each token gets 8/T' warps (T' = T rounded up to a power
// of two); each of them takes a slice of the experts (level 1), then one warp
// merges the slices' candidates (level 2). ckey/cid: 2 * 8 * 16 entries; zsm:
// T * (E + 1) floats.
__device__ void block_topk(const RouteParams &p, int tok0, int T, uint32_t *ckey, int32_t *cid, float *zsm)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E, k = p.k;
    const float *lg = p.logits + size_t(tok0) * (E + 1);
    for (int i = threadIdx.x; i < T * (E + 1); i += blockDim.x) zsm[i] = __ldcg(lg + i);
    __syncthreads();
    int tp = 1;
    while (tp < T) tp <<= 1;
    const int wpt = 8 / tp;                     // warps per token
    const int t = warp / wpt, sl = warp % wpt;
    if (t < T) {
        const int span = (E + wpt - 1) / wpt;
        const int e0 = sl * span, e1 = min(E, e0 + span);
        slice_topk_any((span + 31) / 32, zsm + t * (E + 1), p.bias, e0, e1, k, ckey + warp * 16, cid + warp * 16,
                       lane);
    }
    __syncthreads();
    if (t < T && sl == 0) {
        uint32_t *fk = ckey + 8 * 16 + warp * 16;
        int32_t *fi = cid + 8 * 16 + warp * 16;
        topk_merge(ckey + warp * 16, cid + warp * 16, wpt, k, fk, fi, lane);
        __syncwarp();
        write_choice(p, tok0 + t, fk, fi, zsm[t * (E + 1) + E], lane);
    }
}

__global__ void __launch_bounds__(256) route_logits_kernel(const RouteParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = p.H, E = p.E, T = p.T;
    // [router rows 8 x H | tokens 8 x H], later the logits for the top-k; barriers last
    uint16_t *wrow = reinterpret_cast<uint16_t *>(smem);                 // [8][H]
    uint16_t *xs = wrow + kRouteRows * H;                                 // [8][H]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + route_region_bytes(H, E, p.fused_topk ? T : 0));   // [2]
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
        float acc[kRouteToks];
        router_dot_multi<kRouteToks>(wrow + warp * H, xs, H, ntok, lane, acc);
        if (lane < ntok) {
            float z = acc[0];
#pragma unroll
            for (int t = 1; t < kRouteToks; ++t) z = lane == t ? acc[t] : z;
            p.logits[size_t(tok0 + lane) * (E + 1) + row] = z;
        }
    }
    if (!p.fused_topk) return;

    __syncthreads();
    if (tid == 0) {
        const uint32_t n = gridDim.x * gridDim.y;
        last = (ticket_add(p.counter, 1u) == n - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!last) return;
    __shared__ uint32_t ckey[2 * 8 * 16];
    __shared__ int32_t cid[2 * 8 * 16];
    block_topk(p, 0, T, ckey, cid, reinterpret_cast<float *>(wrow));   // the router rows are no longer needed
    if (tid == 0) atomicExch(p.counter, 0u);
}

// One warp per token (large T): a single level over all E experts (the
// threshold pass of warp_topk_thresh first), and the token's shared-gate logit
// w_s . x_t by router_dot, as the small-T path computes it.
__global__ void __launch_bounds__(256) topk_kernel(const RouteParams p)
{
    __shared__ uint32_t ckey[8 * 16];
    __shared__ int32_t cid[8 * 16];
    __shared__ uint32_t cand_k[8 * 64];
    __shared__ int32_t cand_i[8 * 64];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.T) return;
    token_topk_any((p.E + 31) / 32, p.logits + size_t(t) * (p.E + 1), p.bias, p.E, p.k, ckey + warp * 16,
                   cid + warp * 16, lane, cand_k + warp * 64, cand_i + warp * 64);
    const float zs = p.gate_in_logits ? __ldcg(p.logits + size_t(t) * (p.E + 1) + p.E)
                                      : router_dot(p.ws, p.x + size_t(t) * p.H, p.H, lane);
    __syncwarp();
    write_choice(p, t, ckey + warp * 16, cid + warp * 16, zs, lane);
}

// One token per CTA (8 < T <= kRouteGemvMaxT, after the GEMV kernel): the
// token's 8 warps each rank a slice of the experts and warp 0 merges them, as
// the fused top-k does for T <= 8, so a token's top-k takes one warp's share
// of E / 8 experts instead of all E.
__global__ void __launch_bounds__(256) topk_cta_kernel(const RouteParams p)
{
    __shared__ uint32_t ckey[2 * 8 * 16];
    __shared__ int32_t cid[2 * 8 * 16];
    __shared__ float zsm[1024 + 1];
    pdl_wait();
    pdl_trigger();
    block_topk(p, int(blockIdx.x), 1, ckey, cid, zsm);
}

cudaError_t route_config()
{
    return cudaFuncSetAttribute(route_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                route_region_bytes(2048, 1024, kDecodeMaxT) + 16);
}

cudaError_t launch_route(const RouteParams &p0, cudaStream_t st)
{
    RouteParams p = p0;
    if (p.T > kRouteGemvMaxT) {    // logits on tensor cores, then one warp per token
        cudaError_t e = launch_router_gemm(p, st);
        if (e != cudaSuccess) return e;
        return launch_pdl(topk_kernel, dim3((p.T + 7) / 8), dim3(256), 0, st, p);
    }
    // small T: the GEMV kernel over (row block, token block) CTAs; above kDecodeMaxT
    // it stops at the logits (row E: the shared-gate logit) and one warp per token
    // takes the top-k
    p.fused_topk = p.T <= kDecodeMaxT ? 1 : 0;
    p.gate_in_logits = 1;
    const int smem = route_region_bytes(p.H, p.E, p.fused_topk ? p.T : 0) + 16;
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
    return launch_pdl(topk_cta_kernel, dim3(p.T), dim3(256), 0, st, p);
}

}  // namespace smoe
