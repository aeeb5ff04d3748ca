// debug.cu -- a plain CUDA path for the MoE layer, for checking the fast
// kernels on the device itself: one CTA per token, every weight decoded one at
// a time from the blob's atom layout (s * q + b in fp32), fp32 dot products, the
// routed experts in route order and then the shared expert, one bf16 rounding.
// No tensor cores, no staging, no split work. The layer it computes is the
// sparse MoE layer of the pages (xix.ai article, paragraph on how it works;
// agentlenshq article, how expert streaming works); the pages ask for a
// scalar path to hold the fast ones to (the paper-digest page, its notes on
// correctness against an exact reference).
#include <cuda_fp16.h>

#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

constexpr int kDbgThreads = 256;

// Weight (row, col) of one 16-row x 64-column atom: logical row lr (g = lr % 8,
// upper = lr / 8), column cc. Lane 4 g + t holds the words (g, cols 16 t ..
// 16 t + 7), (g, 16 t + 8 ..), (g + 8, 16 t ..), (g + 8, 16 t + 8 ..); in a word
// for columns c0 .. c0 + 7, column c0 + 2 m sits in bits 4 m .. 4 m + 3 and
// column c0 + 2 m + 1 in bits 16 + 4 m ..; fp16 (s, b) of row g, then of row
// g + 8, at byte 512 + 8 g. An 8-bit atom holds two such 512-byte nibble
// planes (low nibbles, then high nibbles: q = low + 16 high) and its (s, b)
// at byte 1024 + 8 g.
__device__ unsigned atom_nibble(const uint8_t *plane, int lr, int cc)
{
    const int g = lr & 7, upper = lr >> 3, t = cc >> 4, half = (cc >> 3) & 1, cl = cc & 7;
    const uint32_t word = *reinterpret_cast<const uint32_t *>(plane + 16 * (4 * g + t) + 4 * (2 * upper + half));
    const int shift = (cl & 1) ? 16 + 4 * (cl >> 1) : 4 * (cl >> 1);
    return (word >> shift) & 15u;
}

__device__ float atom_weight(const uint8_t *atom, int lr, int cc, bool eight)
{
    const int g = lr & 7, upper = lr >> 3;
    const unsigned q = eight ? atom_nibble(atom, lr, cc) + 16u * atom_nibble(atom + kAtomQBytes, lr, cc)
                             : atom_nibble(atom, lr, cc);
    const uint16_t *sb = reinterpret_cast<const uint16_t *>(atom + (eight ? 2 : 1) * kAtomQBytes + 8 * g + 4 * upper);
    return __half2float(__ushort_as_half(sb[0])) * float(q) + __half2float(__ushort_as_half(sb[1]));
}

struct DebugParams {
    const uint16_t *x;
    const int32_t *ids;
    const float *w;
    const float *gate;
    const uint8_t *pool;
    const uint8_t *shared_blob;
    const int32_t *table_row;
    uint64_t stride, down_off;
    int64_t n_slots;
    int atom_bytes;                 // 576 (4-bit atoms) or 1088 (8-bit: two nibble planes)
    const uint16_t *residual;
    uint16_t *out;
    int32_t *err;
    int T, H, E, k, I;
};

__global__ void __launch_bounds__(kDbgThreads) debug_forward_kernel(const DebugParams p)
{
    extern __shared__ float dsm[];
    float *xs = dsm;                 // [H] the token
    float *hs = dsm + p.H;           // [I] h of the current expert
    const int t = blockIdx.x, tid = threadIdx.x;
    const int H = p.H, I = p.I, ngH = H / kGroup, ngI = I / kGroup;
    const size_t ab = size_t(p.atom_bytes);
    const bool eight = p.atom_bytes != kAtomBytes;
    for (int c = tid; c < H; c += kDbgThreads) xs[c] = __uint_as_float(uint32_t(p.x[size_t(t) * H + c]) << 16);
    constexpr int kRows = 2048 / kDbgThreads;                     // outputs per thread (H <= 2048)
    float acc[kRows];
#pragma unroll
    for (int q = 0; q < kRows; ++q) acc[q] = 0.f;
    for (int j = 0; j <= p.k; ++j) {                              // route order, then the shared expert
        const uint8_t *blob = p.shared_blob;
        float wt = p.gate[t];
        if (j < p.k) {
            const int e = p.ids[size_t(t) * p.k + j];
            const int64_t slot = (e >= 0 && e < p.E) ? int64_t(p.table_row[e]) : -1;
            wt = p.w[size_t(t) * p.k + j];
            if (e < 0 || e >= p.E) {
                if (tid == 0) set_error(p.err, SMOE_DEV_BAD_EXPERT);
                continue;
            }
            if (slot < 0 || slot >= p.n_slots) {
                if (tid == 0) set_error(p.err, SMOE_DEV_BAD_SLOT);
                continue;
            }
            blob = p.pool + uint64_t(slot) * p.stride;
        }
        __syncthreads();                                          // xs ready; hs free
        for (int i = tid; i < I; i += kDbgThreads) {              // gate row i and up row i
            const uint8_t *row_atoms = blob + size_t(i / 8) * ngH * ab;
            float gs = 0.f, us = 0.f;
            for (int c = 0; c < H; ++c) {
                const uint8_t *atom = row_atoms + size_t(c / kGroup) * ab;
                gs = fmaf(atom_weight(atom, i % 8, c % kGroup, eight), xs[c], gs);
                us = fmaf(atom_weight(atom, 8 + i % 8, c % kGroup, eight), xs[c], us);
            }
            hs[i] = gs / (1.f + expf(-gs)) * us;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kRows; ++q) {                         // down rows
            const int r = tid + q * kDbgThreads;
            if (r >= H) break;
            const uint8_t *row_atoms = blob + p.down_off + size_t(r / 16) * ngI * ab;
            float y = 0.f;
            for (int i = 0; i < I; ++i)
                y = fmaf(atom_weight(row_atoms + size_t(i / kGroup) * ab, r % 16, i % kGroup, eight), hs[i], y);
            acc[q] = fmaf(wt, y, acc[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < kRows; ++q) {
        const int r = tid + q * kDbgThreads;
        if (r >= H) break;
        float v = acc[q];
        if (p.residual) v += __uint_as_float(uint32_t(p.residual[size_t(t) * H + r]) << 16);
        p.out[size_t(t) * H + r] = f32_to_bf16_bits(v);
    }
}

}  // namespace smoe

extern "C" int moe_forward_debug(const smoe_ctx *ctx, int32_t layer, const uint16_t *x, int32_t T, const int32_t *ids,
                                 const float *w, const float *gate, const void *pool, uint64_t pool_bytes,
                                 const void *shared_blob, const uint16_t *residual, uint16_t *out, int32_t *err,
                                 void *stream)
{
    using namespace smoe;
    if (!ctx || T < 0 || T > SMOE_MAX_TOKENS) return SMOE_EINVAL;
    if (layer < 0 || layer >= ctx->n_layers) return SMOE_EINVAL;
    if (T == 0) return SMOE_OK;                      // nothing to do; the buffers may be null
    if (!x || !ids || !w || !gate || !pool || !shared_blob || !out || !err) return SMOE_EINVAL;
    auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    if (!a16(x) || !a16(pool) || !a16(shared_blob) || !a16(out) || (residual && !a16(residual))) return SMOE_EINVAL;
    if (pool_bytes < uint64_t(ctx->n_slots) * ctx->layout.blob) return SMOE_ENOMEM;
    DebugParams p = {};
    p.x = x;
    p.ids = ids;
    p.w = w;
    p.gate = gate;
    p.pool = static_cast<const uint8_t *>(pool);
    p.shared_blob = static_cast<const uint8_t *>(shared_blob);
    p.table_row = ctx->table_dev + size_t(layer) * ctx->shape.E;
    p.stride = ctx->layout.blob;
    p.down_off = ctx->layout.down_off;
    p.n_slots = ctx->n_slots;
    p.atom_bytes = ctx->shape.bits == 8 ? 2 * kAtomQBytes + 64 : kAtomBytes;
    p.residual = residual;
    p.out = out;
    p.err = err;
    p.T = T;
    p.H = ctx->shape.H;
    p.E = ctx->shape.E;
    p.k = ctx->shape.k;
    p.I = ctx->shape.I;
    const size_t smem = size_t(p.H + p.I) * 4;
    debug_forward_kernel<<<T, kDbgThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SMOE_OK : SMOE_ECUDA;
}
