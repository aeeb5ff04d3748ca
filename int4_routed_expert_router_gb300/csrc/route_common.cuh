// route_common.cuh -- routing arithmetic shared by the routing kernel
// (route.cu) and the multi-layer decode kernel (decode_stack.cu), so that both
// produce the same logits, ids and weights bit for bit.
// Since exp is increasing, the k largest probabilities are the k largest
// logits, and the renormalised weight of a chosen expert is
//   w_j = exp(z_j - z_max) / sum_{chosen i} exp(z_i - z_max),
// the full softmax denominator cancelling (xix.ai article, paragraph on how it
// works: top-k routing over the experts).
#pragma once

#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

// One router row (bf16 [H]) dotted with one token (bf16 [H]) by a warp: lane l
// takes columns 8 l .. 8 l + 7 of every 256; within them column 8 l + j goes
// to partial sum j % 4 (four independent fp32 chains of fused multiply-adds,
// in column order), the four are added as (s0 + s1) + (s2 + s3), then a
// butterfly sum over the lanes. Every lane returns the total.
__device__ __forceinline__ float router_dot(const uint16_t *row, const uint16_t *x, int H, int lane)
{
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int c = 8 * lane; c < H; c += 256) {
        const uint4 wv = *reinterpret_cast<const uint4 *>(row + c);
        const uint4 xv = *reinterpret_cast<const uint4 *>(x + c);
        s0 = fmaf(bf16lo(wv.x), bf16lo(xv.x), s0);
        s1 = fmaf(bf16hi(wv.x), bf16hi(xv.x), s1);
        s2 = fmaf(bf16lo(wv.y), bf16lo(xv.y), s2);
        s3 = fmaf(bf16hi(wv.y), bf16hi(xv.y), s3);
        s0 = fmaf(bf16lo(wv.z), bf16lo(xv.z), s0);
        s1 = fmaf(bf16hi(wv.z), bf16hi(xv.z), s1);
        s2 = fmaf(bf16lo(wv.w), bf16lo(xv.w), s2);
        s3 = fmaf(bf16hi(wv.w), bf16hi(xv.w), s3);
    }
    float acc = (s0 + s1) + (s2 + s3);
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// One router row dotted with ntok <= NT tokens (rows t of xs, H apart): each
// result in router_dot's order (per lane four interleaved partial sums over
// the lane's 8-element chunks, then (s0 + s1) + (s2 + s3), then the
// butterfly), so out[t] equals router_dot(row, xs + t H) bit for bit; each
// chunk of the row is loaded once for all tokens, and the tokens' chains are
// independent, so their latencies overlap.
template <int NT>
__device__ __forceinline__ void router_dot_multi(const uint16_t *row, const uint16_t *xs, int H, int ntok, int lane,
                                                 float (&out)[NT])
{
    float s[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
    for (int c = 8 * lane; c < H; c += 256) {
        const uint4 wv = *reinterpret_cast<const uint4 *>(row + c);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < ntok) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xs + size_t(t) * H + c);
                s[t][0] = fmaf(bf16lo(wv.x), bf16lo(xv.x), s[t][0]);
                s[t][1] = fmaf(bf16hi(wv.x), bf16hi(xv.x), s[t][1]);
                s[t][2] = fmaf(bf16lo(wv.y), bf16lo(xv.y), s[t][2]);
                s[t][3] = fmaf(bf16hi(wv.y), bf16hi(xv.y), s[t][3]);
                s[t][0] = fmaf(bf16lo(wv.z), bf16lo(xv.z), s[t][0]);
                s[t][1] = fmaf(bf16hi(wv.z), bf16hi(xv.z), s[t][1]);
                s[t][2] = fmaf(bf16lo(wv.w), bf16lo(xv.w), s[t][2]);
                s[t][3] = fmaf(bf16hi(wv.w), bf16hi(xv.w), s[t][3]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        float acc = (s[t][0] + s[t][1]) + (s[t][2] + s[t][3]);
        for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        out[t] = acc;
    }
}

// Order-preserving map float -> uint32 (larger float, larger key); key 0 is
// reserved for "taken / empty" (no finite or infinite float maps to it).
__device__ __forceinline__ uint32_t fkey(float f)
{
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float fkey_inv(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp picks the k largest keys among its lanes' PER values, in
// descending order, ties to the lower id. Each round: warp max of the lanes'
// current bests, then the lowest id holding that key; the winner removes it.
template <int PER>
__device__ inline void warp_topk(uint32_t (&key)[PER], int32_t (&id)[PER], int k, uint32_t *okey, int32_t *oid,
                          int lane)
{
    for (int s = 0; s < k; ++s) {
        uint32_t bk = 0;
        int32_t bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (key[j] > bk || (key[j] == bk && key[j] != 0u && id[j] < bi)) {
                bk = key[j];
                bi = id[j];
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const int32_t mi = int32_t(__reduce_min_sync(0xffffffffu, uint32_t(bk == mk ? bi : 0x7fffffff)));
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (id[j] == mi && key[j] == mk) key[j] = 0u;
        if (lane == 0) {
            okey[s] = mk;
            oid[s] = mk ? mi : -1;
        }
    }
}

// warp_topk with a threshold pass first: the k-th largest of the 32 lanes'
// maxima bounds the k-th largest key from below (k distinct keys reach it), so
// only keys at or above it can be chosen, ties included. When at most 64 keys
// qualify (the usual case) they are compacted into ck/ci (64 entries, this
// warp's own) and selected from there; otherwise warp_topk runs on all keys.
// The result equals warp_topk's. Needs k <= 32.
template <int PER>
__device__ inline void warp_topk_thresh(uint32_t (&key)[PER], int32_t (&id)[PER], int k, uint32_t *okey,
                                        int32_t *oid, int lane, uint32_t *ck, int32_t *ci)
{
    uint32_t cur = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) cur = max(cur, key[j]);
    uint32_t t0 = 0;
    for (int s = 0; s < k; ++s) {                 // the k-th largest lane maximum
        t0 = __reduce_max_sync(0xffffffffu, cur);
        const uint32_t who = __ballot_sync(0xffffffffu, cur == t0);
        if (lane == __ffs(who) - 1) cur = 0;
    }
    int n = 0;
    if (t0 != 0u) {
        const uint32_t below = (1u << lane) - 1u;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const bool c = key[j] >= t0;
            const uint32_t b = __ballot_sync(0xffffffffu, c);
            const int pos = n + __popc(b & below);
            if (c && pos < 64) {
                ck[pos] = key[j];
                ci[pos] = id[j];
            }
            n += __popc(b);
        }
    }
    if (t0 == 0u || n > 64) {                    // empty slots among the maxima, or too many candidates
        warp_topk<PER>(key, id, k, okey, oid, lane);
        return;
    }
    __syncwarp();
    uint32_t k2[2];
    int32_t i2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c = lane + 32 * u;
        k2[u] = c < n ? ck[c] : 0u;
        i2[u] = c < n ? ci[c] : 0x7fffffff;
    }
    __syncwarp();
    warp_topk<2>(k2, i2, k, okey, oid, lane);
}

// Level 1 for one token slice: values z[e] (+bias) for e in [e0, e1); z may be
// global (read through L2) or a shared-memory copy.
template <int PER>
__device__ inline void slice_topk(const float *z, const float *bias, int e0, int e1, int k, uint32_t *okey, int32_t *oid,
                           int lane)
{
    uint32_t key[PER];
    int32_t id[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = e0 + lane + 32 * j;
        key[j] = 0u;
        id[j] = 0x7fffffff;
        if (e < e1) {
            key[j] = fkey(z[e] + (bias ? bias[e] : 0.f));
            id[j] = e;
        }
    }
    warp_topk<PER>(key, id, k, okey, oid, lane);
}

// slice_topk over all E values of one token with the threshold pass.
template <int PER>
__device__ inline void token_topk(const float *z, const float *bias, int E, int k, uint32_t *okey, int32_t *oid,
                                  int lane, uint32_t *ck, int32_t *ci)
{
    uint32_t key[PER];
    int32_t id[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        key[j] = 0u;
        id[j] = 0x7fffffff;
        if (e < E) {
            key[j] = fkey(z[e] + (bias ? bias[e] : 0.f));
            id[j] = e;
        }
    }
    warp_topk_thresh<PER>(key, id, k, okey, oid, lane, ck, ci);
}

__device__ inline void token_topk_any(int per, const float *z, const float *bias, int E, int k, uint32_t *ok,
                                      int32_t *oi, int lane, uint32_t *ck, int32_t *ci)
{
    if (per <= 1) token_topk<1>(z, bias, E, k, ok, oi, lane, ck, ci);
    else if (per <= 2) token_topk<2>(z, bias, E, k, ok, oi, lane, ck, ci);
    else if (per <= 4) token_topk<4>(z, bias, E, k, ok, oi, lane, ck, ci);
    else if (per <= 8) token_topk<8>(z, bias, E, k, ok, oi, lane, ck, ci);
    else if (per <= 16) token_topk<16>(z, bias, E, k, ok, oi, lane, ck, ci);
    else token_topk<32>(z, bias, E, k, ok, oi, lane, ck, ci);
}

__device__ inline void slice_topk_any(int per, const float *z, const float *bias, int e0, int e1, int k, uint32_t *ok,
                               int32_t *oi, int lane)
{
    if (per <= 1) slice_topk<1>(z, bias, e0, e1, k, ok, oi, lane);
    else if (per <= 2) slice_topk<2>(z, bias, e0, e1, k, ok, oi, lane);
    else if (per <= 4) slice_topk<4>(z, bias, e0, e1, k, ok, oi, lane);
    else if (per <= 8) slice_topk<8>(z, bias, e0, e1, k, ok, oi, lane);
    else if (per <= 16) slice_topk<16>(z, bias, e0, e1, k, ok, oi, lane);
    else slice_topk<32>(z, bias, e0, e1, k, ok, oi, lane);
}

// Level 2 for one token: the k best of the nw * k candidates that nw level-1
// warps left in ckey/cid (16 entries per warp, nw * k <= 128), by one warp,
// into fk/fi in descending order.
__device__ inline void topk_merge(const uint32_t *ckey, const int32_t *cid, int nw, int k, uint32_t *fk, int32_t *fi,
                                  int lane)
{
    uint32_t key[4];
    int32_t id[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = lane + 32 * j;
        const int w = c / k, r = c % k;
        const bool ok = c < nw * k;
        key[j] = ok ? ckey[w * 16 + r] : 0u;
        id[j] = ok && key[j] ? cid[w * 16 + r] : 0x7fffffff;
    }
    warp_topk<4>(key, id, k, fk, fi, lane);
}

// Renormalised weight of choice `lane` (lane < k) from the k chosen keys in
// descending order: each lane forms exp(z_lane - z_max), then every lane sums
// the k terms in choice order (gathered by shuffles), so all lanes agree bit
// for bit. Called by a whole warp.
__device__ __forceinline__ float choice_weight(const uint32_t *fk, int k, int lane)
{
    const float zmax = fkey_inv(fk[0]);
    const float ex = lane < k ? expf(fkey_inv(fk[lane]) - zmax) : 0.f;
    float den = 0.f;
    for (int s = 0; s < k; ++s) den += __shfl_sync(0xffffffffu, ex, s);
    return lane < k ? ex / den : 0.f;
}

__device__ __forceinline__ float shared_gate(float zs) { return 1.0f / (1.0f + expf(-zs)); }

}  // namespace smoe
