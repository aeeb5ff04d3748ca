// decode_common.cuh -- helpers of the small-T expert kernel (decode.cu): the
// down-projection rows, the per-group scale terms, and the routing bookkeeping.
#pragma once

#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

__host__ __device__ inline int align128(int v) { return (v + 127) & ~127; }

__device__ __forceinline__ float silu(float v) { return v / (1.0f + __expf(-v)); }

// s (low half) and b (high half) of one fp16 pair as floats: s and b - 128 s.
__device__ __forceinline__ void scale_bias(uint32_t sb, float &s, float &bp)
{
    s = half_bits_to_f32(uint16_t(sb & 0xffff));
    bp = fmaf(-128.f, s, half_bits_to_f32(uint16_t(sb >> 16)));
}

// s (low half) and b (high half) of one fp16 pair for an 8-bit atom: s and
// b - 2176 s. With q = lo + 16 hi and the (128 + nibble) fragments of the two
// planes, sum_c (s q_c + b) x_c = s (acc_lo + 16 acc_hi) + (b - 2176 s) sum_c x_c
// (128 + 16 * 128 = 2176).
__device__ __forceinline__ void scale_bias8(uint32_t sb, float &s, float &bp)
{
    s = half_bits_to_f32(uint16_t(sb & 0xffff));
    bp = fmaf(-2176.f, s, half_bits_to_f32(uint16_t(sb >> 16)));
}

// Atom geometry of a BITS-bit blob: bytes per atom and the offset of its
// (s, b) pairs; an 8-bit atom holds the low-nibble plane at 0 and the
// high-nibble plane at kAtomQBytes, each in the 4-bit lane layout.
template <int BITS> struct AtomFmt {
    static constexpr int bytes = BITS == 8 ? kAtom8Bytes : kAtomBytes;
    static constexpr int sb = BITS == 8 ? 2 * kAtomQBytes : kAtomQBytes;
};

// Down rows of one 16-row block over groups [kbeg, kend) of h, h given as bf16
// hi + lo parts ([T][I + 8] each) and per-group sums xh[group][8] of hi + lo.
// wB: the block's atoms, rbB * ngI + kb indexing. y = rows (g, g+8) x tokens
// (2 t4, 2 t4 + 1). Groups two at a time; per group the hi and lo halves of h
// accumulate in separate chains (for 8-bit atoms, per nibble plane as well).
template <int BITS>
__device__ __forceinline__ void down_rows(const uint8_t *wB, int rbB, int ngI, int kbeg, int kend,
                                          const uint16_t *hhi, const uint16_t *hlo, const float *xh, int I,
                                          int T, int lane, float (&y)[4])
{
    using F = AtomFmt<BITS>;
    constexpr int NP = BITS == 8 ? 2 : 1;                 // nibble planes
    const int g = lane >> 2, t4 = lane & 3;
    for (int kb0 = kbeg; kb0 < kend; kb0 += 2) {
        float acc[2][NP][2][4];
        uint4 A[2][NP];
        uint2 SB[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int kb = kb0 + q < kend ? kb0 + q : kb0;
            const uint8_t *atom = wB + (rbB * ngI + kb) * F::bytes;
#pragma unroll
            for (int pl = 0; pl < NP; ++pl) {
                A[q][pl] = *reinterpret_cast<const uint4 *>(atom + pl * kAtomQBytes + 16 * lane);
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[q][pl][0][i] = acc[q][pl][1][i] = 0.f;
            }
            SB[q] = *reinterpret_cast<const uint2 *>(atom + F::sb + 8 * g);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int kb = kb0 + q < kend ? kb0 + q : kb0;
            const int col = kb * kGroup + 16 * t4;
            uint4 ha = make_uint4(0, 0, 0, 0), hb = ha, la = ha, lb = ha;
            if (g < T) {
                ha = *reinterpret_cast<const uint4 *>(hhi + g * (I + 8) + col);
                hb = *reinterpret_cast<const uint4 *>(hhi + g * (I + 8) + col + 8);
                la = *reinterpret_cast<const uint4 *>(hlo + g * (I + 8) + col);
                lb = *reinterpret_cast<const uint4 *>(hlo + g * (I + 8) + col + 8);
            }
            const uint32_t ha_[4] = {ha.x, ha.y, ha.z, ha.w}, hb_[4] = {hb.x, hb.y, hb.z, hb.w};
            const uint32_t la_[4] = {la.x, la.y, la.z, la.w}, lb_[4] = {lb.x, lb.y, lb.z, lb.w};
#pragma unroll
            for (int pl = 0; pl < NP; ++pl)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint4 Ap = A[q][pl];
                    const uint32_t a[4] = {nib_pair(Ap.x, m), nib_pair(Ap.z, m), nib_pair(Ap.y, m), nib_pair(Ap.w, m)};
                    mma_bf16(acc[q][pl][0], a, ha_[m], hb_[m]);
                    mma_bf16(acc[q][pl][1], a, la_[m], lb_[m]);
                }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (kb0 + q >= kend) break;
            const int kb = kb0 + q;
            const float2 X = *reinterpret_cast<const float2 *>(xh + kb * kDecodeMaxT + 2 * t4);
            float s0, bp0, s1, bp1;
            if (BITS == 8) {
                scale_bias8(SB[q].x, s0, bp0);
                scale_bias8(SB[q].y, s1, bp1);
            } else {
                scale_bias(SB[q].x, s0, bp0);
                scale_bias(SB[q].y, s1, bp1);
            }
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = acc[q][0][0][i] + acc[q][0][1][i];
                if (NP == 2) v[i] = fmaf(16.f, acc[q][NP - 1][0][i] + acc[q][NP - 1][1][i], v[i]);
            }
            y[0] += fmaf(s0, v[0], bp0 * X.x);
            y[1] += fmaf(s0, v[1], bp0 * X.y);
            y[2] += fmaf(s1, v[2], bp1 * X.x);
            y[3] += fmaf(s1, v[3], bp1 * X.y);
        }
    }
}

// The step's distinct routed experts, block-wide (all threads call it; needs
// T * k <= 128 <= blockDim.x). One token has distinct experts, so its route
// order serves directly (uniq[j] = ids[j]); several tokens are deduplicated
// in ascending id so an expert two tokens share is streamed once. uidx[pair]
// = 1 + the pair's index into uniq, 0 for an out-of-range id (which also sets
// the error word). Returns the number of entries of uniq; expert index u = 0
// denotes the shared expert, u >= 1 routed expert uniq[u - 1].
__device__ inline int decode_unique_experts(const DecodeParams &p, int *ids_s, int *uidx, int *uniq, int *flags)
{
    const int tid = threadIdx.x, k = p.k, npairs = p.T * k;
    if (p.T == 1) {
        if (tid < k) {
            const int v = p.ids[tid];
            const bool ok = v >= 0 && v < p.E;
            if (!ok) set_error(p.err, SMOE_DEV_BAD_EXPERT);
            uniq[tid] = ok ? v : 0;
            uidx[tid] = ok ? 1 + tid : 0;
        }
        if (tid == 0) flags[0] = k;
        __syncthreads();
    } else {
        if (tid < npairs) ids_s[tid] = p.ids[tid];
        __syncthreads();
        if (tid < npairs) {
            const int v = ids_s[tid];
            const bool ok = v >= 0 && v < p.E;
            if (!ok) set_error(p.err, SMOE_DEV_BAD_EXPERT);
            bool first = ok;
            for (int j = 0; j < tid; ++j)
                if (ids_s[j] == v) first = false;
            flags[2 + tid] = first ? 1 : 0;
        }
        __syncthreads();
        if (tid < npairs) {
            const int v = ids_s[tid];
            int r = 0;
            const bool ok = v >= 0 && v < p.E;
            for (int j = 0; j < npairs; ++j)
                if (flags[2 + j] && ids_s[j] < v) ++r;
            uidx[tid] = ok ? 1 + r : 0;
            if (flags[2 + tid]) uniq[r] = v;
        }
        if (tid == 0) {
            int U = 0;
            for (int j = 0; j < npairs; ++j) U += flags[2 + j];
            flags[0] = U;
        }
        __syncthreads();
    }
    return flags[0];
}

}  // namespace smoe
