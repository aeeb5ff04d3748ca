// decode.cu -- fused expert kernel for small token counts (T <= 8).
//
// One thread-block cluster of cs = I/32 CTAs works on one expert at a time
// (shared expert first, then the routed experts the tokens selected, in
// ascending id); clusters loop over experts. Inside a cluster:
//   phase A: CTA r computes gate/up for intermediates [32r, 32r+32) over all
//            H inputs and applies SwiGLU -> h slice (fp32, in its shared memory);
//   exchange: every CTA reads the cs slices through distributed shared memory
//            (cluster barriers, no global memory round trip) -> full h;
//   phase B: CTA r computes down rows [r H/cs, (r+1) H/cs) over all I inputs;
//   combine: the expert outputs go to a workspace buffer; per row chunk an
//            arrival ticket picks the last CTA to arrive, which sums, per token,
//            w_j * y_j in route order plus gate * y_shared and writes bf16.
// The weights stream once from HBM with 1-D bulk copies into a ring of shared
// memory stages; each 576-byte atom is the A-operand fragment of 16x8x16 bf16
// tensor-core steps, dequantised in registers: a nibble pair becomes
// bf16x2 (128+q) with one shift and one LOP3, the MMA sums (128+q) x over a
// 64-column group, and the group epilogue applies s and b:
//   sum_c (s q_c + b) x_c = s * sum_c (128 + q_c) x_c + (b - 128 s) * sum_c x_c.
// Pages: fixed-stride expert blobs and MLX int4 group quantisation (xix.ai
// article, paragraphs on how it works and on the Metal kernels); combining
// the shared expert (agentlenshq article, how expert streaming works).
#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

struct DecodeSmem {
    int x_s, xsum, wB, ring, hslice, hhi, hlo, xh, red, ints, bars, total;
};

__host__ __device__ inline int align128(int v) { return (v + 127) & ~127; }

__host__ __device__ inline DecodeSmem decode_smem(int T, int H, int I, int cs, int nst)
{
    DecodeSmem L;
    int o = 0;
    L.x_s = o;    o = align128(o + T * (2 * H + 16));
    L.xsum = o;   o = align128(o + (H / kGroup) * kDecodeMaxT * 4);
    L.wB = o;     o = align128(o + (H / cs / 16) * (I / kGroup) * kAtomBytes);
    L.ring = o;   o = align128(o + nst * kChunkBytes);
    L.hslice = o; o = align128(o + kDecodeMaxT * kSlice * 4);
    L.hhi = o;    o = align128(o + T * (I + 8) * 2);
    L.hlo = o;    o = align128(o + T * (I + 8) * 2);
    L.xh = o;     o = align128(o + (I / kGroup) * kDecodeMaxT * 4);
    L.red = o;    o = align128(o + kRowBlocksA * 32 * 16);
    L.ints = o;   o = align128(o + 640 * 4);
    L.bars = o;   o = align128(o + (2 * nst + 2) * 8);
    L.total = o;
    return L;
}

__device__ __forceinline__ float silu(float v) { return v / (1.0f + __expf(-v)); }

__device__ __forceinline__ void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(const DecodeParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int T = p.T, H = p.H, I = p.I, k = p.k, nst = p.nst;
    const DecodeSmem L = decode_smem(T, H, I, p.cs, nst);
    uint16_t *x_s = reinterpret_cast<uint16_t *>(smem + L.x_s);
    float *xsum = reinterpret_cast<float *>(smem + L.xsum);      // [H/64][8]
    uint8_t *wB = smem + L.wB;
    uint8_t *ring = smem + L.ring;
    float *hslice = reinterpret_cast<float *>(smem + L.hslice);  // [8][32]
    uint16_t *hhi = reinterpret_cast<uint16_t *>(smem + L.hhi);  // [T][I+8]
    uint16_t *hlo = reinterpret_cast<uint16_t *>(smem + L.hlo);
    float *xh = reinterpret_cast<float *>(smem + L.xh);          // [I/64][8]
    float4 *red = reinterpret_cast<float4 *>(smem + L.red);      // [4][32]
    int *ints = reinterpret_cast<int *>(smem + L.ints);
    int *ids_s = ints;            // [128]
    int *uidx = ints + 128;       // [128] unique index (1..U) of each pair, 0 if invalid
    int *uniq = ints + 256;       // [<=128] unique expert ids, ascending
    int *flags = ints + 384;      // [0] U, [1] is-last, [2..130) first-occurrence marks
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + nst;
    uint64_t *xbar = empty + nst;
    uint64_t *wbar = xbar + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const uint32_t rank = cluster_ctarank();
    const uint32_t clus = cluster_id_x(), nclus = ncluster_x();
    const int nchunks = H / kChunkCols;
    const int ngH = H / kGroup, ngI = I / kGroup;
    const int rowsB = H / p.cs;
    const int nrbB = rowsB / 16;
    const uint32_t wB_bytes = uint32_t(nrbB * ngI * kAtomBytes);
    const uint64_t down_off = uint64_t(I / 8) * ngH * kAtomBytes;
    const bool producer = warp == kDecodeConsumerWarps;
    const int xstride = H + 8;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kDecodeConsumerWarps);
        }
        mbar_init(xbar, 1);
        mbar_init(wbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t pol_stream = policy_evict_first();
    uint32_t qnext = 0;      // producer: chunks issued so far (ring sequence)
    uint32_t qdone = 0;      // consumers: chunks consumed so far
    uint32_t nw = 0;         // phase-B weight loads consumed
    bool x_ready = false;    // uniform across the CTA: x rows were waited for
    bool bad = false;        // this thread's bounded wait gave up: skip later waits
                             // (never used to skip a barrier, so all threads still
                             // reach every barrier and the kernel finishes)
    int pre_chunks = 0;
    bool pre_w = false;

    auto issue_chunk = [&](const uint8_t *blob, int c) {
        const uint32_t slot = qnext % nst;
        if (qnext >= (uint32_t)nst && !mbar_wait(&empty[slot], ((qnext / nst) - 1) & 1, p.err))
            return false;
        mbar_arrive_expect_tx(&full[slot], kChunkBytes);
        uint8_t *dst = ring + slot * kChunkBytes;
        const int per_rb = (kChunkCols / kGroup) * kAtomBytes;
        for (int rb = 0; rb < kRowBlocksA; ++rb) {
            const uint64_t atom = uint64_t(rank * kRowBlocksA + rb) * ngH + uint64_t(c) * (kChunkCols / kGroup);
            bulk_g2s(dst + rb * per_rb, blob + atom * kAtomBytes, per_rb, &full[slot], pol_stream);
        }
        ++qnext;
        return true;
    };
    auto issue_w = [&](const uint8_t *blob) {
        mbar_arrive_expect_tx(wbar, wB_bytes);
        bulk_g2s(wB, blob + down_off + uint64_t(rank) * wB_bytes, wB_bytes, wbar, pol_stream);
    };

    // The shared expert (u = 0) needs no routing, so cluster 0 starts streaming
    // it before waiting for the kernel that produced the routing.
    if (producer && lane == 0 && clus == 0) {
        issue_w(p.shared_blob);
        pre_w = true;
        for (int c = 0; c < nchunks && c < nst; ++c) {
            issue_chunk(p.shared_blob, c);
            ++pre_chunks;
        }
    }
    pdl_wait();
    pdl_trigger();
    if (producer && lane == 0) {
        mbar_arrive_expect_tx(xbar, uint32_t(T * H * 2));
        for (int t = 0; t < T; ++t)
            bulk_g2s_plain(x_s + t * xstride, p.x + size_t(t) * H, uint32_t(H * 2), xbar);
    }

    // ---- routing bookkeeping: unique experts and pair -> unique index (1..U).
    // One token has distinct experts, so its route order serves directly;
    // several tokens are deduplicated (ascending id) so a shared expert is
    // streamed once. Either way the mapping only decides which cluster
    // computes what; every pair still reads its own expert's output.
    const int npairs = T * k;
    if (T == 1) {
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
    const int U_total = flags[0] + 1;

    int it = 0;
    for (int u = int(clus); u < U_total; u += int(nclus), ++it) {
        if (it > 0) cluster_wait();   // peers are done reading our previous h slice

        const uint8_t *blob = nullptr;
        bool valid = true;
        if (u == 0) {
            blob = p.shared_blob;
        } else {
            const int e = uniq[u - 1];
            const int64_t slot = p.table_row[e];
            if (slot < 0 || slot >= p.n_slots) {
                valid = false;
                set_error(p.err, SMOE_DEV_BAD_SLOT);
            } else {
                blob = p.pool + uint64_t(slot) * p.stride;
            }
        }

        if (producer) {
            if (lane == 0 && valid && !bad) {
                if (!(it == 0 && pre_w)) issue_w(blob);
                for (int c = (it == 0 ? pre_chunks : 0); c < nchunks; ++c)
                    if (!issue_chunk(blob, c)) { bad = true; break; }
            }
            __syncwarp();
        } else {
            const int rb = warp & 3, gh = warp >> 2;
            float aG0 = 0.f, aG1 = 0.f, aU0 = 0.f, aU1 = 0.f;
            if (valid) {
                if (!x_ready) {
                    if (!bad && !mbar_wait(xbar, 0, p.err)) bad = true;
                    // per-group sums of x for the bias term: warp w sums groups w, w+8, ...
                    for (int grp = warp; grp < ngH; grp += kDecodeConsumerWarps)
                        for (int t = 0; t < T; ++t) {
                            const uint32_t v = *reinterpret_cast<const uint32_t *>(x_s + t * xstride + grp * 64 + 2 * lane);
                            float s = bf16lo(v) + bf16hi(v);
                            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                            if (lane == 0) xsum[grp * kDecodeMaxT + t] = s;
                        }
                    named_bar(1, kDecodeConsumerWarps * 32);
                }
                for (int c = 0; c < nchunks; ++c, ++qdone) {
                    const uint32_t slot = qdone % nst;
                    if (!bad && !mbar_wait(&full[slot], (qdone / nst) & 1, p.err)) bad = true;
                    const uint8_t *base = ring + slot * kChunkBytes + rb * (kChunkCols / kGroup) * kAtomBytes;
#pragma unroll
                    for (int gg = 0; gg < 2; ++gg) {
                        const int gl = 2 * gh + gg;
                        const uint8_t *atom = base + gl * kAtomBytes;
                        const uint4 A = *reinterpret_cast<const uint4 *>(atom + 16 * lane);
                        const uint2 SB = *reinterpret_cast<const uint2 *>(atom + kAtomQBytes + 8 * g);
                        const int grp = c * (kChunkCols / kGroup) + gl;
                        const int col = grp * kGroup + 16 * t4;
                        uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
                        if (g < T) {
                            xa = *reinterpret_cast<const uint4 *>(x_s + g * xstride + col);
                            xb = *reinterpret_cast<const uint4 *>(x_s + g * xstride + col + 8);
                        }
                        const uint32_t xl[4] = {xa.x, xa.y, xa.z, xa.w};
                        const uint32_t xh4[4] = {xb.x, xb.y, xb.z, xb.w};
                        float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int m = 0; m < 4; m += 2) {   // two independent chains of two
                            const uint32_t a0[4] = {nib_pair(A.x, m), nib_pair(A.z, m), nib_pair(A.y, m),
                                                    nib_pair(A.w, m)};
                            const uint32_t a1[4] = {nib_pair(A.x, m + 1), nib_pair(A.z, m + 1),
                                                    nib_pair(A.y, m + 1), nib_pair(A.w, m + 1)};
                            mma_bf16(acc, a0, xl[m], xh4[m]);
                            mma_bf16(acc2, a1, xl[m + 1], xh4[m + 1]);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
                        const float2 X = *reinterpret_cast<const float2 *>(xsum + grp * kDecodeMaxT + 2 * t4);
                        const float sg = half_bits_to_f32(uint16_t(SB.x & 0xffff));
                        const float bg = half_bits_to_f32(uint16_t(SB.x >> 16));
                        const float su = half_bits_to_f32(uint16_t(SB.y & 0xffff));
                        const float bu = half_bits_to_f32(uint16_t(SB.y >> 16));
                        const float bpg = fmaf(-128.f, sg, bg), bpu = fmaf(-128.f, su, bu);
                        aG0 += fmaf(sg, acc[0], bpg * X.x);
                        aG1 += fmaf(sg, acc[1], bpg * X.y);
                        aU0 += fmaf(su, acc[2], bpu * X.x);
                        aU1 += fmaf(su, acc[3], bpu * X.y);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                }
            }
            // combine the two K halves, SwiGLU, h slice -> own shared memory
            if (gh == 1) red[rb * 32 + lane] = make_float4(aG0, aG1, aU0, aU1);
            named_bar(1, kDecodeConsumerWarps * 32);
            if (gh == 0) {
                const float4 v = red[rb * 32 + lane];
                aG0 += v.x; aG1 += v.y; aU0 += v.z; aU1 += v.w;
                const int il = rb * 8 + g;
                const int t0 = 2 * t4, t1 = t0 + 1;
                if (t0 < T) hslice[t0 * kSlice + il] = (valid && !bad) ? silu(aG0) * aU0 : 0.f;
                if (t1 < T) hslice[t1 * kSlice + il] = (valid && !bad) ? silu(aG1) * aU1 : 0.f;
            }
        }

        if (valid) x_ready = true;   // every thread: valid is uniform in the cluster

        // ---- exchange h slices inside the cluster
        cluster_arrive();
        cluster_wait();
        if (!producer) {
            const int nitems = p.cs * T * (kSlice / 4);
            for (int i = tid; i < nitems; i += kDecodeConsumerWarps * 32) {
                const int q4 = i % (kSlice / 4);
                const int rest = i / (kSlice / 4);
                const int tok = rest % T, peer = rest / T;
                const float4 v = dsmem_ld_f4(dsmem_addr(hslice + tok * kSlice + q4 * 4, uint32_t(peer)));
                const uint32_t h01 = pack_bf16x2(v.x, v.y), h23 = pack_bf16x2(v.z, v.w);
                const uint32_t l01 = pack_bf16x2(v.x - bf16lo(h01), v.y - bf16hi(h01));
                const uint32_t l23 = pack_bf16x2(v.z - bf16lo(h23), v.w - bf16hi(h23));
                const int col = peer * kSlice + q4 * 4;
                *reinterpret_cast<uint2 *>(hhi + tok * (I + 8) + col) = make_uint2(h01, h23);
                *reinterpret_cast<uint2 *>(hlo + tok * (I + 8) + col) = make_uint2(l01, l23);
            }
            named_bar(1, kDecodeConsumerWarps * 32);
            for (int grp = warp; grp < ngI; grp += kDecodeConsumerWarps)
                for (int t = 0; t < T; ++t) {
                    const uint32_t vh = *reinterpret_cast<const uint32_t *>(hhi + t * (I + 8) + grp * 64 + 2 * lane);
                    const uint32_t vl = *reinterpret_cast<const uint32_t *>(hlo + t * (I + 8) + grp * 64 + 2 * lane);
                    float s = (bf16lo(vh) + bf16lo(vl)) + (bf16hi(vh) + bf16hi(vl));
                    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (lane == 0) xh[grp * kDecodeMaxT + t] = s;
                }
            named_bar(1, kDecodeConsumerWarps * 32);
        }
        cluster_arrive();   // done reading peers' slices; matched by the wait at the next iteration / exit

        // ---- phase B: down rows of this CTA, full K = I
        if (!producer) {
            const bool run = valid && !bad;
            if (run) {
                if (!mbar_wait(wbar, nw & 1, p.err)) bad = true;
                ++nw;
            }
            float *yp = p.ypair + size_t(u) * T * H;
            for (int rbB = warp; rbB < nrbB; rbB += kDecodeConsumerWarps) {
                float y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
                if (run && !bad) {
                    // groups two at a time; per group the hi and lo halves of h
                    // accumulate in separate chains (four independent chains)
                    for (int kb0 = 0; kb0 < ngI; kb0 += 2) {
                        float acc[2][2][4];
                        uint4 A[2];
                        uint2 SB[2];
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int kb = kb0 + q < ngI ? kb0 + q : kb0;
                            const uint8_t *atom = wB + (rbB * ngI + kb) * kAtomBytes;
                            A[q] = *reinterpret_cast<const uint4 *>(atom + 16 * lane);
                            SB[q] = *reinterpret_cast<const uint2 *>(atom + kAtomQBytes + 8 * g);
#pragma unroll
                            for (int i = 0; i < 4; ++i) acc[q][0][i] = acc[q][1][i] = 0.f;
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int kb = kb0 + q < ngI ? kb0 + q : kb0;
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
                            for (int m = 0; m < 4; ++m) {
                                const uint32_t a[4] = {nib_pair(A[q].x, m), nib_pair(A[q].z, m),
                                                       nib_pair(A[q].y, m), nib_pair(A[q].w, m)};
                                mma_bf16(acc[q][0], a, ha_[m], hb_[m]);
                                mma_bf16(acc[q][1], a, la_[m], lb_[m]);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            if (kb0 + q >= ngI) break;
                            const int kb = kb0 + q;
                            const float2 X = *reinterpret_cast<const float2 *>(xh + kb * kDecodeMaxT + 2 * t4);
                            const float s0 = half_bits_to_f32(uint16_t(SB[q].x & 0xffff));
                            const float b0 = half_bits_to_f32(uint16_t(SB[q].x >> 16));
                            const float s1 = half_bits_to_f32(uint16_t(SB[q].y & 0xffff));
                            const float b1 = half_bits_to_f32(uint16_t(SB[q].y >> 16));
                            const float bp0 = fmaf(-128.f, s0, b0), bp1 = fmaf(-128.f, s1, b1);
                            y0 += fmaf(s0, acc[q][0][0] + acc[q][1][0], bp0 * X.x);
                            y1 += fmaf(s0, acc[q][0][1] + acc[q][1][1], bp0 * X.y);
                            y2 += fmaf(s1, acc[q][0][2] + acc[q][1][2], bp1 * X.x);
                            y3 += fmaf(s1, acc[q][0][3] + acc[q][1][3], bp1 * X.y);
                        }
                    }
                }
                const int row = int(rank) * rowsB + rbB * 16 + g;
                const int t0 = 2 * t4, t1 = t0 + 1;
                if (t0 < T) { yp[size_t(t0) * H + row] = y0; yp[size_t(t0) * H + row + 8] = y2; }
                if (t1 < T) { yp[size_t(t1) * H + row] = y1; yp[size_t(t1) * H + row + 8] = y3; }
            }

            // ---- arrival ticket for this row chunk; the last arrival combines
            named_bar(1, kDecodeConsumerWarps * 32);
            if (tid == 0) {
                __threadfence();
                const uint32_t old = atomicAdd(&p.counters[rank], 1u);
                flags[1] = (old == uint32_t(U_total - 1)) ? 1 : 0;
            }
            named_bar(1, kDecodeConsumerWarps * 32);
            if (flags[1]) {
                __threadfence();
                for (int i = tid; i < T * rowsB; i += kDecodeConsumerWarps * 32) {
                    const int tok = i / rowsB;
                    const int row = int(rank) * rowsB + i % rowsB;
                    // all loads first (k <= 16), then the sum in route order
                    float yv[16], wv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        yv[j] = 0.f;
                        wv[j] = 0.f;
                        if (j < k) {
                            const int uu = uidx[tok * k + j];
                            if (uu > 0) {
                                yv[j] = __ldcg(p.ypair + (size_t(uu) * T + tok) * H + row);
                                wv[j] = p.w[tok * k + j];
                            }
                        }
                    }
                    const float ys = __ldcg(p.ypair + size_t(tok) * H + row);
                    const float gt = p.gate[tok];
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < k) acc = fmaf(wv[j], yv[j], acc);
                    acc = fmaf(gt, ys, acc);
                    if (p.residual) acc += __uint_as_float(uint32_t(p.residual[size_t(tok) * H + row]) << 16);
                    p.out[size_t(tok) * H + row] = f32_to_bf16_bits(acc);
                }
                named_bar(1, kDecodeConsumerWarps * 32);
                if (tid == 0) atomicExch(&p.counters[rank], 0u);
            }
        }
        __syncthreads();
    }
    if (it > 0) cluster_wait();
    if (!x_ready) {               // x rows were loaded but never waited for: do not exit with
        if (tid == 0) mbar_wait(xbar, 0, p.err);   // a copy into this CTA still in flight
        __syncthreads();
    }
}

cudaError_t decode_config(smoe_ctx *ctx)
{
    const smoe_shape &s = ctx->shape;
    const int nchunks = s.H / kChunkCols;
    int max_smem_optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device);
    if (e != cudaSuccess) return e;
    int worst = 0;
    for (int T = 1; T <= kDecodeMaxT; ++T) {
        int nst = nchunks < 8 ? nchunks : 8;
        // prefer two CTAs per SM (<= 113 KB each) while keeping >= 4 stages in flight
        while (nst > 4 && decode_smem(T, s.H, s.I, ctx->cs, nst).total > 113 * 1024) --nst;
        while (nst > 2 && decode_smem(T, s.H, s.I, ctx->cs, nst).total > max_smem_optin) --nst;
        const int sm = decode_smem(T, s.H, s.I, ctx->cs, nst).total;
        if (sm > max_smem_optin) return cudaErrorInvalidValue;
        ctx->decode[T].nst = nst;
        ctx->decode[T].smem = sm;
        if (sm > worst) worst = sm;
    }
    e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, worst);
    if (e != cudaSuccess) return e;
    if (ctx->cs > 8) {
        e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    for (int T = 1; T <= kDecodeMaxT; ++T) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(ctx->cs * 64);
        lc.blockDim = dim3(kDecodeThreads);
        lc.dynamicSmemBytes = ctx->decode[T].smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = ctx->cs;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, decode_kernel, &lc);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        ctx->decode[T].max_clusters = n;
    }
    return cudaSuccess;
}

cudaError_t launch_decode(const smoe_ctx *ctx, const DecodeParams &p0, cudaStream_t st)
{
    DecodeParams p = p0;
    const DecodeCfg &cfg = ctx->decode[p.T];
    p.nst = cfg.nst;
    p.cs = ctx->cs;
    const int umax = (p.E < p.T * p.k ? p.E : p.T * p.k) + 1;
    const int nclus = umax < cfg.max_clusters ? umax : cfg.max_clusters;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(nclus * p.cs);
    lc.blockDim = dim3(kDecodeThreads);
    lc.dynamicSmemBytes = cfg.smem;
    lc.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = p.cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 2;
    return cudaLaunchKernelEx(&lc, decode_kernel, p);
}

}  // namespace smoe
