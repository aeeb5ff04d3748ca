// decode.cu -- fused expert kernel for small token counts (T <= 8).
//
// One thread-block cluster of cs = I/32 CTAs works on one expert at a time
// (shared expert first, then the routed experts the tokens selected); the
// clusters loop over experts. Inside a cluster:
//   phase A: CTA r computes gate/up for intermediates [32r, 32r+32) over all
//            H inputs and applies SwiGLU -> h slice (fp32, in its shared memory);
//   exchange: every CTA reads the cs slices through distributed shared memory
//            (cluster barriers, no global memory round trip) -> full h;
//   phase B: CTA r computes down rows [r H/cs, (r+1) H/cs) over all I inputs;
//   combine: the expert outputs go to a workspace buffer; per row chunk an
//            arrival ticket picks the last CTA to arrive, which sums, per token,
//            w_j * y_j in route order plus gate * y_shared and writes bf16.
// Weights stream once from HBM with 1-D bulk copies into a ring of shared
// memory slots, one slot per 256-column chunk of phase A, all requested at
// once; phase B's weights then fill the first slots as phase A frees them.
// Each 576-byte atom is the A-operand fragment of 16x8x16 bf16 tensor-core
// steps, dequantised in registers: a nibble pair becomes bf16x2 (128 + q) with
// one shift and one LOP3, the MMA sums (128 + q) x over a 64-column group, and
// the group epilogue applies s and b:
//   sum_c (s q_c + b) x_c = s * sum_c (128 + q_c) x_c + (b - 128 s) * sum_c x_c.
// NCW consumer warps per CTA: 16 when the clusters fit one CTA per SM, 8 when
// two CTAs must share an SM.
// Pages: fixed-stride expert blobs and MLX int4 group quantisation (xix.ai
// article, paragraphs on how it works and on the Metal kernels); combining
// the shared expert (agentlenshq article, how expert streaming works).
#include "decode_common.cuh"

namespace smoe {

struct DecodeSmem {
    int x_s, xsum, ring, hslice, hhi, hlo, xh, red, ints, bars, total, nst;
};

// float4 entries of the cross-warp reduction buffer (per lane)
__host__ __device__ inline int red_entries(int ncw, int H, int cs)
{
    const int a = (ncw / 4 - 1) * kRowBlocksA;            // phase A partials
    const int nrbB = H / cs / 16;
    const int splitB = ncw > nrbB ? ncw / nrbB : 1;
    const int b = (splitB - 1) * nrbB;                     // phase B partials
    const int m = a > b ? a : b;
    return m > 1 ? m : 1;
}

// Bytes of one ring slot (one 256-column chunk of a CTA's gate/up rows) for
// BITS-bit atoms.
__host__ __device__ constexpr int chunk_bytes(int bits)
{
    return kRowBlocksA * (kChunkCols / kGroup) * (bits == 8 ? kAtom8Bytes : kAtomBytes);
}

__host__ __device__ inline DecodeSmem decode_smem(int T, int H, int I, int cs, int ncw, int bits)
{
    DecodeSmem L;
    L.nst = H / kChunkCols;
    int o = 0;
    L.x_s = o;    o = align128(o + T * (2 * H + 16));
    L.xsum = o;   o = align128(o + (H / kGroup) * kDecodeMaxT * 4);
    L.ring = o;   o = align128(o + L.nst * chunk_bytes(bits));
    L.hslice = o; o = align128(o + kDecodeMaxT * kSlice * 4);
    L.hhi = o;    o = align128(o + T * (I + 8) * 2);
    L.hlo = o;    o = align128(o + T * (I + 8) * 2);
    L.xh = o;     o = align128(o + (I / kGroup) * kDecodeMaxT * 4);
    L.red = o;    o = align128(o + red_entries(ncw, H, cs) * 32 * 16);
    L.ints = o;   o = align128(o + 640 * 4);
    L.bars = o;   o = align128(o + (2 * L.nst + 1) * 8);
    L.total = o;
    return L;
}

__device__ __forceinline__ void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// BITS: 4, or 8 for MLX 8-bit experts (two-plane atoms; each plane runs the
// 4-bit fragment path and the group epilogue weights the high plane by 16).
template <int NCW, int BITS>
__global__ void __launch_bounds__((NCW + 1) * 32, 16 / NCW) decode_kernel(const DecodeParams p)
{
    using Fmt = AtomFmt<BITS>;
    constexpr int NP = BITS == 8 ? 2 : 1;           // nibble planes per atom
    constexpr int kCB = chunk_bytes(BITS);          // ring slot bytes
    constexpr int kCons = NCW * 32;                 // consumer threads (named barrier 1)
    constexpr int kGQ = NCW / 4;                    // warps sharing one gate/up row block
    constexpr int kGPW = (kChunkCols / kGroup) / kGQ;   // groups per chunk per warp
    extern __shared__ __align__(1024) uint8_t smem[];
    const int T = p.T, H = p.H, I = p.I, k = p.k;
    const DecodeSmem L = decode_smem(T, H, I, p.cs, NCW, BITS);
    const int nst = L.nst;
    uint16_t *x_s = reinterpret_cast<uint16_t *>(smem + L.x_s);
    float *xsum = reinterpret_cast<float *>(smem + L.xsum);      // [H/64][8]
    uint8_t *ring = smem + L.ring;
    float *hslice = reinterpret_cast<float *>(smem + L.hslice);  // [8][32]
    uint16_t *hhi = reinterpret_cast<uint16_t *>(smem + L.hhi);  // [T][I+8]
    uint16_t *hlo = reinterpret_cast<uint16_t *>(smem + L.hlo);
    float *xh = reinterpret_cast<float *>(smem + L.xh);          // [I/64][8]
    float4 *red = reinterpret_cast<float4 *>(smem + L.red);      // [entries][32]
    int *ints = reinterpret_cast<int *>(smem + L.ints);
    int *ids_s = ints;            // [128]
    int *uidx = ints + 128;       // [128] unique index (1..U) of each pair, 0 if invalid
    int *uniq = ints + 256;       // [<=128] unique expert ids
    int *flags = ints + 384;      // [0] U, [1] is-last, [2..130) first-occurrence marks
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + nst;
    uint64_t *xbar = empty + nst;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const uint32_t rank = cluster_ctarank();
    const uint32_t clus = cluster_id_x(), nclus = ncluster_x();
    const int ngH = H / kGroup, ngI = I / kGroup;
    const int rowsB = H / p.cs;
    const int nrbB = rowsB / 16;
    const int splitB = NCW > nrbB ? NCW / nrbB : 1;      // NCW, nrbB powers of two
    const uint32_t wB_bytes = uint32_t(nrbB * ngI * Fmt::bytes);
    const int nB = int((wB_bytes + kCB - 1) / kCB);      // phase B slots (<= nst)
    const uint64_t down_off = uint64_t(I / 8) * ngH * Fmt::bytes;
    const bool producer = warp == NCW;
    const int xstride = H + 8;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t pol_stream = policy_evict_first();
    // Slot s is filled 1 + (s < nB) times per valid expert, so before the
    // expert with valid-index vit it has been filled vit * (1 + (s < nB)) times.
    auto fills = [&](int vit, int s) { return uint32_t(vit * (1 + (s < nB ? 1 : 0))); };
    bool x_ready = false;    // uniform across the CTA: x rows were waited for
    bool bad = false;        // this thread's bounded wait gave up: skip later waits
                             // (never used to skip a barrier, so all threads still
                             // reach every barrier and the kernel finishes)

    // producer: fill f of slot s (waits for the consumers to free the previous fill)
    auto fill_slot = [&](int s, uint32_t f, const uint8_t *blob, bool phaseA) {
        if (f >= 1 && !mbar_wait(&empty[s], (f - 1) & 1, p.err)) return false;
        uint8_t *dst = ring + s * kCB;
        if (phaseA) {
            mbar_arrive_expect_tx(&full[s], kCB);
            const int per_rb = (kChunkCols / kGroup) * Fmt::bytes;
            for (int rb = 0; rb < kRowBlocksA; ++rb) {
                const uint64_t atom = uint64_t(rank * kRowBlocksA + rb) * ngH + uint64_t(s) * (kChunkCols / kGroup);
                bulk_g2s(dst + rb * per_rb, blob + atom * Fmt::bytes, per_rb, &full[s], pol_stream);
            }
        } else {
            const uint32_t off = uint32_t(s) * kCB;
            const uint32_t bytes = wB_bytes - off < uint32_t(kCB) ? wB_bytes - off : uint32_t(kCB);
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_g2s(dst, blob + down_off + uint64_t(rank) * wB_bytes + off, bytes, &full[s], pol_stream);
        }
        return true;
    };

    // The shared expert (u = 0) needs no routing, so cluster 0 starts streaming
    // its phase-A weights before waiting for the kernel that produced the routing.
    bool pre = false;
    if (producer && lane == 0 && clus == 0) {
        for (int s = 0; s < nst; ++s) fill_slot(s, 0, p.shared_blob, true);
        pre = true;
    }
    pdl_wait();
    pdl_trigger();
    if (producer && lane == 0) {
        mbar_arrive_expect_tx(xbar, uint32_t(T * H * 2));
        for (int t = 0; t < T; ++t)
            bulk_g2s_plain(x_s + t * xstride, p.x + size_t(t) * H, uint32_t(H * 2), xbar);
    }

    // ---- routing bookkeeping: unique experts and pair -> unique index (1..U).
    // The mapping only decides which cluster computes what; every pair still
    // reads its own expert's output.
    const int U_total = decode_unique_experts(p, ids_s, uidx, uniq, flags) + 1;

    int it = 0, vit = 0;
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
                if (!(it == 0 && pre))
                    for (int s = 0; s < nst && !bad; ++s)
                        if (!fill_slot(s, fills(vit, s), blob, true)) bad = true;
                for (int s = 0; s < nB && !bad; ++s)           // phase B into freed slots
                    if (!fill_slot(s, fills(vit, s) + 1, blob, false)) bad = true;
            }
            __syncwarp();
        } else {
            const int rb = warp & 3, gq = warp >> 2;
            float aG0 = 0.f, aG1 = 0.f, aU0 = 0.f, aU1 = 0.f;
            if (valid) {
                if (!x_ready) {
                    if (!bad && !mbar_wait(xbar, 0, p.err)) bad = true;
                    // per-group sums of x for the bias term
                    for (int grp = warp; grp < ngH; grp += NCW)
                        for (int t = 0; t < T; ++t) {
                            const uint32_t v = *reinterpret_cast<const uint32_t *>(x_s + t * xstride + grp * 64 + 2 * lane);
                            float s = bf16lo(v) + bf16hi(v);
                            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                            if (lane == 0) xsum[grp * kDecodeMaxT + t] = s;
                        }
                    named_bar(1, kCons);
                }
                for (int c = 0; c < nst; ++c) {
                    if (!bad && !mbar_wait(&full[c], fills(vit, c) & 1, p.err)) bad = true;
                    const uint8_t *base = ring + c * kCB + rb * (kChunkCols / kGroup) * Fmt::bytes;
#pragma unroll
                    for (int gg = 0; gg < kGPW; ++gg) {
                        const int gl = gq * kGPW + gg;
                        const uint8_t *atom = base + gl * Fmt::bytes;
                        const uint2 SB = *reinterpret_cast<const uint2 *>(atom + Fmt::sb + 8 * g);
                        const int grp = c * (kChunkCols / kGroup) + gl;
                        const int col = grp * kGroup + 16 * t4;
                        uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
                        if (g < T) {
                            xa = *reinterpret_cast<const uint4 *>(x_s + g * xstride + col);
                            xb = *reinterpret_cast<const uint4 *>(x_s + g * xstride + col + 8);
                        }
                        const uint32_t xl[4] = {xa.x, xa.y, xa.z, xa.w};
                        const uint32_t xh4[4] = {xb.x, xb.y, xb.z, xb.w};
                        float v[4];
#pragma unroll
                        for (int pl = 0; pl < NP; ++pl) {         // nibble planes (8-bit: low, then high)
                            const uint4 A = *reinterpret_cast<const uint4 *>(atom + pl * kAtomQBytes + 16 * lane);
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
                            for (int i = 0; i < 4; ++i)
                                v[i] = pl == 0 ? acc[i] + acc2[i] : fmaf(16.f, acc[i] + acc2[i], v[i]);
                        }
                        const float2 X = *reinterpret_cast<const float2 *>(xsum + grp * kDecodeMaxT + 2 * t4);
                        float sg, bpg, su, bpu;
                        if (BITS == 8) {
                            scale_bias8(SB.x, sg, bpg);
                            scale_bias8(SB.y, su, bpu);
                        } else {
                            scale_bias(SB.x, sg, bpg);
                            scale_bias(SB.y, su, bpu);
                        }
                        aG0 += fmaf(sg, v[0], bpg * X.x);
                        aG1 += fmaf(sg, v[1], bpg * X.y);
                        aU0 += fmaf(su, v[2], bpu * X.x);
                        aU1 += fmaf(su, v[3], bpu * X.y);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[c]);
                }
            }
            // add the K parts of each row block, SwiGLU, h slice -> own shared memory
            if (gq > 0) red[((gq - 1) * kRowBlocksA + rb) * 32 + lane] = make_float4(aG0, aG1, aU0, aU1);
            named_bar(1, kCons);
            if (gq == 0) {
#pragma unroll
                for (int q = 1; q < kGQ; ++q) {
                    const float4 v = red[((q - 1) * kRowBlocksA + rb) * 32 + lane];
                    aG0 += v.x; aG1 += v.y; aU0 += v.z; aU1 += v.w;
                }
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
            for (int i = tid; i < nitems; i += kCons) {
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
            named_bar(1, kCons);
            for (int grp = warp; grp < ngI; grp += NCW)
                for (int t = 0; t < T; ++t) {
                    const uint32_t vh = *reinterpret_cast<const uint32_t *>(hhi + t * (I + 8) + grp * 64 + 2 * lane);
                    const uint32_t vl = *reinterpret_cast<const uint32_t *>(hlo + t * (I + 8) + grp * 64 + 2 * lane);
                    float s = (bf16lo(vh) + bf16lo(vl)) + (bf16hi(vh) + bf16hi(vl));
                    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (lane == 0) xh[grp * kDecodeMaxT + t] = s;
                }
            named_bar(1, kCons);
        }
        cluster_arrive();   // done reading peers' slices; matched by the wait at the next iteration / exit

        // ---- phase B: down rows of this CTA, full K = I, from ring slots 0..nB-1
        if (!producer) {
            if (valid)
                for (int s = 0; s < nB; ++s)
                    if (!bad && !mbar_wait(&full[s], (fills(vit, s) + 1) & 1, p.err)) bad = true;
            float *yp = p.ypair + size_t(u) * T * H;
            const int t0 = 2 * t4, t1 = t0 + 1;
            auto store = [&](int rbB, const float (&y)[4]) {
                const int row = int(rank) * rowsB + rbB * 16 + g;
                if (t0 < T) { yp[size_t(t0) * H + row] = y[0]; yp[size_t(t0) * H + row + 8] = y[2]; }
                if (t1 < T) { yp[size_t(t1) * H + row] = y[1]; yp[size_t(t1) * H + row + 8] = y[3]; }
            };
            if (splitB > 1) {
                // one (row block, K part) per warp; the K parts meet in shared memory
                const int rbB = warp % nrbB, sp = warp / nrbB;
                const int kb_per = (ngI + splitB - 1) / splitB;
                const int kbeg = sp * kb_per < ngI ? sp * kb_per : ngI;
                const int kend = kbeg + kb_per < ngI ? kbeg + kb_per : ngI;
                float y[4] = {0.f, 0.f, 0.f, 0.f};
                if (valid && !bad) down_rows<BITS>(ring, rbB, ngI, kbeg, kend, hhi, hlo, xh, I, T, lane, y);
                if (valid) {
                    __syncwarp();
                    if (lane == 0)
                        for (int s = 0; s < nB; ++s) mbar_arrive(&empty[s]);
                }
                if (sp > 0) red[((sp - 1) * nrbB + rbB) * 32 + lane] = make_float4(y[0], y[1], y[2], y[3]);
                named_bar(1, kCons);
                if (sp == 0) {
                    for (int q = 1; q < splitB; ++q) {
                        const float4 v = red[((q - 1) * nrbB + rbB) * 32 + lane];
                        y[0] += v.x; y[1] += v.y; y[2] += v.z; y[3] += v.w;
                    }
                    store(rbB, y);
                }
            } else {
                for (int rbB = warp; rbB < nrbB; rbB += NCW) {
                    float y[4] = {0.f, 0.f, 0.f, 0.f};
                    if (valid && !bad) down_rows<BITS>(ring, rbB, ngI, 0, ngI, hhi, hlo, xh, I, T, lane, y);
                    store(rbB, y);
                }
                if (valid) {
                    __syncwarp();
                    if (lane == 0)
                        for (int s = 0; s < nB; ++s) mbar_arrive(&empty[s]);
                }
            }

            // ---- arrival ticket for this row chunk; the last arrival combines
            named_bar(1, kCons);
            if (tid == 0) {
                const uint32_t old = ticket_add(&p.counters[rank], 1u);
                flags[1] = (old == uint32_t(U_total - 1)) ? 1 : 0;
            }
            named_bar(1, kCons);
            if (flags[1]) {
                for (int i = tid; i < T * rowsB; i += kCons) {
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
                named_bar(1, kCons);
                if (tid == 0) atomicExch(&p.counters[rank], 0u);
            }
        }
        if (valid) ++vit;
        __syncthreads();
    }
    if (it > 0) cluster_wait();
    if (!x_ready) {               // x rows were loaded but never waited for: do not exit with
        if (tid == 0) mbar_wait(xbar, 0, p.err);   // a copy into this CTA still in flight
        __syncthreads();
    }
}

template <int NCW, int BITS>
static cudaError_t config_one(smoe_ctx *ctx, int max_smem_optin, int *smem_out, int *clusters_out)
{
    const smoe_shape &s = ctx->shape;
    int worst = 0;
    for (int T = 1; T <= kDecodeMaxT; ++T) {
        const int sm = decode_smem(T, s.H, s.I, ctx->cs, NCW, BITS).total;
        smem_out[T] = sm;
        if (sm > worst) worst = sm;
    }
    if (worst > max_smem_optin) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<NCW, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, worst);
    if (e == cudaSuccess && ctx->cs > 8)
        e = cudaFuncSetAttribute(decode_kernel<NCW, BITS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    for (int T = 1; T <= kDecodeMaxT; ++T) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(ctx->cs * 64);
        lc.blockDim = dim3((NCW + 1) * 32);
        lc.dynamicSmemBytes = smem_out[T];
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = ctx->cs;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, decode_kernel<NCW, BITS>, &lc);
        if (e != cudaSuccess) return e;
        clusters_out[T] = n;
    }
    return cudaSuccess;
}

template <int BITS>
static cudaError_t decode_config_bits(smoe_ctx *ctx)
{
    int max_smem_optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device);
    if (e != cudaSuccess) return e;
    int sm8[kDecodeMaxT + 1], cl8[kDecodeMaxT + 1], sm16[kDecodeMaxT + 1], cl16[kDecodeMaxT + 1];
    e = config_one<8, BITS>(ctx, max_smem_optin, sm8, cl8);
    if (e != cudaSuccess) return e;
    e = config_one<16, BITS>(ctx, max_smem_optin, sm16, cl16);
    if (e != cudaSuccess) return e;
    for (int T = 1; T <= kDecodeMaxT; ++T) {
        if (cl8[T] < 1) return cudaErrorInvalidConfiguration;
        ctx->decode[T].nst = ctx->shape.H / kChunkCols;
        ctx->decode[T].smem = sm8[T];
        ctx->decode[T].max_clusters = cl8[T];
        ctx->decode[T].smem16 = sm16[T];
        ctx->decode[T].max_clusters16 = cl16[T];
    }
    return cudaSuccess;
}

cudaError_t decode_config(smoe_ctx *ctx)
{
    ctx->decode_ok = false;
    if (ctx->shape.bits == 8) {
        // 8-bit contexts also serve routing and the plain path, so a shape whose
        // 8-bit ring does not fit leaves the fast kernel unavailable (ENOTSUP)
        // instead of failing the context
        const cudaError_t e = decode_config_bits<8>(ctx);
        if (e == cudaErrorInvalidValue || e == cudaErrorInvalidConfiguration) {
            cudaGetLastError();
            return cudaSuccess;
        }
        if (e == cudaSuccess) ctx->decode_ok = true;
        return e;
    }
    const cudaError_t e = decode_config_bits<4>(ctx);
    if (e == cudaSuccess) ctx->decode_ok = true;
    return e;
}

cudaError_t launch_decode(const smoe_ctx *ctx, const DecodeParams &p0, cudaStream_t st)
{
    DecodeParams p = p0;
    const DecodeCfg &cfg = ctx->decode[p.T];
    p.cs = ctx->cs;
    const int umax = (p.E < p.T * p.k ? p.E : p.T * p.k) + 1;
    // 16 consumer warps (one CTA per SM) when every expert gets its own
    // co-resident cluster that way; otherwise 8 (two CTAs per SM).
    const bool wide = umax * p.cs <= ctx->num_sms && cfg.max_clusters16 >= umax;
    const int maxc = wide ? cfg.max_clusters16 : cfg.max_clusters;
    const int nclus = umax < maxc ? umax : maxc;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(nclus * p.cs);
    lc.blockDim = dim3(((wide ? 16 : 8) + 1) * 32);
    lc.dynamicSmemBytes = wide ? cfg.smem16 : cfg.smem;
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
    if (ctx->shape.bits == 8)
        return wide ? cudaLaunchKernelEx(&lc, decode_kernel<16, 8>, p) : cudaLaunchKernelEx(&lc, decode_kernel<8, 8>, p);
    return wide ? cudaLaunchKernelEx(&lc, decode_kernel<16, 4>, p) : cudaLaunchKernelEx(&lc, decode_kernel<8, 4>, p);
}

}  // namespace smoe
