// prefill.cu -- the token-bucketed path for T > 8 (batched decode, prefill).
//
//   bucketing: a deterministic counting sort of the T*k (token, slot) pairs by
//     expert (per-chunk counts, one scan, an ordered scatter), plus the list of
//     GEMM tiles: per expert, runs of up to 256 of its pairs; the shared
//     expert takes all T tokens;
//   gate/up GEMM: per tile, 128 weight rows (64 gate + 64 up rows, interleaved
//     in blocks of 8 as the blob stores them) x its tokens, K = H; the int4
//     atoms are dequantised to bf16 in shared memory (128-byte swizzled,
//     K-major) and multiplied on tcgen05 tensor cores with the accumulator in
//     TMEM; the epilogue applies SwiGLU and writes h;
//   down GEMM: per tile, 128 down rows x its pairs, K = I, B = h rows; the
//     epilogue scales by the routing weight (or the shared-expert gate);
//   combine: per token, the k pair outputs in route order, then the shared
//     expert (and the residual), rounded once to bf16.
// The expert GEMMs take fp16 operands (weights s q + b and h keep 11
// significant bits; x converts exactly for |x| < 65504, else the error word is
// set); the same kernel with bf16 router rows and bf16 x computes the router
// logits for large T. Swap-AB: weights take the 128-row M side, tokens the N side,
// so a tile fits an expert's ~160 tokens without padding to 128.
// Pages: the sparse MoE layer (xix.ai article, paragraph on how it works);
// prefill as the slow part on the pages' hardware (paper-digest, Community
// Reactions).
#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

constexpr int kPfM = 128;          // weight rows per tile
constexpr int kPfK = 64;           // K per pipeline stage (one quantisation group)
constexpr int kPfMaxN = 256;       // tokens per tile
constexpr int kPfStages = 3;
constexpr int kPfWorkers = 8;      // warps: B loads, A dequant, epilogue
constexpr int kPfThreads = (kPfWorkers + 2) * 32;   // + producer warp + MMA warp
constexpr int kPfRawBytes = 5120;  // 8 atoms (4608 B) rounded up to 1 KiB
constexpr int kPfABytes = kPfM * kPfK * 2;          // 16 KiB
constexpr int kPfBBytes = kPfMaxN * kPfK * 2;       // 32 KiB
constexpr int kPfStageBytes = kPfRawBytes + kPfABytes + kPfBBytes;
constexpr int kPfSmem = kPfStages * kPfStageBytes + 1024 /*align*/ + 256 /*barriers*/;
constexpr int kBucketTok = 64;     // tokens per bucketing chunk

__device__ __forceinline__ uint32_t sw128(int r, int c)   // byte offset of (row, col) in a 64-col bf16 tile
{
    return uint32_t(r * 128 + ((((c * 2) >> 4) ^ (r & 7)) << 4) + ((c * 2) & 15));
}

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr)
{
    uint64_t d = uint64_t((saddr & 0x3FFFF) >> 4);   // start address
    d |= uint64_t(1) << 16;                          // leading byte offset (unused: 128 B swizzle, K-major)
    d |= uint64_t(1024 >> 4) << 32;                  // stride byte offset: 8 rows of 128 B
    d |= uint64_t(1) << 46;                          // descriptor version
    d |= uint64_t(2) << 61;                          // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: f32 accumulator, K-major A and B, M = 128,
// operands fp16 (bf16 = false) or bf16 (bf16 = true).
__device__ __forceinline__ uint32_t umma_idesc(int n, bool bf16)
{
    const uint32_t fmt = bf16 ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(kPfM >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float v)
{
    uint16_t r;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}

// x (bf16) -> fp16 for the expert GEMMs: exact for |x| < 65504 (and subnormal
// below 2^-14, an absolute error under 3e-8); larger values set the error word.
__global__ void __launch_bounds__(256) x_to_half_kernel(const uint16_t *x, uint16_t *xh, long long n8, int32_t *err)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const uint4 v = reinterpret_cast<const uint4 *>(x)[i];
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = bf16lo(in[j]), b = bf16hi(in[j]);
            bad |= !(fabsf(a) < 65504.f) || !(fabsf(b) < 65504.f);
            o[j] = pack_f16x2(a, b);
        }
        if (bad) set_error(err, SMOE_DEV_RANGE);
        reinterpret_cast<uint4 *>(xh)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__device__ __forceinline__ void umma(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte cp.async into shared memory; src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + __expf(-v)); }

// ---------------------------------------------------------------- bucketing

__global__ void __launch_bounds__(256) bucket_count_kernel(const PrefillParams p)
{
    __shared__ int cnt[1024];
    const int c = blockIdx.x;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int t0 = c * kBucketTok, t1 = min(p.T, t0 + kBucketTok);
    for (int q = t0 * p.k + threadIdx.x; q < t1 * p.k; q += blockDim.x) {
        const int e = p.ids[q];
        if (e >= 0 && e < p.E) atomicAdd(&cnt[e], 1);
        else set_error(p.err, SMOE_DEV_BAD_EXPERT);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) p.counts[size_t(c) * p.E + e] = cnt[e];
}

// One CTA: per-expert chunk prefixes, expert offsets, and the tile list.
__global__ void __launch_bounds__(1024) bucket_scan_kernel(const PrefillParams p)
{
    __shared__ int buf[1024];
    __shared__ int tbuf[1024];
    const int e = threadIdx.x;
    const int nch = (p.T + kBucketTok - 1) / kBucketTok;
    int total = 0;
    if (e < p.E)
        for (int c = 0; c < nch; ++c) {
            const int v = p.counts[size_t(c) * p.E + e];
            p.chunk_base[size_t(c) * p.E + e] = total;
            total += v;
        }
    const int nt = e < p.E ? (total + kPfMaxN - 1) / kPfMaxN : 0;
    buf[e] = e < p.E ? total : 0;
    tbuf[e] = nt;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {       // inclusive scans of totals and tile counts
        const int a = e >= off ? buf[e - off] : 0, b = e >= off ? tbuf[e - off] : 0;
        __syncthreads();
        buf[e] += a;
        tbuf[e] += b;
        __syncthreads();
    }
    const int start = buf[e] - (e < p.E ? total : 0);     // exclusive
    const int tstart = tbuf[e] - nt;
    if (e < p.E) {
        p.offsets[e] = start;
        for (int c = 0; c < nch; ++c) p.chunk_base[size_t(c) * p.E + e] += start;
        for (int i = 0; i < nt; ++i) {
            PfTile tl;
            tl.kind = 0;
            tl.expert = e;
            tl.p0 = start + i * kPfMaxN;
            tl.n = min(kPfMaxN, total - i * kPfMaxN);
            p.tiles[tstart + i] = tl;
        }
    }
    if (e == 0) {
        const int P = buf[1023];
        const int ntr = tbuf[1023];
        p.offsets[p.E] = P;
        const int nts = (p.T + kPfMaxN - 1) / kPfMaxN;
        for (int i = 0; i < nts; ++i) {
            PfTile tl;
            tl.kind = 1;
            tl.expert = -1;
            tl.p0 = i * kPfMaxN;
            tl.n = min(kPfMaxN, p.T - i * kPfMaxN);
            p.tiles[ntr + i] = tl;
        }
        *p.ntiles = ntr + nts;
    }
}

// One warp per chunk: pairs in token order, each to its expert's next slot.
__global__ void __launch_bounds__(32) bucket_scatter_kernel(const PrefillParams p)
{
    __shared__ int base[1024];
    const int c = blockIdx.x, lane = threadIdx.x;
    for (int e = lane; e < p.E; e += 32) base[e] = p.chunk_base[size_t(c) * p.E + e];
    __syncwarp();
    const int t0 = c * kBucketTok, t1 = min(p.T, t0 + kBucketTok);
    for (int t = t0; t < t1; ++t) {
        const int q = t * p.k + lane;
        const bool act = lane < p.k;
        const int e = act ? p.ids[q] : -1;
        const bool ok = act && e >= 0 && e < p.E;
        // lanes naming the same expert take consecutive slots in lane order
        const uint32_t same = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
        const int rank = __popc(same & ((1u << lane) - 1u));
        int pos = -1;
        if (ok) pos = base[e] + rank;
        __syncwarp();
        if (ok && rank == __popc(same) - 1) base[e] = pos + 1;
        if (ok) {
            p.pair_token[pos] = t;
            p.pair_j[pos] = lane;
        }
        if (act) p.pair_pos[q] = pos;
        __syncwarp();
    }
}

// ---------------------------------------------------------- grouped GEMM

// mode 0 gate/up, 1 down, 2 router logits. Tile = blockIdx.x / m_tiles.
__global__ void __launch_bounds__(kPfThreads, 1) grouped_gemm_kernel(const GemmParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPfStages * kPfStageBytes);
    uint64_t *rawfull = bars, *afull = bars + kPfStages, *bfull = bars + 2 * kPfStages, *empty = bars + 3 * kPfStages;
    uint64_t *accfull = bars + 4 * kPfStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4 * kPfStages + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = blockIdx.x / p.m_tiles, mt = blockIdx.x % p.m_tiles;
    PfTile tl;
    if (p.mode == 2) {
        tl.kind = 1;
        tl.expert = -1;
        tl.p0 = nt * kPfMaxN;
        tl.n = min(kPfMaxN, p.T - tl.p0);
    } else {
        if (nt >= *p.ntiles) return;                  // uniform: more tiles were launched than exist
        tl = p.tiles[nt];
    }
    if (tl.n <= 0) return;
    const int n = tl.n, N = (n + 15) & ~15;
    const int K = p.mode == 1 ? p.I : p.H;
    const int nk = K / kPfK;
    const int ngH = p.H / kGroup, ngI = p.I / kGroup;

    const uint8_t *blob = nullptr;
    bool valid = true;
    if (p.mode != 2) {
        if (tl.kind == 1) {
            blob = p.shared_blob;
        } else {
            const int64_t slot = p.table_row[tl.expert];
            if (slot < 0 || slot >= p.n_slots) {
                valid = false;
                set_error(p.err, SMOE_DEV_BAD_SLOT);
            } else {
                blob = p.pool + uint64_t(slot) * p.stride;
            }
        }
    }
    // rows of the B operand / outputs: routed pairs at p0.., shared tokens at P + p0..
    const int rowbase = tl.kind == 1 ? p.P + tl.p0 : tl.p0;

    if (!valid) {                                     // contributes zeros
        if (p.mode == 0) {
            for (int i = tid; i < n * 64; i += kPfThreads)
                p.hbuf[size_t(rowbase + i / 64) * p.I + mt * 64 + i % 64] = 0;
        } else {
            for (int i = tid; i < n * kPfM; i += kPfThreads)
                p.ypair[size_t(rowbase + i / kPfM) * p.H + mt * kPfM + i % kPfM] = 0.f;
        }
        return;
    }

    if (tid == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(&rawfull[s], 1);
            mbar_init(&afull[s], kPfWorkers * 32);
            mbar_init(&bfull[s], kPfWorkers * 32);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accfull, 1);
        fence_mbar_init();
    }
    if (warp == kPfWorkers + 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(tmem_slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == kPfWorkers) {
        // ---- producer: raw int4 atoms (8 row blocks x one group) per stage
        if (lane == 0 && p.mode != 2) {
            const uint64_t pol = policy_evict_first();
            const uint64_t down_off = uint64_t(p.I / 8) * ngH * kAtomBytes;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % kPfStages;
                if (kb >= kPfStages && !mbar_wait(&empty[s], ((kb / kPfStages) - 1) & 1, p.err)) break;
                mbar_arrive_expect_tx(&rawfull[s], 8 * kAtomBytes);
                uint8_t *raw = smem + s * kPfStageBytes;
                for (int a = 0; a < 8; ++a) {
                    const int rb = 8 * mt + a;
                    const uint64_t atom = p.mode == 0 ? uint64_t(rb) * ngH + kb : down_off / kAtomBytes + uint64_t(rb) * ngI + kb;
                    bulk_g2s(raw + a * kAtomBytes, blob + atom * kAtomBytes, kAtomBytes, &rawfull[s], pol);
                }
            }
        }
    } else if (warp == kPfWorkers + 1) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc(N, p.mode == 2);
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % kPfStages;
                const uint32_t par = (kb / kPfStages) & 1;
                if (!mbar_wait(&afull[s], par, p.err) || !mbar_wait(&bfull[s], par, p.err)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint8_t *sa = smem + s * kPfStageBytes + kPfRawBytes;
                const uint8_t *sb = sa + kPfABytes;
                const uint64_t ad = umma_desc(smem_u32(sa)), bd = umma_desc(smem_u32(sb));
#pragma unroll
                for (int k4 = 0; k4 < kPfK / 16; ++k4)
                    umma(tmem, ad + uint64_t(k4 * 2), bd + uint64_t(k4 * 2), idesc, (kb | k4) ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            umma_commit(accfull);
        }
    } else {
        // ---- workers: B rows by cp.async, A by dequantisation (or cp.async for the router)
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kPfStages;
            const uint32_t par = (kb / kPfStages) & 1;
            if (kb >= kPfStages) mbar_wait(&empty[s], par ^ 1, p.err);
            uint8_t *st = smem + s * kPfStageBytes;
            uint8_t *sa = st + kPfRawBytes, *sb = sa + kPfABytes;
            const uint32_t sb_u = smem_u32(sb), sa_u = smem_u32(sa);
            for (int i = tid; i < N * 8; i += kPfWorkers * 32) {
                const int r = i >> 3, c8 = i & 7;
                const int rr = r < n ? r : 0;         // padded rows repeat row 0; their outputs are dropped
                const uint16_t *src;
                if (p.mode == 1) {
                    src = p.hbuf + size_t(rowbase + rr) * p.I + kb * kPfK + c8 * 8;
                } else {
                    const int tok = tl.kind == 1 ? tl.p0 + rr : p.pair_token[tl.p0 + rr];
                    src = p.x + size_t(tok) * p.H + kb * kPfK + c8 * 8;
                }
                cp_async16(sb_u + sw128(r, c8 * 8), src, 16);
            }
            if (p.mode == 2) {                        // A = router rows (row E is the shared-gate vector)
                for (int i = tid; i < kPfM * 8; i += kPfWorkers * 32) {
                    const int r = i >> 3, c8 = i & 7;
                    const int e = mt * kPfM + r;
                    const uint16_t *src = e < p.E ? p.Wr + size_t(e) * p.H : p.ws;
                    cp_async16(sa_u + sw128(r, c8 * 8), src + kb * kPfK + c8 * 8, e <= p.E ? 16u : 0u);
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            if (p.mode != 2) {
                if (!mbar_wait(&rawfull[s], par, p.err)) { /* bounded; continue */ }
                // lane-chunk `tid`: atom a, lane L -> rows (g, g+8) of row block a, 16 columns
                const int a = tid >> 5, L = tid & 31, g = L >> 2, t = L & 3;
                const uint8_t *atom = st + a * kAtomBytes;
                const uint4 q = *reinterpret_cast<const uint4 *>(atom + 16 * L);
                const uint2 sbp = *reinterpret_cast<const uint2 *>(atom + kAtomQBytes + 8 * g);
                const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int half = w & 1, hi = w >> 1;      // column half, row g or g+8
                    const uint32_t sbw = hi ? sbp.y : sbp.x;
                    const float sc = half_bits_to_f32(uint16_t(sbw & 0xffff));
                    const float bp = fmaf(-128.f, sc, half_bits_to_f32(uint16_t(sbw >> 16)));
                    uint32_t o[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t pr = nib_pair(words[w], m);   // (128 + q_even, 128 + q_odd)
                        o[m] = pack_f16x2(fmaf(bf16lo(pr), sc, bp), fmaf(bf16hi(pr), sc, bp));
                    }
                    const int row = 16 * a + g + 8 * hi;
                    *reinterpret_cast<uint4 *>(sa + sw128(row, 16 * t + 8 * half)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_async_smem();
                mbar_arrive(&afull[s]);
            }
            if (kb >= 1) {                            // the previous stage's cp.async data is complete
                asm volatile("cp.async.wait_group 1;" ::: "memory");
                fence_async_smem();
                const int sp = (kb - 1) % kPfStages;
                if (p.mode == 2) mbar_arrive(&afull[sp]);
                mbar_arrive(&bfull[sp]);
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        fence_async_smem();
        if (p.mode == 2) mbar_arrive(&afull[(nk - 1) % kPfStages]);
        mbar_arrive(&bfull[(nk - 1) % kPfStages]);

        // ---- epilogue: TMEM lanes = tile rows, columns = tokens of the tile
        mbar_wait(accfull, 0, p.err);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int q = warp & 3, colhalf = warp >> 2;
        const int r = 32 * q + lane;
        for (int c16 = colhalf; c16 < N / 16; c16 += 2) {
            uint32_t v[16];
            tmem_ld16(tmem + (uint32_t(32 * q) << 16) + uint32_t(c16 * 16), v);
            if (p.mode == 0) {
                const bool gate_row = (lane & 8) == 0;
                const int inter = 64 * mt + 8 * (r >> 4) + (r & 7);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float gv = __uint_as_float(v[j]);
                    const float uv = __shfl_xor_sync(0xffffffffu, gv, 8);
                    const int c = c16 * 16 + j;
                    if (gate_row && c < n) {
                        const float h = silu_f(gv) * uv;
                        if (!(fabsf(h) < 65504.f)) set_error(p.err, SMOE_DEV_RANGE);
                        p.hbuf[size_t(rowbase + c) * p.I + inter] = f32_to_f16_bits(h);
                    }
                }
            } else if (p.mode == 1) {
                const int R = kPfM * mt + r;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = c16 * 16 + j;
                    if (c < n) {
                        float wt;
                        if (tl.kind == 1) {
                            wt = p.gate[tl.p0 + c];
                        } else {
                            const int pp = tl.p0 + c;
                            wt = p.w[size_t(p.pair_token[pp]) * p.k + p.pair_j[pp]];
                        }
                        p.ypair[size_t(rowbase + c) * p.H + R] = __uint_as_float(v[j]) * wt;
                    }
                }
            } else {
                const int e = kPfM * mt + r;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = c16 * 16 + j;
                    if (c < n && e <= p.E) p.logits[size_t(tl.p0 + c) * (p.E + 1) + e] = __uint_as_float(v[j]);
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kPfWorkers + 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
}

// ---------------------------------------------------------------- combine

// out[t] = sum_j ypair[pos(t, j)] (route order) + ypair[P + t] (+ residual).
__global__ void __launch_bounds__(256) combine_kernel(const PrefillParams p)
{
    const int t = blockIdx.y;
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (c >= p.H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < p.k; ++j) {
        const int pos = p.pair_pos[size_t(t) * p.k + j];
        if (pos < 0) continue;
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.ypair + size_t(pos) * p.H + c));
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.ypair + size_t(p.P + t) * p.H + c));
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    if (p.residual) {
        const uint2 r = *reinterpret_cast<const uint2 *>(p.residual + size_t(t) * p.H + c);
        acc.x += bf16lo(r.x); acc.y += bf16hi(r.x); acc.z += bf16lo(r.y); acc.w += bf16hi(r.y);
    }
    *reinterpret_cast<uint2 *>(p.out + size_t(t) * p.H + c) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
}

// ------------------------------------------------------------------ host

cudaError_t prefill_config()
{
    return cudaFuncSetAttribute(grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
}

int prefill_max_tiles(int T, int k, int E) { return (T * k + kPfMaxN - 1) / kPfMaxN + E + (T + kPfMaxN - 1) / kPfMaxN; }

cudaError_t launch_router_gemm(const RouteParams &r, cudaStream_t st)
{
    GemmParams g = {};
    g.mode = 2;
    g.x = r.x;
    g.Wr = r.Wr;
    g.ws = r.ws;
    g.logits = r.logits;
    g.err = r.err;
    g.T = r.T;
    g.H = r.H;
    g.E = r.E;
    g.k = r.k;
    g.m_tiles = (r.E + 1 + kPfM - 1) / kPfM;
    const int ntile = (r.T + kPfMaxN - 1) / kPfMaxN;
    grouped_gemm_kernel<<<ntile * g.m_tiles, kPfThreads, kPfSmem, st>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams &p, const GemmParams &g0, cudaStream_t st, const cudaEvent_t *prof,
                           int nprof)
{
    const int nch = (p.T + kBucketTok - 1) / kBucketTok;
    const long long n8 = (long long)p.T * p.H / 8;
    x_to_half_kernel<<<unsigned(n8 / 256 + 1 < 4096 ? n8 / 256 + 1 : 4096), 256, 0, st>>>(g0.x_bf16, const_cast<uint16_t *>(g0.x), n8, p.err);
    bucket_count_kernel<<<nch, 256, 0, st>>>(p);
    bucket_scan_kernel<<<1, 1024, 0, st>>>(p);
    bucket_scatter_kernel<<<nch, 32, 0, st>>>(p);
    const int maxt = prefill_max_tiles(p.T, p.k, p.E);
    GemmParams g = g0;
    g.mode = 0;
    g.m_tiles = g.I / 64;
    cudaError_t e = prof_record(nprof > 0 ? prof[0] : nullptr, st);
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<<<maxt * g.m_tiles, kPfThreads, kPfSmem, st>>>(g);
    if ((e = prof_record(nprof > 1 ? prof[1] : nullptr, st)) != cudaSuccess) return e;
    g.mode = 1;
    g.m_tiles = p.H / kPfM;
    grouped_gemm_kernel<<<maxt * g.m_tiles, kPfThreads, kPfSmem, st>>>(g);
    if ((e = prof_record(nprof > 2 ? prof[2] : nullptr, st)) != cudaSuccess) return e;
    combine_kernel<<<dim3((p.H / 4 + 255) / 256, p.T), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace smoe
