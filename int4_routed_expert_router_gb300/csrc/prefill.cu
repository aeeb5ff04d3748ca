// prefill.cu -- the token-bucketed path for T > 8 (batched decode, prefill).
//
//   bucketing: a deterministic counting sort of the T*k (token, slot) pairs by
//     expert (per-chunk counts, one scan, an ordered scatter), plus the list of
//     GEMM tiles: per expert, runs of up to 192 of its pairs; the shared
//     expert takes all T tokens;
//   token conversion: x to fp16 in the MMA's K order, one row per token;
//   gate/up GEMM: per tile, 128 weight rows (64 gate + 64 up rows, interleaved
//     in blocks of 8 as the blob stores them) x its tokens (at most 192), K = H;
//     the int4 atoms are dequantised to fp16 straight into tensor memory, the
//     tile's token rows are gathered into 128-byte-swizzled shared memory, and
//     tcgen05 tensor cores multiply them (A from TMEM, B from shared memory)
//     into an accumulator in TMEM, 128 K columns per pipeline step (256 for
//     T <= 64, whose tiles are narrower); the epilogue applies SwiGLU and
//     writes h in expert order;
//   down GEMM: per tile, 128 down rows x its pairs, K = I, B = h rows; the
//     epilogue stores each pair's expert output;
//   combine: per token, the k pair outputs times their routing weights in route
//     order, then the shared expert times its gate (and the residual), summed in
//     fp32 and rounded once to bf16.
// The expert GEMMs take fp16 operands (weights s q + b and h keep 11
// significant bits; x converts exactly for |x| < 65504, else the error word is
// set); the same kernel with bf16 router rows and bf16 x computes the router
// logits for large T. Swap-AB: weights take the 128-row M side, tokens the N side,
// so a tile fits an expert's ~160 tokens without padding to 128.
// Pages: the sparse MoE layer (xix.ai article, paragraph on how it works);
// prefill as the slow part on the pages' hardware (paper-digest, Community
// Reactions).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "smoe_dev.cuh"
#include "smoe_internal.h"

namespace smoe {

constexpr int kPfM = 128;          // weight rows per tile
constexpr int kPfK = 64;           // K of one quantisation group (a 128-byte swizzled panel of 16-bit values)
constexpr int kPfMaxN = 256;       // tokens per tile
constexpr int kPfAB = 4;           // router GEMM: A/B operand stages
constexpr int kPfBoxRows = 64;     // B rows per TMA box
constexpr int kPfWorkers = 8;      // warps: A (dequantisation, or router rows)
constexpr int kPfEpi = 8;          // warps: epilogue (two per TMEM lane quadrant)
constexpr int kPfRawWarp = kPfWorkers + kPfEpi;   // bulk copies of the raw atoms
constexpr int kPfBWarp = kPfRawWarp + 1;          // B by TMA boxes (router tokens; the down GEMM's h rows)
constexpr int kPfMma = kPfBWarp + 1;              // tcgen05.mma issuer
constexpr int kPfThreads = (kPfMma + 1) * 32;
constexpr int kPfABytes = kPfM * kPfK * 2;          // 16 KiB
constexpr int kPfBBytes = kPfMaxN * kPfK * 2;       // 32 KiB
constexpr int kPfStageBytes = kPfABytes + kPfBBytes;
constexpr int kPfSmem = kPfAB * kPfStageBytes + 1024 /*align*/ + 512 /*barriers*/;
static_assert(kPfSmem <= 232448, "shared memory per CTA");

// Expert GEMMs (gate/up, down): A (the dequantised weights) lives in tensor
// memory. TMEM columns: Acc accumulators of MaxN columns, then Stg A stages of
// Ks / 2 columns (128 rows x Ks fp16 K values). Shared memory holds only the
// B stages and the raw atoms.
constexpr int kXMaxN = 192;        // tokens per expert tile (the bucketing's bound)
constexpr int kXRaw = 16;          // raw atom slots
constexpr int kXAcc = 2;           // accumulator buffers in TMEM (the epilogue of a tile overlaps the next)
constexpr int kXGatherW0 = 19;     // gate/up: warps 19 .. 22 gather the B rows (cp.async)
constexpr int kXGatherWarps = 4;
constexpr int kXThreads = (kXGatherW0 + kXGatherWarps) * 32;

// Ring shape of the expert GEMMs: MAXN tokens per tile (the accumulators' and
// B stages' width), STG operand stages (A in TMEM and B in shared memory, one
// barrier pair each), GDEPTH K steps a gather thread keeps in flight past the
// one it signals (at most STG - 2, or the gather and the MMAs take turns).
// Wide takes any tile. Narrow serves T <= kXNarrowT, where a tile holds at most
// T tokens: its narrower accumulators leave tensor memory for 8 stages, so the
// gathered rows (about a microsecond from request to landing) are asked for 6
// steps ahead instead of 2.
// KS: K columns per step (64 or 128; a step's B stage is KS / 64 panels of
// MAXN rows x 128 bytes, its A stage KS / 2 tensor-memory columns).
template <int MAXN, int STG, int GDEPTH, int KS = 64, int ACC = kXAcc>
struct XCfg {
    static constexpr int MaxN = MAXN, Stg = STG, GDepth = GDEPTH, Ks = KS, Acc = ACC;
    static constexpr int Panels = KS / 64;                             // 64-column K panels per step
    static constexpr int PanelBytes = MAXN * 128;
    static constexpr int BBytes = Panels * PanelBytes;                 // one B stage
    static constexpr uint32_t ACol0 = ACC * MAXN;                      // first A column
    static constexpr int ACols = KS / 2;                               // A stage columns
    static constexpr int GChunks = KS / 8;                             // 16-byte pieces of a row per step
    static constexpr int GRStep = kXGatherWarps * 32 / GChunks;        // rows between one thread's pieces
    static constexpr int GRows = MAXN / GRStep;                        // rows per gather thread per K step
    static_assert(ACol0 + STG * ACols <= 512, "TMEM columns");
    static_assert(GDEPTH <= STG - 2 && MAXN % 64 == 0 && (KS == 64 || KS == 128 || KS == 256) && ACC >= 1,
                  "ring shape");
};
// The shapes in use. A step's fixed cost (the operand ring's waits and
// arrivals, the gather's round trip, the MMA thread's commit) is paid per K
// step, so the largest K step that tensor and shared memory allow wins:
// wide tiles take 128 columns per step with one accumulator (three stages),
// narrow ones 256 (their accumulators are a third as wide). K (H for gate/up,
// I for down) must be a multiple of the step; I that is not falls back to
// 64-column steps for the down GEMM. The wide down GEMM loads B by TMA (no
// gather to run ahead), so it trades the third stage for a second accumulator
// and its epilogue overlaps the next tile's MMAs.
using XWide = XCfg<kXMaxN, 3, 1, 128, 1>;
using XWideDown = XCfg<kXMaxN, 2, 0, 128, 2>;
using XWide64 = XCfg<kXMaxN, 4, 2, 64, 2>;
using XNarrow = XCfg<64, 3, 1, 256>;
using XNarrow64 = XCfg<64, 8, 6, 64>;
constexpr int kXNarrowT = 64;

// The raw-atom ring of the expert GEMMs for BITS-bit experts: bytes per atom,
// bytes per K step (8 atoms per 64 columns), slots (the K lead of 16 or 12
// 64-column steps where shared memory allows, else what fits), and the CTA's
// shared memory.
template <int BITS, typename CFG>
struct XRaw {
    static constexpr int AB = BITS == 8 ? kAtom8Bytes : kAtomBytes;
    static constexpr int Step = 8 * AB * CFG::Panels;
    static constexpr int Budget = 232448 - 2048 - CFG::Stg * CFG::BBytes;
    static constexpr int Want = (BITS == 8 ? 12 : kXRaw) / CFG::Panels;
    static constexpr int Slots = Want * Step <= Budget ? Want : Budget / Step;
    static constexpr int Smem = CFG::Stg * CFG::BBytes + Slots * Step + 1024 /*align*/ + 1024 /*barriers*/;
    static_assert(Slots >= 2 && Smem <= 232448, "shared memory per CTA");
};

// The kernel and its shared memory for one launch.
struct XLaunch {
    void (*kern)(const GemmParams, const CUtensorMap, const CUtensorMap, const CUtensorMap);
    int smem;
};

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

// tmem_ld32: 32 lanes x 32 consecutive 32-bit columns into 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
                   "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
                   "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tmem_ld16x256x8: 16 lanes x 64 columns; thread 4 g + t gets registers 4 r ..
// 4 r + 3 = (lane g, column 8 r + 2 t), (g, 8 r + 2 t + 1), (g + 8, 8 r + 2 t),
// (g + 8, 8 r + 2 t + 1), r = 0 .. 7 (lanes relative to the address's lane).
__device__ __forceinline__ void tmem_ld16x256x8(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
                   "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
                   "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void umma(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// tcgen05.mma with A read from tensor memory (a_tmem: column of the stage,
// lane 0) and B from a shared-memory descriptor.
__device__ __forceinline__ void umma_ts(uint32_t tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// 16 lanes x 32 columns from registers: thread 4g + t's registers 4r .. 4r + 3
// land at (lane g, column 8r + 2t), (g, 8r + 2t + 1), (g + 8, 8r + 2t),
// (g + 8, 8r + 2t + 1) of the 16-lane block at taddr.
__device__ __forceinline__ void tmem_st16x256x4(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                   "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

// K order inside a 64-column group as the expert GEMMs see it: MMA position
// 16 a + 4 b + c holds column 16 b + 4 a + c (the 4-column blocks transposed),
// which is the order in which a thread's atom fragment meets the 16x256b
// tensor-memory store. The map is its own inverse; B rows (x and h) are stored
// in the same order so the products pair up.
__device__ __forceinline__ int perm64(int c) { return ((c & 12) << 2) | ((c >> 2) & 12) | (c & 3); }

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// 16-byte cp.async into shared memory; src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ float silu_f(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// ---------------------------------------------------------------- bucketing
constexpr int kBucketSmallT = 256;   // up to this T: one CTA buckets (at most 32 chunks of 8 tokens)

// Dynamic shared memory of bucket_small_kernel's bucketing CTA for E experts.
__host__ __device__ inline int bucket_small_smem(int E) { return (32 * E + 2 * 1024 + kBucketSmallT * 16) * 4; }

// counts and chunk_base are [E][chunks] (chunks of bucket_tok(T) tokens): the
// scan's warps (one per expert) read and write an expert's row coalesced.

__global__ void __launch_bounds__(256) bucket_count_kernel(const PrefillParams p)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    __shared__ int cnt[1024];
    const int c = blockIdx.x, nch = gridDim.x, ct = bucket_tok(p.T);
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int t0 = c * ct, t1 = min(p.T, t0 + ct);
    for (int q = t0 * p.k + threadIdx.x; q < t1 * p.k; q += blockDim.x) {
        const int e = p.ids[q];
        if (e >= 0 && e < p.E) atomicAdd(&cnt[e], 1);
        else set_error(p.err, SMOE_DEV_BAD_EXPERT);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) p.counts[size_t(e) * nch + c] = cnt[e];
}

// Thread e of a 1024-thread CTA (e < E: its expert, with `total` pairs from
// pair row `start` and nt tiles from tile tstart; ntr: all routed tiles):
// the expert's tiles, runs of at most kXMaxN pairs of near-equal size, its
// slot resolved; then the shared expert's runs over T and the tile count.
__device__ void write_tiles(const PrefillParams &p, int e, int total, int nt, int start, int tstart, int ntr)
{
    if (e < p.E) {
        const int64_t slot = p.table_row[e];
        for (int i = 0; i < nt; ++i) {
            PfTile tl;
            tl.kind = 0;
            tl.slot = (slot < 0 || slot >= p.n_slots) ? -1 : int(slot);
            tl.p0 = start + int((int64_t(i) * total) / nt);               // runs of near-equal size
            tl.n = int((int64_t(i + 1) * total) / nt) - int((int64_t(i) * total) / nt);
            p.tiles[tstart + i] = tl;
        }
    }
    const int nts = (p.T + kXMaxN - 1) / kXMaxN;
    for (int i = e; i < nts; i += blockDim.x) {       // the shared expert: runs of near-equal size over T
        PfTile tl;
        tl.kind = 1;
        tl.slot = 0;
        tl.p0 = int((int64_t(i) * p.T) / nts);
        tl.n = int((int64_t(i + 1) * p.T) / nts) - tl.p0;
        p.tiles[ntr + i] = tl;
    }
    if (e == 0) *p.ntiles = ntr + nts;
}

// Inclusive scans over the 1024 threads of a CTA of a[] and b[] (in place).
__device__ void block_scan2(int *a, int *b)
{
    const int e = threadIdx.x;
    for (int off = 1; off < 1024; off <<= 1) {
        const int x = e >= off ? a[e - off] : 0, y = e >= off ? b[e - off] : 0;
        __syncthreads();
        a[e] += x;
        b[e] += y;
        __syncthreads();
    }
}

// One warp per expert: chunk_base[e][c] = pairs of expert e in chunks before
// c (warp scans of 32 chunks at a time), the expert's total into offsets[e].
// The last CTA to finish (arrival ticket) turns the totals into the expert
// offsets (exclusive prefix) and writes the tile list: per expert, runs of at
// most kXMaxN pairs of near-equal size; then the shared expert's runs over T.
__global__ void __launch_bounds__(1024) bucket_scan_kernel(const PrefillParams p)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    __shared__ int buf[1024];
    __shared__ int tbuf[1024];
    __shared__ int last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (p.T + bucket_tok(p.T) - 1) / bucket_tok(p.T);
    const int ew = blockIdx.x * 32 + warp;
    if (ew < p.E) {
        const int *row = p.counts + size_t(ew) * nch;
        int *brow = p.chunk_base + size_t(ew) * nch;
        int carry = 0;
        for (int c0 = 0; c0 < nch; c0 += 32) {
            const int c = c0 + lane;
            const int v = c < nch ? row[c] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (c < nch) brow[c] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            p.offsets[ew] = carry;
            __threadfence();
        }
    }
    __syncthreads();
    if (tid == 0) last = ticket_add(p.ticket, 1u) == gridDim.x - 1 ? 1 : 0;
    __syncthreads();
    if (!last) return;
    const int e = tid;
    const int total = e < p.E ? __ldcg(p.offsets + e) : 0;
    const int nt = (total + kXMaxN - 1) / kXMaxN;
    buf[e] = total;
    tbuf[e] = nt;
    __syncthreads();
    block_scan2(buf, tbuf);                           // inclusive scans of totals and tile counts
    const int start = buf[e] - total;                 // exclusive
    if (e < p.E) p.offsets[e] = start;                // the scatter adds it to the chunk prefixes
    write_tiles(p, e, total, nt, start, tbuf[e] - nt, tbuf[1023]);
    if (e == 0) {
        p.offsets[p.E] = buf[1023];
        atomicExch(p.ticket, 0u);                     // ready for the next call
    }
}

// One warp per chunk: pairs in token order, each to its expert's next slot,
// with its token and routing weight. The chunk's ids are staged in shared
// memory first so the ordered loop only touches shared memory.
__global__ void __launch_bounds__(32) bucket_scatter_kernel(const PrefillParams p)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    __shared__ int base[1024];
    __shared__ int ids_s[kBucketTok * 16];
    const int c = blockIdx.x, nch = gridDim.x, lane = threadIdx.x;
    for (int e = lane; e < p.E; e += 32) base[e] = p.offsets[e] + p.chunk_base[size_t(e) * nch + c];
    const int ct = bucket_tok(p.T), t0 = c * ct, t1 = min(p.T, t0 + ct);
    for (int q = t0 * p.k + lane; q < t1 * p.k; q += 32) ids_s[q - t0 * p.k] = p.ids[q];
    __syncwarp();
    for (int t = t0; t < t1; ++t) {
        const int q = t * p.k + lane;
        const bool act = lane < p.k;
        const int e = act ? ids_s[q - t0 * p.k] : -1;
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
        }
        if (act) p.pair_pos[q] = pos;
        __syncwarp();
    }
}

// ------------------------------------------------------ token conversion
// One warp per token t: xt[t] = fp16(x[t]) with the columns in the expert
// GEMMs' K order (perm64 inside each 64-column group); the gate/up GEMM gathers
// its B rows from xt by token. fp16 is exact for |x| < 65504 (subnormal below
// 2^-14, an absolute error under 3e-8); larger values set the error word.
__device__ void convert_x_token(const GemmParams &g, int tok, int lane)
{
    const uint4 *src = reinterpret_cast<const uint4 *>(g.x_bf16 + size_t(tok) * g.H);
    uint2 *dst2 = reinterpret_cast<uint2 *>(const_cast<uint16_t *>(g.x) + size_t(tok) * g.H);
    bool bad = false;
    for (int i = lane; i < g.H / 8; i += 32) {
        const uint4 v = __ldg(src + i);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = bf16lo(in[j]), b = bf16hi(in[j]);
            bad |= !(fabsf(a) < 65504.f) || !(fabsf(b) < 65504.f);
            o[j] = pack_f16x2(a, b);
        }
        // columns 8 i .. 8 i + 7 are two 4-column blocks; each goes to its permuted place
        const int c0 = 8 * i, base = c0 & ~63;
        dst2[(base + perm64(c0 & 63)) / 4] = make_uint2(o[0], o[1]);
        dst2[(base + perm64((c0 & 63) + 4)) / 4] = make_uint2(o[2], o[3]);
    }
    if (bad) set_error(g.err, SMOE_DEV_RANGE);
}

__global__ void __launch_bounds__(256) convert_x_kernel(const GemmParams g)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    const int tok = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (tok < g.T) convert_x_token(g, tok, lane);
}

// -------------------------------------------- bucketing of a small batch
// T <= kBucketSmallT (chunks of bucket_tok(T) = 8 tokens, at most 32): CTA 0
// runs the three bucketing steps above in shared memory, warp c taking chunk
// c, with the same results (pairs by expert, then by token; the same tile
// list); the other CTAs convert x, one warp per token. A small batch then
// costs one launch instead of four, each of which was mostly launch and
// serial latency at T = 64.
__global__ void __launch_bounds__(1024) bucket_small_kernel(const PrefillParams p, const GemmParams g)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (blockIdx.x > 0) {
        const int tok = (int(blockIdx.x) - 1) * 32 + warp;
        if (tok < g.T) convert_x_token(g, tok, lane);
        return;
    }
    extern __shared__ int sm[];
    const int E = p.E, k = p.k, ct = bucket_tok(p.T), nch = (p.T + ct - 1) / ct;
    int *cnt = sm;                                // [32 chunks][E]: counts, then the chunk's next slot per expert
    int *buf = sm + 32 * E, *tbuf = buf + 1024;
    int *ids_s = tbuf + 1024;                     // [T * k] (k <= 16): the batch's expert ids
    for (int i = tid; i < 32 * E; i += 1024) cnt[i] = 0;
    for (int q = tid; q < p.T * k; q += 1024) ids_s[q] = p.ids[q];
    __syncthreads();
    if (warp < nch) {
        const int t0 = warp * ct, t1 = min(p.T, t0 + ct);
        for (int q = t0 * k + lane; q < t1 * k; q += 32) {
            const int e = ids_s[q];
            if (e >= 0 && e < E) atomicAdd(&cnt[warp * E + e], 1);
            else set_error(p.err, SMOE_DEV_BAD_EXPERT);
        }
    }
    __syncthreads();
    const int e = tid;
    int total = 0;
    if (e < E)
        for (int c = 0; c < nch; ++c) {            // chunk prefixes of expert e
            const int v = cnt[c * E + e];
            cnt[c * E + e] = total;
            total += v;
        }
    const int nt = (total + kXMaxN - 1) / kXMaxN;
    buf[e] = total;
    tbuf[e] = nt;
    __syncthreads();
    block_scan2(buf, tbuf);
    const int start = buf[e] - total;
    write_tiles(p, e, total, nt, start, tbuf[e] - nt, tbuf[1023]);
    if (e < E)
        for (int c = 0; c < nch; ++c) cnt[c * E + e] += start;
    __syncthreads();
    if (warp < nch) {                             // warp c: chunk c's pairs in token order
        int *base = cnt + warp * E;
        const int t0 = warp * ct, t1 = min(p.T, t0 + ct);
        for (int t = t0; t < t1; ++t) {
            const int q = t * k + lane;
            const bool act = lane < k;
            const int ex = act ? ids_s[q] : -1;
            const bool ok = act && ex >= 0 && ex < E;
            // lanes naming the same expert take consecutive slots in lane order
            const uint32_t same = __match_any_sync(0xffffffffu, ok ? ex : -1 - lane);
            const int rank = __popc(same & ((1u << lane) - 1u));
            int pos = -1;
            if (ok) pos = base[ex] + rank;
            __syncwarp();
            if (ok && rank == __popc(same) - 1) base[ex] = pos + 1;
            if (ok) p.pair_token[pos] = t;
            if (act) p.pair_pos[q] = pos;
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------- grouped GEMM

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// fp16x2 (q_even, q_odd) of nibble pair m of a blob word: 0x6400 is 1024.0 in
// fp16, whose unit in the last place is 1, so OR-ing the nibble in gives
// 1024 + q and subtracting 1024 is exact.
__device__ __forceinline__ uint32_t nib_pair_f16(uint32_t w, int m)
{
    uint32_t r;
    const uint32_t v = w >> (4 * m);
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x64006400u));
    return hsub2(r, 0x64006400u);
}

// fp16x2 (q_even, q_odd) of value pair m of an 8-bit atom's two nibble planes
// (wl: the low nibbles, wh: the high nibbles, each in the 4-bit word layout):
// 1024 + lo + 16 hi is exact in fp16 for q <= 255, and subtracting 1024 too.
__device__ __forceinline__ uint32_t byte_pair_f16(uint32_t wl, uint32_t wh, int m)
{
    const uint32_t lo = (wl >> (4 * m)) & 0x000F000Fu, hi = (wh >> (4 * m)) & 0x000F000Fu;
    return hsub2(lo | (hi << 4) | 0x64006400u, 0x64006400u);
}

// Bounded wait for the persistent GEMM: gives up after kWaitLimitNs of
// global time, and once any wait of the CTA has given up (*abort set) every
// later wait returns at once, so a failed CTA drains in bounded time.
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, int32_t *err, volatile int *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_error(err, SMOE_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// pf_wait that first polls without sleeping (the phase is usually complete
// already, and a non-blocking test returns sooner than a suspending try).
__device__ __forceinline__ bool pf_wait_fast(uint64_t *bar, uint32_t parity, int32_t *err, volatile int *abort)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok ? true : pf_wait(bar, parity, err, abort);
}

struct TileInfo {
    int n, N, rowbase, p0, kind;
    int slot;              // pool slot of the tile's expert (0 for the shared expert)
    bool valid;
};

__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, int tile)
{
    TileInfo t;
    PfTile tl;
    if (p.mode == 2) {
        tl.kind = 1;
        tl.slot = 0;
        tl.p0 = tile * kPfMaxN;
        tl.n = min(kPfMaxN, p.T - tl.p0);
    } else {
        tl = p.tiles[tile];
    }
    t.n = tl.n;
    t.N = (tl.n + 15) & ~15;
    t.p0 = tl.p0;
    t.kind = tl.kind;
    t.rowbase = tl.kind == 1 ? p.P + tl.p0 : tl.p0;   // rows of B / outputs: pairs, then shared tokens
    t.slot = tl.slot;
    t.valid = p.mode == 2 || tl.slot >= 0;
    return t;
}

// TMA load of a box (64 columns x kPfBoxRows rows) of a 2-D tensor map at
// (column col, row row) into shared memory, 128-byte swizzled.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int col, int row, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(col), "r"(row), "r"(smem_u32(bar))
                 : "memory");
}

// The raw 8-bit atoms of one K step (8 row blocks x one group, 8704 bytes) as
// one box {136 words, 2 halves, 8 row blocks, 1 slot} of the 4-D map
// [slot][row block][group x 2 halves][136 words]: a 1088-byte atom is 272
// words, more than a box dimension may hold, so each atom is two halves.
__device__ __forceinline__ void tma_raw8(uint32_t dst, const CUtensorMap *map, int kb, int mt, int slot, uint64_t *bar,
                                         uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
                 ::"r"(dst), "l"(map), "r"(0), "r"(2 * kb), "r"(8 * mt), "r"(slot), "r"(smem_u32(bar)), "l"(policy)
                 : "memory");
}

// The raw atoms of one K step: 8 row blocks (8 mt .. 8 mt + 7) x one group,
// one box {144 words, 8 row blocks, 1 slot} of the pool's 3-D tensor map
// [slot][row block][group x 144 words] (no swizzle), 4608 bytes.
__device__ __forceinline__ void tma_raw(uint32_t dst, const CUtensorMap *map, int kb, int mt, int slot, uint64_t *bar,
                                        uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%2, %3, %4}], [%5], %6;"
                 ::"r"(dst), "l"(map), "r"(kb * (kAtomBytes / 4)), "r"(8 * mt), "r"(slot), "r"(smem_u32(bar)),
                   "l"(policy)
                 : "memory");
}

// Router logits for large T on tensor cores: logits[t][e] = W_r[e] . x[t]
// for e < E, bf16 operands, fp32 accumulation (the shared-gate logit is one
// warp dot per token in the top-k kernel).
// Persistent: CTA b handles tiles b, b + grid, ... (tile = 256 tokens x 128
// router rows); roles: 8 warps copy the router rows into A stages
// (cp.async, one step ahead), one warp loads the tokens (B) with TMA, one
// issues the MMAs into a double-buffered TMEM accumulator, 8 warps store the
// logits.
__global__ void __launch_bounds__(kPfThreads, 1) router_gemm_kernel(const GemmParams p,
                                                                    const __grid_constant__ CUtensorMap bmap)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ab = smem;                                           // kPfAB x (A 16 KiB | B 32 KiB)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPfAB * kPfStageBytes);
    uint64_t *afull = bars, *bfull = afull + kPfAB, *empty = bfull + kPfAB;
    uint64_t *accfull = empty + kPfAB, *accempty = accfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accempty + 2);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (p.T + kPfMaxN - 1) / kPfMaxN * p.m_tiles;
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;
    if (my_tiles == 0) return;                                    // uniform
    const int nk = p.H / kPfK;
    const int total = my_tiles * nk;
    auto tile_of = [&](int i) { return int(blockIdx.x) + i * int(gridDim.x); };

    if (tid == 0) {
        for (int s = 0; s < kPfAB; ++s) {
            mbar_init(&afull[s], kPfWorkers * 32);
            mbar_init(&bfull[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], kPfEpi * 32);
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kPfMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == kPfBWarp) {
        // ---- B: tokens p0 .. p0 + N - 1 in boxes of kPfBoxRows rows
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&bmap) : "memory");
            TileInfo ti;
            int issued = 0;
            for (int gk = 0; gk < total; ++gk) {
                const int i = gk / nk, kb = gk % nk, s = gk % kPfAB;
                if (kb == 0) ti = tile_info(p, tile_of(i) / p.m_tiles);
                const int nbox = (ti.N + kPfBoxRows - 1) / kPfBoxRows;
                if (gk >= kPfAB && !pf_wait(&empty[s], ((gk / kPfAB) - 1) & 1, p.err, abort)) break;
                mbar_arrive_expect_tx(&bfull[s], uint32_t(nbox) * kPfBoxRows * (kPfK * 2));
                const uint32_t dst = smem_u32(ab + s * kPfStageBytes + kPfABytes);
                for (int j = 0; j < nbox; ++j)
                    tma_load_2d(dst + j * (kPfBoxRows * kPfK * 2), &bmap, kb * kPfK, ti.rowbase + j * kPfBoxRows, &bfull[s]);
                ++issued;
            }
            // the last copy into each stage lands before the CTA can exit (also after an abort)
            for (int g2 = issued - 1; g2 >= 0 && g2 >= issued - kPfAB; --g2)
                mbar_wait(&bfull[g2 % kPfAB], (g2 / kPfAB) & 1, p.err);
        }
    } else if (warp == kPfMma) {
        // ---- MMA issuer: tile i accumulates in TMEM buffer i % 2 (256 columns each)
        if (lane == 0) {
            uint32_t idesc = 0;
            for (int gk = 0; gk < total; ++gk) {
                const int i = gk / nk, kb = gk % nk, s = gk % kPfAB, b = i & 1;
                if (kb == 0) {
                    idesc = umma_idesc(tile_info(p, tile_of(i) / p.m_tiles).N, true);
                    if (i >= 2) pf_wait(&accempty[b], ((i / 2) - 1) & 1, p.err, abort);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                }
                const uint32_t par = (gk / kPfAB) & 1;
                pf_wait(&afull[s], par, p.err, abort);
                pf_wait(&bfull[s], par, p.err, abort);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint8_t *sa = ab + s * kPfStageBytes, *sb = sa + kPfABytes;
                const uint64_t ad = umma_desc(smem_u32(sa)), bd = umma_desc(smem_u32(sb));
                const uint32_t acc_t = tmem + uint32_t(b * 256);
#pragma unroll
                for (int k4 = 0; k4 < kPfK / 16; ++k4)
                    umma(acc_t, ad + uint64_t(k4 * 2), bd + uint64_t(k4 * 2), idesc, (kb | k4) ? 1u : 0u);
                umma_commit(&empty[s]);
                if (kb == nk - 1) umma_commit(&accfull[b]);
            }
            mbar_wait(&accfull[(my_tiles - 1) & 1], ((my_tiles - 1) / 2) & 1, p.err);
        }
    } else if (warp < kPfWorkers) {
        // ---- A = router rows (rows past E zero), one step ahead
        auto issue_a = [&](int gi) {
            if (gi < total) {
                const int i = gi / nk, kb = gi % nk, s = gi % kPfAB;
                if (gi >= kPfAB) pf_wait(&empty[s], ((gi / kPfAB) - 1) & 1, p.err, abort);
                const int mt = tile_of(i) % p.m_tiles;
                const uint32_t sa_u = smem_u32(ab + s * kPfStageBytes);
                for (int q = tid; q < kPfM * 8; q += kPfWorkers * 32) {
                    const int r = q >> 3, c8 = q & 7;
                    const int e = mt * kPfM + r;
                    const uint16_t *src = p.Wr + size_t(e < p.E ? e : 0) * p.H;
                    cp_async16(sa_u + sw128(r, c8 * 8), src + kb * kPfK + c8 * 8, e < p.E ? 16u : 0u);
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");   // one group per step, even if empty
        };
        issue_a(0);
        for (int gk = 0; gk < total; ++gk) {
            issue_a(gk + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");  // this step's rows have landed
            fence_async_smem();
            mbar_arrive(&afull[gk % kPfAB]);
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else if (warp < kPfWorkers + kPfEpi) {
        // ---- epilogue warps: TMEM lanes 32q..32q+31 (q = e % 4) = router rows,
        // column chunks of 32 tokens j = 2u + e / 4
        const int e = warp - kPfWorkers, q = e & 3, half = e >> 2;
        const int r = 32 * q + lane;
        for (int i = 0; i < my_tiles; ++i) {
            const int b = i & 1;
            const TileInfo ti = tile_info(p, tile_of(i) / p.m_tiles);
            const int ex = kPfM * (tile_of(i) % p.m_tiles) + r;
            pf_wait(&accfull[b], (i / 2) & 1, p.err, abort);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = 2 * u + half;
                if (32 * j < ti.N) {                      // uniform over the warp
                    uint32_t v[32];
                    tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(b * 256 + 32 * j), v);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int c = 32 * j + jj;
                        if (c < ti.n && ex < p.E) p.logits[size_t(ti.p0 + c) * (p.E + 1) + ex] = __uint_as_float(v[jj]);
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            mbar_arrive(&accempty[b]);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kPfMma)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

// Epilogue of the expert GEMMs: warp w reads TMEM lanes 32 (w % 4) .. + 31
// (tile rows; a warp may only access its own lane quadrant).
// Gate/up: 8 warps, 2 per quadrant, each the 16 lanes of 8 units (rows g:
// gate, g + 8: up) in chunks of 64 tokens, loaded so that a thread holds both
// rows of its unit; h = silu(gate) * up, and units g, g + 1 (adjacent columns of
// h in the down GEMM's K order) share a 4-byte store.
// Down: 12 warps, 3 per quadrant, chunks of 32 tokens; each pair's fp16
// output, two rows per 4-byte store (neighbouring lanes swap halves).
template <int MAXN, int ACC, typename TileOf>
__device__ __forceinline__ void epilogue(const GemmParams &p, uint32_t tmem, uint64_t *accfull, uint64_t *accempty,
                                         volatile int *abort, int warp, int lane, int my_tiles, TileOf tile_of)
{
    const int q = warp & 3;
    const int h = warp >= kXGatherW0 ? 2 : (warp - kPfWorkers) >> 2;   // warp within its quadrant
    uint32_t ymax = 0;                                            // largest |fp16| bits stored, per half
    TileInfo tnext = tile_info(p, tile_of(0) / p.m_tiles);
    for (int i = 0; i < my_tiles; ++i) {
        const int b = i % ACC;
        const TileInfo ti = tnext;
        const int mt = tile_of(i) % p.m_tiles;
        if (i + 1 < my_tiles) tnext = tile_info(p, tile_of(i + 1) / p.m_tiles);
        pf_wait(&accfull[b], (i / ACC) & 1, p.err, abort);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (!ti.valid) set_error(p.err, SMOE_DEV_BAD_SLOT);       // and the tile's outputs are zeros
        if (p.mode == 0) {
            // units 8 (2 q + h) + g, g = lane / 4: h of unit g for tokens c0, c0 + 1
            // (c0 = 64 cc + 8 r + 2 t, t = lane % 4); the even unit of a pair stores
            // both units' h of token c0, the odd one those of token c0 + 1
            const int g = lane >> 2, t = lane & 3, godd = g & 1;
            const int inter = 64 * mt + 8 * (2 * q + h) + (g & ~1);
            const int hcol = (inter & ~63) | perm64(inter & 63);        // units g & ~1, (g & ~1) + 1
            const uint32_t sel = godd ? 0x3276u : 0x5410u;
            for (int cc = 0; 64 * cc < ti.N; ++cc) {                    // uniform over the warp
                uint32_t v[32];
                tmem_ld16x256x8(tmem + (uint32_t(32 * q + 16 * h) << 16) + uint32_t(b * MAXN + 64 * cc), v);
                const int c0 = 64 * cc + 2 * t + godd;                  // this thread's token, + 8 r
                uint32_t *hp = reinterpret_cast<uint32_t *>(p.hbuf + size_t(ti.rowbase + c0) * p.I + hcol);
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const float ha = silu_f(__uint_as_float(v[4 * rr])) * __uint_as_float(v[4 * rr + 2]);
                    const float hb = silu_f(__uint_as_float(v[4 * rr + 1])) * __uint_as_float(v[4 * rr + 3]);
                    const uint32_t h2 = pack_f16x2(ha, hb);
                    const uint32_t nb = __shfl_xor_sync(0xffffffffu, h2, 4);
                    const uint32_t o = ti.valid ? __byte_perm(h2, nb, sel) : 0u;
                    if (c0 + 8 * rr < ti.n) {
                        ymax = __vmaxu2(ymax, o & 0x7fff7fffu);
                        hp[size_t(8 * rr) * (p.I / 2)] = o;
                    }
                }
            }
        } else {
            // chunks j of 32 tokens; lane = row R of the down projection. Tokens 2 m
            // (even lane) and 2 m + 1 (odd lane) of rows R0, R0 + 1: each lane packs
            // its row's two tokens, swaps with its neighbour, and stores one token
            // of both rows
            const int odd = lane & 1;
            const int R0 = kPfM * mt + 32 * q + lane - odd;
            const uint32_t sel = odd ? 0x3276u : 0x5410u;
            for (int j = h; 32 * j < ti.N; j += 3) {                    // uniform over the warp
                uint32_t v[32];
                tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(b * MAXN + 32 * j), v);
                uint32_t *y = reinterpret_cast<uint32_t *>(p.ypair + size_t(ti.rowbase + 32 * j + odd) * p.H + R0);
                const int nc = ti.n - 32 * j - odd;                     // stored when 2 m < nc
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const uint32_t h2 = pack_f16x2(__uint_as_float(v[2 * m]), __uint_as_float(v[2 * m + 1]));
                    const uint32_t nb = __shfl_xor_sync(0xffffffffu, h2, 1);
                    const uint32_t o = ti.valid ? __byte_perm(h2, nb, sel) : 0u;
                    if (2 * m < nc) {
                        ymax = __vmaxu2(ymax, o & 0x7fff7fffu);
                        y[size_t(2 * m) * (p.H / 2)] = o;
                    }
                }
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        mbar_arrive(&accempty[b]);
    }
    // 0x7bff is 65504, the largest finite fp16; above it: infinities and NaN
    if ((ymax & 0xffffu) >= 0x7bffu || (ymax >> 16) >= 0x7bffu) set_error(p.err, SMOE_DEV_RANGE);
}

// ------------------------------------------------- expert GEMMs, A in TMEM
// Persistent like router_gemm_kernel (tiles b, b + grid, ...; every role walks
// the same K steps) for mode 0 (gate/up, K = H) and mode 1 (down, K = I), but
// the eight dequantising warps write A straight into tensor memory
// (tcgen05.st) and the MMAs read it there, so shared memory carries only the
// raw atoms and B. Roles: warps 0-7 dequantise (warp w writes atom a = 2 (w % 4)
// + w / 4, rows 16 a .. 16 a + 15, inside the lane quadrant w % 4 that the warp
// may access); warps 8-15 run the epilogue; warp 16 streams the raw atoms;
// warp 17 loads B with TMA in the down GEMM; warp 18 issues the MMAs; warps
// 19-22 gather B rows by token in the gate/up GEMM and join the epilogue in
// the down GEMM. A and B of a K step share one stage of a CFG::Stg-deep ring.
template <int BITS, typename CFG>
__global__ void __launch_bounds__(kXThreads, 1) expert_gemm_kernel(const GemmParams p,
                                                                    const __grid_constant__ CUtensorMap bmap,
                                                                    const __grid_constant__ CUtensorMap amap,
                                                                    const __grid_constant__ CUtensorMap amap_shared)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *bst = smem;                                          // CFG::Stg x 24 KiB, 128-byte swizzled rows
    using RW = XRaw<BITS, CFG>;
    uint8_t *raw = smem + CFG::Stg * CFG::BBytes;                       // RW::Slots x RW::Step bytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(raw + RW::Slots * RW::Step);
    uint64_t *rawfull = bars, *rawempty = bars + RW::Slots;
    uint64_t *full = bars + 2 * RW::Slots, *empty = full + CFG::Stg;     // stage s: A (TMEM) + B (smem)
    uint64_t *accfull = empty + CFG::Stg, *accempty = accfull + CFG::Acc;
    uint64_t *bfull = accempty + CFG::Acc;                           // down: B copies of stage s (TMA)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bfull + CFG::Stg);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = *p.ntiles * p.m_tiles;
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;
    if (my_tiles == 0) return;                                    // uniform
    const int nk = (p.mode == 1 ? p.I : p.H) / CFG::Ks;
    const int total = my_tiles * nk;
    auto tile_of = [&](int i) { return int(blockIdx.x) + i * int(gridDim.x); };

    if (tid == 0) {
        for (int r = 0; r < RW::Slots; ++r) {
            mbar_init(&rawfull[r], 1);
            mbar_init(&rawempty[r], kPfWorkers);
        }
        for (int s = 0; s < CFG::Stg; ++s) {
            // the A threads, plus in gate/up the 128 gathering threads (the down
            // GEMM's B copies complete on bfull instead)
            mbar_init(&full[s], kPfWorkers * 32 + (p.mode == 0 ? kXGatherWarps * 32 : 0));
            mbar_init(&empty[s], 1);
            mbar_init(&bfull[s], 1);
        }
        for (int b = 0; b < CFG::Acc; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], (p.mode == 1 ? kPfEpi + kXGatherWarps : kPfEpi) * 32);   // epilogue threads
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kPfMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    // Ring positions advance by one per K step (index and phase bit); a producer
    // waits for the slot's release with the opposite parity, which a fresh
    // barrier passes, so the first round needs no special case.
    // epilogue warps: 8..15, and in the down GEMM also the gather warps (idle there)
    const bool epi_role = (warp >= kPfWorkers && warp < kPfWorkers + kPfEpi) || (p.mode == 1 && warp >= kXGatherW0);
    if (epi_role) {
        epilogue<CFG::MaxN, CFG::Acc>(p, tmem, accfull, accempty, abort, warp, lane, my_tiles, tile_of);
    } else if (warp == kPfRawWarp) {
        // ---- raw atoms (8 row blocks x one group) per K step: one TMA box each
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&amap) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&amap_shared) : "memory");
            const uint64_t pol = policy_evict_first();
            int r = 0, done = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int i = 0; i < my_tiles && ok; ++i) {
                const TileInfo ti = tile_info(p, tile_of(i) / p.m_tiles);
                const int mt = tile_of(i) % p.m_tiles;
                const CUtensorMap *map = ti.kind == 1 ? &amap_shared : &amap;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!pf_wait(&rawempty[r], ph ^ 1u, p.err, abort)) { ok = false; break; }
                    if (ti.valid) {
                        mbar_arrive_expect_tx(&rawfull[r], RW::Step);
#pragma unroll
                        for (int j = 0; j < CFG::Panels; ++j) {            // one box per 64-column group
                            const uint32_t dst = smem_u32(raw + r * RW::Step + j * 8 * RW::AB);
                            if constexpr (BITS == 8) tma_raw8(dst, map, kb * CFG::Panels + j, mt, ti.slot, &rawfull[r], pol);
                            else tma_raw(dst, map, kb * CFG::Panels + j, mt, ti.slot, &rawfull[r], pol);
                        }
                    } else {
                        mbar_arrive(&rawfull[r]);              // nothing to load; the epilogue writes zeros
                    }
                    ++done;
                    if (++r == RW::Slots) { r = 0; ph ^= 1u; }
                }
            }
            // let the last copy into each slot land before the CTA can exit
            for (int g2 = done - 1; g2 >= 0 && g2 >= done - RW::Slots; --g2)
                mbar_wait(&rawfull[g2 % RW::Slots], (g2 / RW::Slots) & 1, p.err);
        }
    } else if (warp >= kXGatherW0) {
        if (p.mode == 0) {
            // ---- B (gate/up): the tile's N token rows of xt, one 16-byte chunk per
            // thread and row: thread g takes chunk g % 8 of rows g / 8 + 16 u. Rows
            // n .. N - 1 repeat row n - 1 (their accumulator columns are never
            // stored). A step is signalled once its copies have landed, CFG::GDepth
            // steps later (cp.async groups), after a proxy fence for the MMA.
            // (KS = 128: thread g takes piece g % 16 of rows g / 16 + 8 u, the
            // pieces 8 .. 15 going to the step's second panel)
            const int gt = tid - kXGatherW0 * 32, c = gt % CFG::GChunks, r0 = gt / CFG::GChunks;
            const int c8 = c & 7, pan = c >> 3;
            // byte offsets: source row u = token row start + piece; destination row
            // r0 + GRStep u at sw128(r0 + GRStep u, 8 c8) of the piece's panel (with
            // KS = 256 the step is 4 rows, so the row's swizzle phase changes with u)
            auto rows_of = [&](const TileInfo &t, uint32_t (&off)[CFG::GRows]) {
#pragma unroll
                for (int u = 0; u < CFG::GRows; ++u) {
                    const int rr = min(r0 + CFG::GRStep * u, t.n - 1);
                    const int tok = t.kind == 1 ? t.p0 + rr : p.pair_token[t.p0 + rr];
                    off[u] = uint32_t(tok) * uint32_t(2 * p.H) + uint32_t(16 * c);   // < 2^32: T <= SMOE_MAX_TOKENS, H <= 2048
                }
            };
            const char *xt = reinterpret_cast<const char *>(p.x);
            const uint32_t dst0 = smem_u32(bst) + uint32_t(pan * CFG::PanelBytes);
            uint32_t cur[CFG::GRows], nxt[CFG::GRows];
            TileInfo tnext = tile_info(p, tile_of(0) / p.m_tiles);
            rows_of(tnext, nxt);
            int sb = 0, sd = 0, issued = 0;
            uint32_t ph = 0;
            for (int i = 0; i < my_tiles; ++i) {
                const TileInfo ti = tnext;
#pragma unroll
                for (int u = 0; u < CFG::GRows; ++u) cur[u] = nxt[u];
                if (i + 1 < my_tiles) {
                    tnext = tile_info(p, tile_of(i + 1) / p.m_tiles);
                    rows_of(tnext, nxt);
                }
                const int urows = (ti.N - r0 + CFG::GRStep - 1) / CFG::GRStep;   // rows r0 + GRStep u < N
                for (int kb = 0; kb < nk; ++kb) {
                    pf_wait(&empty[sb], ph ^ 1u, p.err, abort);
                    const uint32_t dst = dst0 + uint32_t(sb * CFG::BBytes);
                    const char *src = xt + kb * (CFG::Ks * 2);
#pragma unroll
                    for (int u = 0; u < CFG::GRows; ++u)
                        if (u < urows) cp_async16(dst + sw128(r0 + CFG::GRStep * u, 8 * c8), src + cur[u], 16u);
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    if (++sb == CFG::Stg) { sb = 0; ph ^= 1u; }
                    if (++issued > CFG::GDepth) {
                        asm volatile("cp.async.wait_group %0;" ::"n"(CFG::GDepth) : "memory");
                        fence_async_smem();
                        mbar_arrive(&full[sd]);
                        if (++sd == CFG::Stg) sd = 0;
                    }
                }
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            fence_async_smem();
            for (int j = 0; j < min(issued, CFG::GDepth); ++j) {
                mbar_arrive(&full[sd]);
                if (++sd == CFG::Stg) sd = 0;
            }
        }
    } else if (warp == kPfBWarp) {
        if (p.mode == 1 && lane == 0) {
            // ---- B (down): rows rowbase .. rowbase + N - 1 of hbuf, in boxes of kPfBoxRows rows
            asm volatile("prefetch.tensormap [%0];" ::"l"(&bmap) : "memory");
            int sb = 0, issued = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int i = 0; i < my_tiles && ok; ++i) {
                const TileInfo ti = tile_info(p, tile_of(i) / p.m_tiles);
                const int nbox = (ti.N + kPfBoxRows - 1) / kPfBoxRows;
                const uint32_t bytes = uint32_t(CFG::Panels * nbox) * kPfBoxRows * (kPfK * 2);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!pf_wait(&empty[sb], ph ^ 1u, p.err, abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bfull[sb], bytes);
                    const uint32_t dst = smem_u32(bst + sb * CFG::BBytes);
                    for (int pn = 0; pn < CFG::Panels; ++pn)
                        for (int j = 0; j < nbox; ++j)
                            tma_load_2d(dst + pn * CFG::PanelBytes + j * (kPfBoxRows * kPfK * 2), &bmap,
                                        kb * CFG::Ks + pn * kPfK, ti.rowbase + j * kPfBoxRows, &bfull[sb]);
                    ++issued;
                    if (++sb == CFG::Stg) { sb = 0; ph ^= 1u; }
                }
            }
            // the last copy into each stage lands before the CTA can exit (also after an abort)
            for (int g2 = issued - 1; g2 >= 0 && g2 >= issued - CFG::Stg; --g2)
                mbar_wait(&bfull[g2 % CFG::Stg], (g2 / CFG::Stg) & 1, p.err);
        }
    } else if (warp == kPfMma) {
        // ---- MMA issuer: tile i accumulates in TMEM columns (i % 2) * MaxN ..
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int nextN = tile_info(p, tile_of(0) / p.m_tiles).N;
            for (int i = 0; i < my_tiles; ++i) {
                const int b = i % CFG::Acc;
                const uint32_t idesc = umma_idesc(nextN, false);
                if (i + 1 < my_tiles) nextN = tile_info(p, tile_of(i + 1) / p.m_tiles).N;   // used one tile later
                pf_wait(&accempty[b], ((i / CFG::Acc) & 1) ^ 1u, p.err, abort);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t acc_t = tmem + uint32_t(b * CFG::MaxN);
                for (int kb = 0; kb < nk; ++kb) {
                    pf_wait_fast(&full[s], ph, p.err, abort);
                    if (p.mode == 1) pf_wait_fast(&bfull[s], ph, p.err, abort);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t bs = smem_u32(bst + s * CFG::BBytes);
                    const uint32_t a_t = tmem + CFG::ACol0 + uint32_t(CFG::ACols * s);
#pragma unroll
                    for (int k4 = 0; k4 < CFG::Ks / 16; ++k4) {
                        const uint64_t bd = umma_desc(bs + uint32_t((k4 >> 2) * CFG::PanelBytes));
                        umma_ts(acc_t, a_t + uint32_t(8 * k4), bd + uint64_t((k4 & 3) * 2), idesc, (kb | k4) ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);
                    if (++s == CFG::Stg) { s = 0; ph ^= 1u; }
                }
                umma_commit(&accfull[b]);
            }
            // the tensor cores are done with TMEM and shared memory before the CTA exits
            mbar_wait(&accfull[(my_tiles - 1) % CFG::Acc], ((my_tiles - 1) / CFG::Acc) & 1, p.err);
        }
    } else if (warp < kPfWorkers) {
        // ---- A: dequantise atom a of each K step into the fragment order of the
        // 16x256b store: register 4r + {0, 1} = row g, columns 16 t + 4 r .. + 3;
        // 4r + {2, 3} = row g + 8 (MMA K order: perm64)
        const int a = 2 * (warp & 3) + (warp >> 2), g = lane >> 2;
        const uint32_t lane_base = uint32_t(16 * a) << 16;
        int r = 0, sa = 0;
        uint32_t phr = 0, pha = 0;                                // raw ring, operand ring
        for (int gk = 0; gk < total; ++gk) {
            pf_wait(&rawfull[r], phr, p.err, abort);
            uint4 q[CFG::Panels], qh[CFG::Panels];
            uint2 sbp[CFG::Panels];
#pragma unroll
            for (int j = 0; j < CFG::Panels; ++j) {                    // group j of the step
                const uint8_t *atom = raw + r * RW::Step + j * 8 * RW::AB + a * RW::AB;
                q[j] = *reinterpret_cast<const uint4 *>(atom + 16 * lane);          // (low nibbles, 8-bit)
                qh[j] = make_uint4(0u, 0u, 0u, 0u);                                 // 8-bit: the high nibbles
                if constexpr (BITS == 8) qh[j] = *reinterpret_cast<const uint4 *>(atom + kAtomQBytes + 16 * lane);
                sbp[j] = *reinterpret_cast<const uint2 *>(atom + (BITS == 8 ? 2 : 1) * kAtomQBytes + 8 * g);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&rawempty[r]);
            if (++r == RW::Slots) { r = 0; phr ^= 1u; }
            pf_wait(&empty[sa], pha ^ 1u, p.err, abort);
#pragma unroll
            for (int j = 0; j < CFG::Panels; ++j) {
                const uint32_t s0 = __byte_perm(sbp[j].x, 0, 0x1010), b0 = __byte_perm(sbp[j].x, 0, 0x3232);   // row g
                const uint32_t s1 = __byte_perm(sbp[j].y, 0, 0x1010), b1 = __byte_perm(sbp[j].y, 0, 0x3232);   // row g + 8
                const uint32_t wg[2] = {q[j].x, q[j].y}, wh[2] = {q[j].z, q[j].w};
                const uint32_t wg8[2] = {qh[j].x, qh[j].y}, wh8[2] = {qh[j].z, qh[j].w};
                uint32_t v[16];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int m0 = 2 * (rr & 1);
                    if constexpr (BITS == 8) {
                        v[4 * rr + 0] = hfma2(byte_pair_f16(wg[rr >> 1], wg8[rr >> 1], m0), s0, b0);
                        v[4 * rr + 1] = hfma2(byte_pair_f16(wg[rr >> 1], wg8[rr >> 1], m0 + 1), s0, b0);
                        v[4 * rr + 2] = hfma2(byte_pair_f16(wh[rr >> 1], wh8[rr >> 1], m0), s1, b1);
                        v[4 * rr + 3] = hfma2(byte_pair_f16(wh[rr >> 1], wh8[rr >> 1], m0 + 1), s1, b1);
                    } else {
                        v[4 * rr + 0] = hfma2(nib_pair_f16(wg[rr >> 1], m0), s0, b0);
                        v[4 * rr + 1] = hfma2(nib_pair_f16(wg[rr >> 1], m0 + 1), s0, b0);
                        v[4 * rr + 2] = hfma2(nib_pair_f16(wh[rr >> 1], m0), s1, b1);
                        v[4 * rr + 3] = hfma2(nib_pair_f16(wh[rr >> 1], m0 + 1), s1, b1);
                    }
                }
                tmem_st16x256x4(tmem + lane_base + CFG::ACol0 + uint32_t(CFG::ACols * sa + 32 * j), v);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&full[sa]);
            if (++sa == CFG::Stg) { sa = 0; pha ^= 1u; }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kPfMma)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

// ---------------------------------------------------------------- combine

// out[t] = sum_j w[t][j] ypair[pos(t, j)] (route order) + gate[t] ypair[P + t]
// (+ residual), from the fp16 expert outputs, in fp32. Block b: token b / nxb,
// columns 1024 (b % nxb) .. + 1023 (nxb = H / 1024 rounded up; the token
// index is in x, whose range covers SMOE_MAX_TOKENS, unlike y's 65,535).
__global__ void __launch_bounds__(256) combine_kernel(const PrefillParams p)
{
    pdl_wait();                                   // the predecessor's writes are visible
    pdl_trigger();
    const int nxb = (p.H / 4 + 255) / 256;
    const int t = int(blockIdx.x) / nxb;
    const int c = ((int(blockIdx.x) - t * nxb) * blockDim.x + threadIdx.x) * 4;
    if (c >= p.H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](int row, float wt) {
        const uint2 v = __ldcg(reinterpret_cast<const uint2 *>(p.ypair + size_t(row) * p.H + c));
        float2 a, b;
        asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}" : "=f"(a.x), "=f"(a.y) : "r"(v.x));
        asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}" : "=f"(b.x), "=f"(b.y) : "r"(v.y));
        acc.x = fmaf(wt, a.x, acc.x);
        acc.y = fmaf(wt, a.y, acc.y);
        acc.z = fmaf(wt, b.x, acc.z);
        acc.w = fmaf(wt, b.y, acc.w);
    };
    for (int j = 0; j < p.k; ++j) {
        const int pos = p.pair_pos[size_t(t) * p.k + j];
        if (pos >= 0) add(pos, p.w[size_t(t) * p.k + j]);
    }
    add(p.P + t, p.gate[t]);
    if (p.residual) {
        const uint2 r = *reinterpret_cast<const uint2 *>(p.residual + size_t(t) * p.H + c);
        acc.x += bf16lo(r.x); acc.y += bf16hi(r.x); acc.z += bf16lo(r.y); acc.w += bf16hi(r.y);
    }
    *reinterpret_cast<uint2 *>(p.out + size_t(t) * p.H + c) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
}

// ------------------------------------------------------------------ host

template <int BITS, typename CFG>
static XLaunch xlaunch()
{
    return {expert_gemm_kernel<BITS, CFG>, XRaw<BITS, CFG>::Smem};
}

// The shape for one expert GEMM launch: narrow for T <= kXNarrowT, wide above;
// the 64-column variant where K is not a multiple of the shape's step.
static XLaunch pick_gemm(bool b8, bool narrow, bool down, int K)
{
    if (narrow) {
        if (K % XNarrow::Ks == 0) return b8 ? xlaunch<8, XNarrow>() : xlaunch<4, XNarrow>();
        return b8 ? xlaunch<8, XNarrow64>() : xlaunch<4, XNarrow64>();
    }
    if (down && K % XWideDown::Ks == 0) return b8 ? xlaunch<8, XWideDown>() : xlaunch<4, XWideDown>();
    if (K % XWide::Ks == 0) return b8 ? xlaunch<8, XWide>() : xlaunch<4, XWide>();
    return b8 ? xlaunch<8, XWide64>() : xlaunch<4, XWide64>();
}

cudaError_t prefill_config()
{
    cudaError_t e = cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    const XLaunch all[10] = {xlaunch<4, XWide>(), xlaunch<8, XWide>(), xlaunch<4, XWideDown>(), xlaunch<8, XWideDown>(),
                             xlaunch<4, XWide64>(), xlaunch<8, XWide64>(), xlaunch<4, XNarrow>(), xlaunch<8, XNarrow>(),
                             xlaunch<4, XNarrow64>(), xlaunch<8, XNarrow64>()};
    for (const XLaunch &x : all)
        if (e == cudaSuccess) e = cudaFuncSetAttribute(x.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, x.smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bucket_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bucket_small_smem(1024));
    return e;
}

int prefill_max_tiles(int T, int k, int E) { return (T * k + kXMaxN - 1) / kXMaxN + E + (T + kXMaxN - 1) / kXMaxN; }

static int g_num_sms = 0;

static int persistent_grid(int max_tiles)
{
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    return max_tiles < g_num_sms ? (max_tiles > 0 ? max_tiles : 1) : g_num_sms;
}

// Tensor map of a row-major [rows][cols] 16-bit matrix for the B operand:
// box 64 columns x kPfBoxRows rows, 128-byte swizzle (the MMA operand layout);
// rows past the end read as zeros.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return encode;
}

// Tensor map of the raw atoms of a pool region as [slot][row block][group x
// 144 words]: base = the pool (or shared blob) plus the region's offset, row
// blocks atom_rows apart (groups x 576 bytes), slots `stride` bytes apart.
static cudaError_t atoms_map(CUtensorMap *m, const void *base, int groups, int row_blocks, int64_t n_slots,
                             uint64_t stride)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {uint64_t(groups) * (kAtomBytes / 4), uint64_t(row_blocks), uint64_t(n_slots)};
    const cuuint64_t strides[2] = {uint64_t(groups) * kAtomBytes, stride};
    const cuuint32_t box[3] = {kAtomBytes / 4, 8, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The same for 8-bit atoms (1088 bytes = 272 words, above the 256 a box
// dimension may hold): [slot][row block][group x 2 halves][136 words], one
// box {136 words, 2 halves, 8 row blocks, 1 slot} = 8 whole atoms per K step.
static cudaError_t atoms_map8(CUtensorMap *m, const void *base, int groups, int row_blocks, int64_t n_slots,
                              uint64_t stride)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    constexpr int kHalfWords = kAtom8Bytes / 8;                  // 136
    const cuuint64_t dims[4] = {uint64_t(kHalfWords), uint64_t(groups) * 2, uint64_t(row_blocks), uint64_t(n_slots)};
    const cuuint64_t strides[3] = {uint64_t(kAtom8Bytes / 2), uint64_t(groups) * kAtom8Bytes, stride};
    const cuuint32_t box[4] = {uint32_t(kHalfWords), 2, 8, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void *>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static cudaError_t rows_map(CUtensorMap *m, const void *base, bool bf16, uint64_t cols, uint64_t rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {uint32_t(kPfK), uint32_t(kPfBoxRows)};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                              const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_router_gemm(const RouteParams &r, cudaStream_t st)
{
    GemmParams g = {};
    g.mode = 2;
    g.x = r.x;
    g.Wr = r.Wr;
    g.logits = r.logits;
    g.err = r.err;
    g.T = r.T;
    g.H = r.H;
    g.E = r.E;
    g.k = r.k;
    g.m_tiles = (r.E + kPfM - 1) / kPfM;
    CUtensorMap xmap;
    cudaError_t e = rows_map(&xmap, r.x, true, uint64_t(r.H), uint64_t(r.T));
    if (e != cudaSuccess) return e;
    const int ntile = (r.T + kPfMaxN - 1) / kPfMaxN;
    return launch_pdl(router_gemm_kernel, dim3(persistent_grid(ntile * g.m_tiles)), dim3(kPfThreads), kPfSmem, st, g,
                      xmap);
}

cudaError_t launch_prefill(const PrefillParams &p, const GemmParams &g0, cudaStream_t st, const cudaEvent_t *prof,
                           int nprof)
{
    const int nch = (p.T + bucket_tok(p.T) - 1) / bucket_tok(p.T);
    CUtensorMap xmap, hmap;
    cudaError_t e = rows_map(&xmap, g0.x, false, uint64_t(p.H), uint64_t(p.T));   // unused: gate/up gathers B itself
    if (e != cudaSuccess) return e;
    if ((e = rows_map(&hmap, g0.hbuf, false, uint64_t(g0.I), uint64_t(p.P + p.T))) != cudaSuccess) return e;
    // raw atoms: gate/up region [I/8 row blocks][H/64 groups], down region [H/16][I/64] at I/8 x H/64 atoms
    const bool b8 = g0.bits == 8;
    const uint64_t down_off = uint64_t(g0.I / 8) * (p.H / kGroup) * (b8 ? kAtom8Bytes : kAtomBytes);
    const uint8_t *shared_down = g0.shared_blob + down_off, *pool_down = g0.pool + down_off;
    auto amap = b8 ? atoms_map8 : atoms_map;
    CUtensorMap gu_pool, gu_shared, dn_pool, dn_shared;
    if ((e = amap(&gu_pool, g0.pool, p.H / kGroup, g0.I / 8, g0.n_slots, g0.stride)) != cudaSuccess) return e;
    if ((e = amap(&gu_shared, g0.shared_blob, p.H / kGroup, g0.I / 8, 1, g0.stride)) != cudaSuccess) return e;
    if ((e = amap(&dn_pool, pool_down, g0.I / kGroup, p.H / 16, g0.n_slots, g0.stride)) != cudaSuccess) return e;
    if ((e = amap(&dn_shared, shared_down, g0.I / kGroup, p.H / 16, 1, g0.stride)) != cudaSuccess) return e;
    if (p.T <= kBucketSmallT) {
        if ((e = launch_pdl(bucket_small_kernel, dim3(1 + (p.T + 31) / 32), dim3(1024), bucket_small_smem(p.E), st, p,
                            g0)) != cudaSuccess)
            return e;
    } else {
        if ((e = launch_pdl(bucket_count_kernel, dim3(nch), dim3(256), 0, st, p)) != cudaSuccess) return e;
        if ((e = launch_pdl(bucket_scan_kernel, dim3((p.E + 31) / 32), dim3(1024), 0, st, p)) != cudaSuccess) return e;
        if ((e = launch_pdl(bucket_scatter_kernel, dim3(nch), dim3(32), 0, st, p)) != cudaSuccess) return e;
        if ((e = launch_pdl(convert_x_kernel, dim3((p.T + 7) / 8), dim3(256), 0, st, g0)) != cudaSuccess) return e;
    }
    const int maxt = prefill_max_tiles(p.T, p.k, p.E);
    GemmParams g = g0;
    g.mode = 0;
    g.m_tiles = g.I / 64;
    if ((e = prof_record(nprof > 0 ? prof[0] : nullptr, st)) != cudaSuccess) return e;
    // T <= kXNarrowT: every tile holds at most T tokens, so the narrow ring shape fits;
    // its 128-column K steps need K (H for gate/up, I for down) a multiple of 128
    const bool narrow = p.T <= kXNarrowT;
    const XLaunch gu = pick_gemm(b8, narrow, false, p.H), dn = pick_gemm(b8, narrow, true, g0.I);
    if ((e = launch_pdl(gu.kern, dim3(persistent_grid(maxt * g.m_tiles)), dim3(kXThreads), gu.smem, st, g, xmap,
                        gu_pool, gu_shared)) != cudaSuccess)
        return e;
    if ((e = prof_record(nprof > 1 ? prof[1] : nullptr, st)) != cudaSuccess) return e;
    g.mode = 1;
    g.m_tiles = p.H / kPfM;
    if ((e = launch_pdl(dn.kern, dim3(persistent_grid(maxt * g.m_tiles)), dim3(kXThreads), dn.smem, st, g, hmap,
                        dn_pool, dn_shared)) != cudaSuccess)
        return e;
    if ((e = prof_record(nprof > 2 ? prof[2] : nullptr, st)) != cudaSuccess) return e;
    return launch_pdl(combine_kernel, dim3(unsigned((p.H / 4 + 255) / 256) * unsigned(p.T)), dim3(256), 0, st, p);
}

}  // namespace smoe
