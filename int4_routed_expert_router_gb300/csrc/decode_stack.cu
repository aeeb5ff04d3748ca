// decode_stack.cu -- one decode step (one token) through a stack of MoE
// layers in a single persistent, cooperative launch: one CTA per SM for the
// whole step.
//
// The CTAs exchange three things per layer -- the router logits, the SwiGLU
// values h, and the layer's output x_{l+1} -- through buffers in the
// workspace that the launch first fills with a sentinel bit pattern (all
// ones: a NaN that the arithmetic never writes; a result with that pattern is
// stored as the canonical NaN instead). A reader polls the words it needs
// with relaxed loads until none holds the sentinel, so the data itself is the
// signal: no arrival counter, no fence, one round trip to L2 per exchange.
// Each word is written once per launch, and every value stands on its own, so
// no ordering between words is needed.
//
// Per layer l, CTA c of G:
//   A. x_l into shared memory (the caller's x_0 by a bulk copy; later layers
//      polled from the exchange buffer).
//   B. Router rows c, c + G, ... (row E is the shared-gate vector; loaded
//      during the previous layer) dotted with x_l; the logits go out.
//   D. Every thread polls its logit and the CTA picks the top k (the same
//      selection and weights as route_common.cuh's, so ids, weights and
//      gate equal moe_route's bit for bit); CTA 0 writes them out.
//   E. The CTA requests its routed gate/up units (expert j in route order,
//      row block rb: 32 contiguous atoms, one bulk copy each) and, for
//      c < H/16, its down rows 16c .. 16c + 15 of every routed expert.
//   C. CTAs c < I/8 compute the shared expert's gate/up unit c (intermediates
//      8c .. 8c + 7; its weights were loaded during the previous layer) while
//      the routed units' first bytes are on their way: done before the
//      top-k, it delayed these CTAs' requests, and the slowest CTA's h gates
//      every output CTA.
//   F. Gate/up units, a batch at a time once the batch has landed -> h as
//      bf16 high and low parts.
//   G. CTAs c < H/16: poll all experts' h, down rows of every expert, combine
//      in route order with the routing weights, + gate * shared expert +
//      x_l, one bf16 rounding -> x_{l+1} (exchange buffer and the caller's
//      xs).
// The per-atom arithmetic is the decode kernel's: bf16 (128 + q) fragments on
// m16n8k16 tensor-core steps, s and b - 128 s applied per group, fp32 sums.
//
// Every wait is bounded. A poll that runs past the limit (two seconds by
// default) stores SMOE_DEV_TIMEOUT and raises the launch's abort word, which
// ends the other CTAs' polls; the CTAs then run to the end on whatever the
// buffers hold (every address stays in bounds). Waits for a CTA's own bulk
// copies keep their own two-second limit, so no CTA leaves with a copy in
// flight.
// Pages: the per-token expert stream of a decode step, fixed-stride blobs and
// one read per expert (xix.ai article, paragraph on how it works); the
// resident router and shared experts (agentlenshq article, how expert
// streaming works).
#include "decode_common.cuh"
#include "route_common.cuh"

namespace smoe {

constexpr int kStkWarps = 16;
constexpr int kStkThreads = kStkWarps * 32;
constexpr int kStkUnitBatch = 5;       // routed gate/up units a warp works on at once (80B: all of a CTA's)
constexpr uint32_t kSentinel32 = 0xFFFFFFFFu;
constexpr uint16_t kSentinel16 = 0xFFFFu;
constexpr int kStkMaxE = 512;           // experts per layer the one-launch step takes (larger E: per-layer calls)

struct StkSmem {
    int x_s, xsum, rows, table, sunit, units, wdn, red, hh, gsum, yd, ysum, mx, cand, sel, ints, bars, total;
};

// Shared memory of the stack kernel. 4-bit atoms: the shared expert's unit,
// nu routed units and the down rows of every expert each have a region of
// their own, so the next layer's shared unit and shared down rows load during
// this layer. 8-bit atoms (twice the bytes): one ring of nslot unit slots
// (the shared unit, if the CTA has one, in slot 0, then the routed units);
// once the units are read, the down rows, h, its group sums and the down
// partial sums reuse the ring.
__host__ __device__ inline StkSmem stk_smem(int H, int E, int I, int U, int nr, int nu, int bits, int nslot)
{
    const int ngH = H / kGroup, ngI = I / kGroup;
    const int AB = bits == 8 ? kAtom8Bytes : kAtomBytes;
    StkSmem L;
    int o = 0;
    L.x_s = o;   o = align128(o + 2 * H + 16);
    L.xsum = o;  o = align128(o + ngH * 4);
    L.rows = o;  o = align128(o + (nr > 0 ? nr : 1) * H * 2);
    L.table = o; o = align128(o + 2 * E * 4);
    if (bits == 8) {
        const int ring = (nslot > 0 ? nslot : 1) * ngH * AB;
        L.sunit = o;
        L.units = o;                                 // + one slot where the CTA has a shared unit
        L.wdn = o;
        L.hh = align128(L.wdn + U * ngI * AB);
        L.gsum = align128(L.hh + U * 2 * I * 2);
        L.yd = align128(L.gsum + U * ngI * 4);
        const int reuse = align128(L.yd + U * ngI * 16 * 4) - o;
        o = align128(o + (ring > reuse ? ring : reuse));
        L.red = o;   o = align128(o + (nu + 1) * kStkWarps * 8 * 8);
    } else {
        L.sunit = o; o = align128(o + ngH * AB);
        L.units = o; o = align128(o + (nu > 0 ? nu : 1) * ngH * AB);
        L.wdn = o;   o = align128(o + U * ngI * AB);
        L.red = o;   o = align128(o + (nu + 1) * kStkWarps * 8 * 8);
        L.hh = o;    o = align128(o + U * 2 * I * 2);
        L.gsum = o;  o = align128(o + U * ngI * 4);
        L.yd = o;    o = align128(o + U * ngI * 16 * 4);
    }
    L.ysum = o;  o = align128(o + U * 16 * 4);
    L.mx = o;    o = align128(o + 2 * kStkWarps * 4 + 8);
    L.cand = o;  o = align128(o + 2 * E * 4);
    L.sel = o;   o = align128(o + 2 * 16 * 4);
    L.ints = o;  o = align128(o + 64 * 4);
    L.bars = o;  o = align128(o + (nu + U + 5) * 8);
    L.total = o;
    return L;
}

__device__ __forceinline__ void bulk_nohint(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint2 ld_relaxed_v2(const void *p)
{
    uint2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_relaxed_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u16(uint16_t *p, uint16_t v)
{
    asm volatile("st.relaxed.gpu.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_v4(void *p, uint4 v)
{
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// No half-word of v is the 16-bit sentinel.
__device__ __forceinline__ bool ready16(uint32_t v)
{
    return (v & 0xFFFFu) != kSentinel16 && (v >> 16) != kSentinel16;
}

// A value that happens to carry the sentinel pattern (a NaN) is stored as the
// canonical NaN of its width.
__device__ __forceinline__ uint16_t canon16(uint16_t v) { return v == kSentinel16 ? uint16_t(0x7FFF) : v; }
__device__ __forceinline__ uint32_t canon32(uint32_t v) { return v == kSentinel32 ? 0x7FFFFFFFu : v; }

// Polls `load` (which re-reads the words it has not yet seen written and
// returns true once all are) until it succeeds for every lane of `mask`, the
// abort word is raised, or limit_ns pass; on the last, stores
// SMOE_DEV_TIMEOUT and raises the abort word. Returns whether the data came.
// All lanes of `mask` call it together and leave it together: every decision
// is taken warp-wide, because a warp whose lanes had left a sleeping loop at
// different times ran the code after it (the top-k, several times over)
// unconverged, about four times slower. Only the words not yet seen written
// are read again, after a short pause: every CTA polls the same few L2 lines
// that the writers are storing to, and re-reading all of them in a tight loop
// delayed those stores by microseconds.
template <typename F>
__device__ __forceinline__ bool poll_rounds(F load, uint32_t mask, uint32_t *abortw, int32_t *err, uint64_t limit_ns,
                                            uint32_t pause)
{
    if (__all_sync(mask, load())) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(pause);                     // sleeps twice the request on this GPU
        if (__all_sync(mask, load())) return true;
        if ((it & 15) == 0) {
            if (__any_sync(mask, ld_relaxed(abortw) != 0u)) return false;
            if (__any_sync(mask, globaltimer_ns() - t0 > limit_ns)) {
                if ((threadIdx.x & 31) == __ffs(mask) - 1) {
                    atomicExch(abortw, 1u);
                    set_error(err, SMOE_DEV_TIMEOUT);
                }
                return false;
            }
        }
    }
}

// Even so, lanes that slept in the loop may wake at different times and stay
// split into groups that the scheduler issues one after another (measured: a
// warp's top-k afterwards took 20,000 cycles instead of 5,000). A warp
// reduction after a __syncwarp merges them again; so every poll ends with one.
template <typename F>
__device__ __forceinline__ bool poll(F load, uint32_t mask, uint32_t *abortw, int32_t *err, uint64_t limit_ns,
                                     uint32_t pause = 32)
{
    const bool ok = poll_rounds(load, mask, abortw, err, limit_ns, pause);
    __syncwarp(mask);
    (void)__reduce_or_sync(mask, 0u);
    return ok;
}

// Thread 0 waits until *ctr >= target (bounded like poll), then an acquire
// fence; the CTA synchronises. Used once, after the sentinel fill.
__device__ void grid_wait(const uint32_t *ctr, uint32_t target, uint32_t *abortw, int32_t *err, uint64_t limit_ns)
{
    if (threadIdx.x == 0) {
        poll([&] { return ld_relaxed(ctr) >= target; }, 1u, abortw, err, limit_ns);
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    __syncthreads();
}

// The token's B fragment of one 64-column group kb of x (the token is MMA
// column 0: lanes 0..3 hold columns 16 t4 .. 16 t4 + 15, the others zeros) and
// the group's sum of x. A warp always works on the same one or two groups, so
// it loads them once per layer.
struct XFrag {
    uint4 xa, xb;
    float xs;
};

__device__ __forceinline__ XFrag load_xfrag(const uint16_t *x_s, const float *xsum, int kb, int ngH, int lane)
{
    XFrag f;
    f.xa = make_uint4(0, 0, 0, 0);
    f.xb = f.xa;
    f.xs = 0.f;
    if (kb < ngH) {
        if (lane < 4) {
            const int col = kb * kGroup + 16 * lane;
            f.xa = *reinterpret_cast<const uint4 *>(x_s + col);
            f.xb = *reinterpret_cast<const uint4 *>(x_s + col + 8);
        }
        f.xs = xsum[kb];
    }
    return f;
}

// The gate/up partial sums of one atom (16 rows x one 64-column group) for
// the token (MMA column 0): lanes 4g (t4 = 0) get gate row g and up row g.
// 8-bit atoms: each nibble plane runs the 4-bit fragments through its own
// tensor-core chains and the epilogue weights the high plane by 16.
template <int BITS>
__device__ __forceinline__ float2 gateup_atom(const uint8_t *atom, const XFrag &f, int lane)
{
    const int g = lane >> 2;
    const uint4 A = *reinterpret_cast<const uint4 *>(atom + 16 * lane);
    uint4 Ah = A;
    if constexpr (BITS == 8) Ah = *reinterpret_cast<const uint4 *>(atom + kAtomQBytes + 16 * lane);
    const uint2 SB = *reinterpret_cast<const uint2 *>(atom + AtomFmt<BITS>::sb + 8 * g);
    const float xs_kb = f.xs;
    const uint32_t xl[4] = {f.xa.x, f.xa.y, f.xa.z, f.xa.w}, xr[4] = {f.xb.x, f.xb.y, f.xb.z, f.xb.w};
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    float hcc[4] = {0.f, 0.f, 0.f, 0.f}, hcc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 4; m += 2) {
        const uint32_t a0[4] = {nib_pair(A.x, m), nib_pair(A.z, m), nib_pair(A.y, m), nib_pair(A.w, m)};
        const uint32_t a1[4] = {nib_pair(A.x, m + 1), nib_pair(A.z, m + 1), nib_pair(A.y, m + 1),
                                nib_pair(A.w, m + 1)};
        mma_bf16(acc, a0, xl[m], xr[m]);
        mma_bf16(acc2, a1, xl[m + 1], xr[m + 1]);
        if constexpr (BITS == 8) {
            const uint32_t b0[4] = {nib_pair(Ah.x, m), nib_pair(Ah.z, m), nib_pair(Ah.y, m), nib_pair(Ah.w, m)};
            const uint32_t b1[4] = {nib_pair(Ah.x, m + 1), nib_pair(Ah.z, m + 1), nib_pair(Ah.y, m + 1),
                                    nib_pair(Ah.w, m + 1)};
            mma_bf16(hcc, b0, xl[m], xr[m]);
            mma_bf16(hcc2, b1, xl[m + 1], xr[m + 1]);
        }
    }
    float sg, bpg, su, bpu;
    if constexpr (BITS == 8) {
        scale_bias8(SB.x, sg, bpg);
        scale_bias8(SB.y, su, bpu);
        return make_float2(fmaf(sg, fmaf(16.f, hcc[0] + hcc2[0], acc[0] + acc2[0]), bpg * xs_kb),
                           fmaf(su, fmaf(16.f, hcc[2] + hcc2[2], acc[2] + acc2[2]), bpu * xs_kb));
    } else {
        scale_bias(SB.x, sg, bpg);
        scale_bias(SB.y, su, bpu);
        return make_float2(fmaf(sg, acc[0] + acc2[0], bpg * xs_kb), fmaf(su, acc[2] + acc2[2], bpu * xs_kb));
    }
}

// One warp's partial sums of a gate/up unit (H/64 <= 32 atoms, one 64-column
// group of x each) when the 16 warps share it: warp w takes atoms w and
// w + 16 (f0, f1: their x fragments), whose tensor-core chains overlap, and
// adds them in that order.
template <int BITS>
__device__ __forceinline__ float2 gateup_partial(const uint8_t *ubase, const XFrag &f0, const XFrag &f1, int ngH,
                                                 int warp, int lane)
{
    float aG = 0.f, aU = 0.f;
    if (warp < ngH) {
        const int kb1 = warp + kStkWarps;
        const float2 a = gateup_atom<BITS>(ubase + warp * AtomFmt<BITS>::bytes, f0, lane);
        float2 b = make_float2(0.f, 0.f);
        if (kb1 < ngH) b = gateup_atom<BITS>(ubase + kb1 * AtomFmt<BITS>::bytes, f1, lane);
        aG += a.x;
        aU += a.y;
        aG += b.x;
        aU += b.y;
    }
    return make_float2(aG, aU);
}

// Warp `warp` (whole warp) finishes a gate/up unit from the nw warps'
// partials red[w * 8 + g] (summed in warp order): h of intermediates
// 8 rb .. 8 rb + 7 as bf16 high parts and low parts (h - high), stored as one
// 16-byte store each into the exchange rows hx_hi, hx_lo (a value with the
// sentinel pattern as the canonical NaN); then one relaxed add on the
// expert's arrival counter. The add may become visible before the stores (a
// release would hold the warp until they are acknowledged, about a microsecond
// on the layer's critical path), so a reader that sees the counter at I/8
// checks the copied h for sentinels and copies again if one is left.
__device__ __forceinline__ void finish_unit(const float2 *red, int nw, bool valid, uint16_t *hx_hi, uint16_t *hx_lo,
                                            uint32_t *cnt, int lane)
{
    const int g = lane >> 2;
    float aG = red[g].x, aU = red[g].y;
    for (int w = 1; w < nw; ++w) {
        const float2 v = red[w * 8 + g];
        aG += v.x;
        aU += v.y;
    }
    const float hv = valid ? silu(aG) * aU : 0.f;
    const uint16_t hi = canon16(f32_to_bf16_bits(hv));
    const uint16_t lo = canon16(f32_to_bf16_bits(hv - __uint_as_float(uint32_t(hi) << 16)));
    uint32_t phi[4], plo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {                       // lanes 4g hold intermediate g
        const uint32_t h0 = __shfl_sync(0xffffffffu, uint32_t(hi), 8 * q);
        const uint32_t h1 = __shfl_sync(0xffffffffu, uint32_t(hi), 8 * q + 4);
        const uint32_t l0 = __shfl_sync(0xffffffffu, uint32_t(lo), 8 * q);
        const uint32_t l1 = __shfl_sync(0xffffffffu, uint32_t(lo), 8 * q + 4);
        phi[q] = h0 | (h1 << 16);
        plo[q] = l0 | (l1 << 16);
    }
    if (lane == 0) {
        *reinterpret_cast<uint4 *>(hx_hi) = make_uint4(phi[0], phi[1], phi[2], phi[3]);
        *reinterpret_cast<uint4 *>(hx_lo) = make_uint4(plo[0], plo[1], plo[2], plo[3]);
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
    }
}

// Down rows 16 c .. 16 c + 15 of one expert over one 64-group of h, with h
// split into bf16 high and low parts as MMA columns 0 and 1: lanes 0..3 (B
// column 0) hold the group's high parts, lanes 4..7 (column 1) the low parts,
// h0: columns 16 t4 .. +7 of the group, h1: +8 .. +15; other lanes hold zeros.
// One m16n8k16 step per 16 columns yields both partial sums (per nibble
// plane for 8-bit atoms); gsum: the group's sum of high + low parts. Lanes 4g
// (t4 = 0) return rows g and g + 8.
template <int BITS>
__device__ __forceinline__ float2 down_atom(const uint8_t *atom, uint4 h0, uint4 h1, float gsum, int lane)
{
    const int g = lane >> 2;
    const uint4 A = *reinterpret_cast<const uint4 *>(atom + 16 * lane);
    uint4 Ah = A;
    if constexpr (BITS == 8) Ah = *reinterpret_cast<const uint4 *>(atom + kAtomQBytes + 16 * lane);
    const uint2 SB = *reinterpret_cast<const uint2 *>(atom + AtomFmt<BITS>::sb + 8 * g);
    const uint32_t ha_[4] = {h0.x, h0.y, h0.z, h0.w}, hb_[4] = {h1.x, h1.y, h1.z, h1.w};
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    float hcc[4] = {0.f, 0.f, 0.f, 0.f}, hcc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 4; m += 2) {
        const uint32_t a0[4] = {nib_pair(A.x, m), nib_pair(A.z, m), nib_pair(A.y, m), nib_pair(A.w, m)};
        const uint32_t a1[4] = {nib_pair(A.x, m + 1), nib_pair(A.z, m + 1), nib_pair(A.y, m + 1),
                                nib_pair(A.w, m + 1)};
        mma_bf16(acc, a0, ha_[m], hb_[m]);
        mma_bf16(acc2, a1, ha_[m + 1], hb_[m + 1]);
        if constexpr (BITS == 8) {
            const uint32_t b0[4] = {nib_pair(Ah.x, m), nib_pair(Ah.z, m), nib_pair(Ah.y, m), nib_pair(Ah.w, m)};
            const uint32_t b1[4] = {nib_pair(Ah.x, m + 1), nib_pair(Ah.z, m + 1), nib_pair(Ah.y, m + 1),
                                    nib_pair(Ah.w, m + 1)};
            mma_bf16(hcc, b0, ha_[m], hb_[m]);
            mma_bf16(hcc2, b1, ha_[m + 1], hb_[m + 1]);
        }
    }
    float s0, bp0, s1, bp1;
    // (row, column 0) + (row, column 1): the high and the low part's sums
    if constexpr (BITS == 8) {
        scale_bias8(SB.x, s0, bp0);
        scale_bias8(SB.y, s1, bp1);
        return make_float2(fmaf(s0, fmaf(16.f, (hcc[0] + hcc2[0]) + (hcc[1] + hcc2[1]),
                                         (acc[0] + acc2[0]) + (acc[1] + acc2[1])), bp0 * gsum),
                           fmaf(s1, fmaf(16.f, (hcc[2] + hcc2[2]) + (hcc[3] + hcc2[3]),
                                         (acc[2] + acc2[2]) + (acc[3] + acc2[3])), bp1 * gsum));
    } else {
        scale_bias(SB.x, s0, bp0);
        scale_bias(SB.y, s1, bp1);
        return make_float2(fmaf(s0, (acc[0] + acc2[0]) + (acc[1] + acc2[1]), bp0 * gsum),
                           fmaf(s1, (acc[2] + acc2[2]) + (acc[3] + acc2[3]), bp1 * gsum));
    }
}

// Every (expert u, group kb) sum of h's high + low parts, gsum[u * ngI + kb]
// (the bias term of down_atom), in a fixed order: four threads per group,
// thread q of them summing the high then the low parts of columns
// 16 q .. 16 q + 15 in column order, then the four partial sums in a fixed
// tree (pairs, then the halves). The whole CTA calls it; each group is summed
// once per layer (4 U I/64 <= 512 threads: one round at the 80B shape). It
// reads every half-word of h once, so it also returns whether this thread met
// the sentinel (a value not yet written when h was copied).
__device__ __forceinline__ bool group_sums(const uint16_t *hh, int U, int I, int ngI, float *gsum)
{
    const int tid = threadIdx.x, q = tid & 3;
    bool miss = false;
    for (int gi = tid >> 2; gi < ((U * ngI + 7) & ~7); gi += kStkThreads / 4) {   // whole warps per round
        float s = 0.f;
        if (gi < U * ngI) {
            const int u = gi / ngI, kb = gi - u * ngI;
            const uint16_t *hi = hh + size_t(u) * I + kb * kGroup + 16 * q, *lo = hi + size_t(U) * I;
            const uint4 a = *reinterpret_cast<const uint4 *>(hi), b = *reinterpret_cast<const uint4 *>(hi + 8);
            const uint4 c = *reinterpret_cast<const uint4 *>(lo), d = *reinterpret_cast<const uint4 *>(lo + 8);
            const uint32_t v[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
            for (int j = 0; j < 16; ++j) s += bf16lo(v[j]) + bf16hi(v[j]);
            // the sentinel is a NaN, so only a non-finite partial sum can hide one:
            // then (rarely: NaN or infinite data) check the half-words themselves
            if (!(fabsf(s) <= 3.402823466e38f))
#pragma unroll
                for (int j = 0; j < 16; ++j) miss |= !ready16(v[j]);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (q == 0 && gi < U * ngI) gsum[gi] = s;
    }
    return miss;
}

// Composite order of the routing keys: larger key first, equal keys by lower id.
__device__ __forceinline__ bool key_before(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

// The k largest of E <= 512 logits (plus the optional offsets), in route
// order, by the whole CTA (thread t holds logit t): each warp's slice maximum;
// the k-th largest of the 16 maxima bounds the k-th largest key from below
// (k distinct keys reach it), so only the keys at or above it are
// candidates (ties: the lower id first, a strict order); a candidate's rank
// among the candidates is its place in route order. The same selection as
// route_common.cuh's, so the ids are moe_route's. ncand must be zero on entry
// and is zero again on return. thr: two words of scratch. Four CTA barriers.
__device__ void block_topk(float z, const float *bias, int E, int k, uint32_t *mx_k, int32_t *mx_i, uint32_t *thr,
                           uint32_t *cand_k, int32_t *cand_i, int *ncand, uint32_t *sel_k, int32_t *sel_i)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t key = tid < E ? fkey(z + (bias ? bias[tid] : 0.f)) : 0u;
    const int32_t id = tid < E ? tid : 0x7fffffff;
    const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
    const int32_t mi = int32_t(__reduce_min_sync(0xffffffffu, key == mk ? uint32_t(id) : 0x7fffffffu));
    if (lane == 0) {
        mx_k[warp] = mk;
        mx_i[warp] = mi;
    }
    __syncthreads();
    // warp 0 finds the bound (each warp doing it was 16 times the issued work
    // for one more barrier's worth of time) and passes it through thr
    if (warp == 0) {
        const int j = lane & (kStkWarps - 1);
        const uint32_t jk = mx_k[j];
        const int32_t ji = mx_i[j];
        int r = 0;
#pragma unroll
        for (int i = 0; i < kStkWarps; ++i) r += key_before(mx_k[i], mx_i[i], jk, ji);
        const uint32_t b = __ballot_sync(0xffffffffu, lane < kStkWarps && r == k - 1);
        const int src = b ? __ffs(b) - 1 : 0;
        const uint32_t tk0 = b ? __shfl_sync(0xffffffffu, jk, src) : 0u;   // no such rank: every key qualifies
        const int32_t ti0 = b ? __shfl_sync(0xffffffffu, ji, src) : 0x7fffffff;
        if (lane == 0) {
            thr[0] = tk0;
            thr[1] = uint32_t(ti0);
        }
    }
    __syncthreads();
    const uint32_t tk = thr[0];
    const int32_t ti = int32_t(thr[1]);
    const bool cand = key != 0u && !key_before(tk, ti, key, id);
    const uint32_t cb = __ballot_sync(0xffffffffu, cand);
    int base = 0;
    if (lane == 0 && cb) base = atomicAdd(ncand, __popc(cb));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (cand) {
        const int pos = base + __popc(cb & ((1u << lane) - 1u));
        cand_k[pos] = key;
        cand_i[pos] = id;
    }
    __syncthreads();
    const int n = *ncand;
    if (tid < n) {
        const uint32_t ck = cand_k[tid];
        const int32_t ci = cand_i[tid];
        int rr = 0;
        for (int q = 0; q < n; ++q) rr += key_before(cand_k[q], cand_i[q], ck, ci);
        if (rr < k) {
            sel_k[rr] = ck;
            sel_i[rr] = ci;
        }
    }
    __syncthreads();
    if (tid == 0) *ncand = 0;
}

// NGI = I / 64 (1, 2, 4 or 8) is a template parameter: the atom and unit
// bookkeeping divides by it and by I / 8, and division by a value known only at
// run time cost tens of instructions per atom. BITS: 4, or 8 for MLX 8-bit
// experts (two-plane atoms, the ring plan of stk_smem).
template <int NGI, int BITS>
__global__ void __launch_bounds__(kStkThreads, 1) decode_stack_kernel(const __grid_constant__ StackParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int ngI = NGI, I = NGI * kGroup, nrb = I / 8;
    constexpr int AB = AtomFmt<BITS>::bytes;
    constexpr bool kRing = BITS == 8;                 // units, then down rows and h, share one ring
    const int H = p.H, E = p.E, k = p.k, U = p.U;
    const int ngH = H / kGroup, nD = H / 16;
    const uint32_t ubytes = uint32_t(ngH * AB), wbytes = uint32_t(ngI * AB);
    const uint64_t down_off = uint64_t(nrb) * ngH * AB;
    const StkSmem L = stk_smem(H, E, I, U, p.nr, p.nu, BITS, p.nslot);
    uint16_t *x_s = reinterpret_cast<uint16_t *>(smem + L.x_s);
    float *xsum = reinterpret_cast<float *>(smem + L.xsum);
    uint16_t *rows = reinterpret_cast<uint16_t *>(smem + L.rows);
    int *tables = reinterpret_cast<int *>(smem + L.table);
    const int c_ = int(blockIdx.x);
    uint8_t *sunit = smem + L.sunit;
    uint8_t *units = smem + L.units + (kRing && c_ < nrb ? ubytes : 0u);   // ring: after the shared unit
    uint8_t *wdn = smem + L.wdn;
    float2 *red = reinterpret_cast<float2 *>(smem + L.red);          // [nu + 1][warps][8]
    uint16_t *hh = reinterpret_cast<uint16_t *>(smem + L.hh);        // [hi, lo][U][I]: h of the layer
    float *gsum_s = reinterpret_cast<float *>(smem + L.gsum);        // [U * ngI] group sums of h
    float *yd = reinterpret_cast<float *>(smem + L.yd);              // [U * ngI atoms][16 rows]
    float *ysum = reinterpret_cast<float *>(smem + L.ysum);          // [U][16 rows]
    uint32_t *mx_k = reinterpret_cast<uint32_t *>(smem + L.mx);      // [16] slice maxima
    int32_t *mx_i = reinterpret_cast<int32_t *>(mx_k + kStkWarps);
    uint32_t *thr = mx_k + 2 * kStkWarps;                            // [2] the top-k's bound
    uint32_t *cand_k = reinterpret_cast<uint32_t *>(smem + L.cand);  // [E] candidates
    int32_t *cand_i = reinterpret_cast<int32_t *>(cand_k + E);
    uint32_t *sel_k = reinterpret_cast<uint32_t *>(smem + L.sel);    // [16] chosen keys, route order
    int32_t *ids_s = reinterpret_cast<int32_t *>(sel_k + 16);        // [16] chosen experts, route order
    int *ints = reinterpret_cast<int *>(smem + L.ints);
    float *w_s = reinterpret_cast<float *>(ints);                    // [16]
    float *gate_s = reinterpret_cast<float *>(ints + 16);
    int *ncand = ints + 17;
    uint32_t *vmask_s = reinterpret_cast<uint32_t *>(ints + 18);     // bit u: expert u's blob is in the pool
    int *giveup_s = ints + 19;                                        // the h copy's retries ran out
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *ubar = bars, *dbar = bars + p.nu, *xbar = dbar + U, *rbar = xbar + 1, *sbar = rbar + 1,
             *hbar = sbar + 1;                                       // the layer's h has landed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = int(gridDim.x), c = int(blockIdx.x);
    uint32_t *abortw = p.sync + 1;
    const uint64_t lim = p.wait_ns;
    const int nr_mine = c <= E ? (E - c) / G + 1 : 0;               // router rows c, c + G, ... <= E
    const bool has_shared = c < nrb;                                 // the shared expert's unit rb = c
    const bool has_down = c < nD;                                    // output rows 16 c .. 16 c + 15
    const int R = k * nrb;                                           // routed units per layer
    // routed unit order: the CTAs without down rows first, then the others from
    // the highest index down, so the CTAs that also take a shared unit (c < I/8)
    // are the last to get a fifth routed unit
    const int ord = c >= nD ? c - nD : (nD - 1 - c) + (G - nD);
    const int n_mine = ord < R ? (R - 1 - ord) / G + 1 : 0;          // routed units r = ord + i G

    auto issue_fixed = [&](int l) {                                  // thread 0: what layer l needs that is known early
        mbar_arrive_expect_tx(rbar, uint32_t(nr_mine * H * 2 + E * 4));
        for (int j = 0; j < nr_mine; ++j) {
            const int r = c + j * G;
            bulk_nohint(rows + size_t(j) * H, r < E ? p.Wr[l] + size_t(r) * H : p.ws[l], uint32_t(H * 2), rbar);
        }
        bulk_nohint(tables + (l & 1) * E, p.table + size_t(l) * E, uint32_t(E * 4), rbar);
    };
    auto issue_shared_unit = [&](int l) {
        mbar_arrive_expect_tx(sbar, ubytes);
        bulk_nohint(sunit, p.shared[l] + size_t(c) * ubytes, ubytes, sbar);
    };
    auto issue_shared_down = [&](int l) {
        mbar_arrive_expect_tx(&dbar[0], wbytes);
        bulk_nohint(wdn, p.shared[l] + down_off + size_t(c) * wbytes, wbytes, &dbar[0]);
    };

    if (tid == 0) {
        for (int i = 0; i < p.nu + U + 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *ncand = 0;
        *giveup_s = 0;
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(xbar, uint32_t(H * 2));
        bulk_nohint(x_s, p.xs, uint32_t(H * 2), xbar);
        issue_fixed(0);
        if (has_shared) issue_shared_unit(0);
        if (has_down && !kRing) issue_shared_down(0);
    }
    // ---- sentinel fill of the exchange buffers (16-byte stores over the grid),
    // then one grid-wide arrival before any CTA writes a value
    {
        uint4 *xb = reinterpret_cast<uint4 *>(p.xbuf);
        const uint4 ones = make_uint4(kSentinel32, kSentinel32, kSentinel32, kSentinel32);
        for (uint64_t i = uint64_t(c) * kStkThreads + tid; i < p.xbuf_words16; i += uint64_t(G) * kStkThreads)
            xb[i] = ones;
        __syncthreads();
        if (tid == 0) ticket_add(&p.sync[0], 1u);
        grid_wait(&p.sync[0], uint32_t(G), abortw, p.err, lim);
    }
    const uint64_t pol = policy_evict_first();
    bool bad = false;                                 // a bounded wait for this CTA's own copies gave up
    uint32_t hpar = 0;                                // phase parity of the next wait on hbar

    for (int l = 0; l < p.n_layers; ++l) {
        const uint32_t par = uint32_t(l & 1);
        const int *table = tables + (l & 1) * E;
        float *zl = p.zl + size_t(l) * (E + kStackZPad);
        uint16_t *hx_hi = p.hx + size_t(l) * 2 * U * I, *hx_lo = hx_hi + size_t(U) * I;
        uint32_t *hcnt = p.hcnt + size_t(l) * U * kStackCntStride;   // expert u's counter at u * stride
        auto blob_of = [&](int u) -> const uint8_t * {              // u = 0: shared; u >= 1: route position u - 1
            if (u == 0) return p.shared[l];
            const int64_t slot = table[ids_s[u - 1]];
            if (slot < 0 || slot >= p.n_slots) return nullptr;
            return p.pool + uint64_t(slot) * p.stride;
        };

        if (kRing && l > 0 && has_shared && tid == 0) issue_shared_unit(l);   // the ring is free again

        // ---- A. x_l
        if (l == 0) {
            if (!bad && !mbar_wait(xbar, 0, p.err)) bad = true;
        } else if (tid < H / 4) {
            // H / 4 (a multiple of 64, at most 512) chunks of 8 bytes: whole warps poll
            const uint16_t *src = p.xe + size_t(l) * H;
            uint2 v;
            bool seen = false;
            poll([&] {
                if (!seen) {
                    v = ld_relaxed_v2(src + 4 * tid);
                    seen = ready16(v.x) && ready16(v.y);
                }
                return seen;
            }, 0xffffffffu, abortw, p.err, lim);
            *reinterpret_cast<uint2 *>(x_s + 4 * tid) = v;
        }
        if (!bad && !mbar_wait(rbar, par, p.err)) bad = true;
        __syncthreads();

        // ---- B. logits of this CTA's router rows; per-group sums of x (bias term)
        for (int j = warp; j < nr_mine; j += kStkWarps) {
            const float z = router_dot(rows + size_t(j) * H, x_s, H, lane);
            if (lane == 0) st_relaxed(reinterpret_cast<uint32_t *>(zl + c + j * G), canon32(__float_as_uint(z)));
        }
        for (int grp = warp; grp < ngH; grp += kStkWarps) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(x_s + grp * kGroup + 2 * lane);
            float s = bf16lo(v) + bf16hi(v);
            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) xsum[grp] = s;
        }
        __syncthreads();
        if (tid == 0 && l + 1 < p.n_layers) {                       // the rows are read; the other table is free
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_fixed(l + 1);
        }
        const XFrag f0 = load_xfrag(x_s, xsum, warp, ngH, lane), f1 = load_xfrag(x_s, xsum, warp + kStkWarps, ngH, lane);

        // ---- D. every thread polls its logit (thread 0 also the shared-gate
        // logit, word E, and under the stall hook word E + 1, which nothing
        // writes), then the CTA's top-k
        {
            const int nz = tid == 0 ? (l == p.stall_layer ? 3 : 2) : (tid < E ? 1 : 0);
            uint32_t zv[3] = {0u, 0u, 0u};
            uint32_t pend = (1u << nz) - 1u;
            poll([&] {
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    if (pend >> q & 1u) zv[q] = ld_relaxed(reinterpret_cast<const uint32_t *>(zl + (q == 0 ? tid : E + q - 1)));
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    if ((pend >> q & 1u) && zv[q] != kSentinel32) pend &= ~(1u << q);
                return pend == 0;
            }, 0xffffffffu, abortw, p.err, lim);
            if (tid == 0) {
                *gate_s = shared_gate(__uint_as_float(zv[1]));
                if (c == 0) p.gate[l] = *gate_s;
            }
            block_topk(__uint_as_float(zv[0]), p.bias, E, k, mx_k, mx_i, thr, cand_k, cand_i, ncand, sel_k,
                       ids_s);
            if (warp == kStkWarps - 1) {                             // weights: needed only by the combine
                const float wl = choice_weight(sel_k, k, lane);
                if (lane < k) {
                    w_s[lane] = wl;
                    if (c == 0) {
                        p.ids[size_t(l) * k + lane] = ids_s[lane];
                        p.w[size_t(l) * k + lane] = wl;
                    }
                }
            }
        }

        // ---- E. request the routed units: lane 0 of warp w issues unit w, w + 16, ...
        // so the copies go out in parallel. The CTAs with output rows request the
        // down rows of every routed expert only once their first unit has landed
        // (in F): they are needed last, and requested with the units they delayed
        // the units' first bytes.
        if (lane == 0)
            for (int it = warp; it < n_mine; it += kStkWarps) {
                const int r = ord + it * G, u = 1 + r / nrb, rb = r % nrb;
                const uint8_t *blob = blob_of(u);
                if (blob) {
                    mbar_arrive_expect_tx(&ubar[it], ubytes);
                    bulk_g2s(units + size_t(it) * ubytes, blob + size_t(rb) * ubytes, ubytes, &ubar[it], pol);
                } else {
                    set_error(p.err, SMOE_DEV_BAD_SLOT);
                    mbar_arrive(&ubar[it]);
                }
            }
        auto issue_down = [&] {                                      // lane 0 of warp w: expert 1 + w
            if (has_down && lane == 0)
                for (int u = 1 + warp; u <= k; u += kStkWarps) {
                    const uint8_t *blob = blob_of(u);
                    if (blob) {
                        mbar_arrive_expect_tx(&dbar[u], wbytes);
                        bulk_g2s(wdn + size_t(u) * wbytes, blob + down_off + size_t(c) * wbytes, wbytes, &dbar[u], pol);
                    } else {
                        mbar_arrive(&dbar[u]);
                    }
                }
        };
        if (n_mine == 0 && !kRing) issue_down();

        // ---- C. the shared expert's unit c (its weights are in shared memory), while
        // the routed units' first bytes are on their way
        if (has_shared) {
            if (!bad && !mbar_wait(sbar, par, p.err)) bad = true;
            const float2 a = gateup_partial<BITS>(sunit, f0, f1, ngH, warp, lane);
            if ((lane & 3) == 0) red[(p.nu * kStkWarps + warp) * 8 + (lane >> 2)] = a;
            __syncthreads();
            if (warp == kStkWarps - 1)
                finish_unit(red + p.nu * kStkWarps * 8, kStkWarps, true, hx_hi + 8 * c, hx_lo + 8 * c, hcnt, lane);
            if (!kRing && tid == 32 && l + 1 < p.n_layers) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_shared_unit(l + 1);
            }
        }

        // ---- F. routed gate/up units; then warp i finishes unit i
        // Up to kStkUnitBatch units at a time, once all of them have landed: the
        // atoms of several units in flight per warp overlap their tensor-core and
        // load latencies, which bound this phase more than the bytes' arrival.
        for (int i = 0; i < n_mine; i += kStkUnitBatch) {
            bool on[kStkUnitBatch], ok[kStkUnitBatch];
#pragma unroll
            for (int q = 0; q < kStkUnitBatch; ++q) {
                on[q] = i + q < n_mine;
                ok[q] = on[q] && blob_of(1 + (ord + (i + q) * G) / nrb) != nullptr;     // uniform
            }
#pragma unroll
            for (int q = 0; q < kStkUnitBatch; ++q)
                if (on[q] && !bad && !mbar_wait(&ubar[i + q], par, p.err)) bad = true;
            if (i == 0 && !kRing) issue_down();
            float2 a[kStkUnitBatch];
#pragma unroll
            for (int q = 0; q < kStkUnitBatch; ++q) {
                a[q] = make_float2(0.f, 0.f);
                if (ok[q] && !bad) a[q] = gateup_partial<BITS>(units + size_t(i + q) * ubytes, f0, f1, ngH, warp, lane);
            }
            if ((lane & 3) == 0) {
#pragma unroll
                for (int q = 0; q < kStkUnitBatch; ++q)
                    if (on[q]) red[((i + q) * kStkWarps + warp) * 8 + (lane >> 2)] = a[q];
            }
        }
        // ring plan: the units are read, so the down rows may overwrite them
        if (kRing) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (kRing) {
            issue_down();
            if (tid == 0 && has_down) issue_shared_down(l);
        }
        for (int i = warp; i < n_mine; i += kStkWarps) {
            const int r = ord + i * G, u = 1 + r / nrb, rb = r % nrb;
            finish_unit(red + i * kStkWarps * 8, kStkWarps, blob_of(u) != nullptr && !bad,
                        hx_hi + size_t(u) * I + 8 * rb, hx_lo + size_t(u) * I + 8 * rb,
                        hcnt + size_t(u) * kStackCntStride, lane);
        }

        // ---- G. down rows 16 c .. 16 c + 15 of every expert, combine -> x_{l+1}.
        // Warp 0 polls the U experts' arrival counters (one per 128-byte line)
        // until every unit has reported, then bulk-copies the layer's h into
        // shared memory (whole lines, so each L2 line is requested once per CTA,
        // not once per 16 bytes). The group sums read every half-word of it; if
        // one still holds the sentinel (its store was overtaken by the relaxed
        // counter add), h is copied again. Then warp w takes atoms
        // a = w, w + 16, ... (expert u = a / (I/64), group kb = a % (I/64)),
        // two at a time.
        if (has_down) {
            const uint32_t hb = uint32_t(U * I * 2);
            auto copy_h = [&] {                                     // one thread
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_arrive_expect_tx(hbar, 2 * hb);
                bulk_nohint(hh, hx_hi, hb, hbar);
                bulk_nohint(hh + size_t(U) * I, hx_lo, hb, hbar);
            };
            if (warp == 0) {
                uint32_t pend = lane < U ? 1u : 0u;
                poll([&] {
                    if (pend && ld_relaxed(hcnt + size_t(lane) * kStackCntStride) >= uint32_t(nrb)) pend = 0;
                    return pend == 0;
                }, 0xffffffffu, abortw, p.err, lim);
                const uint32_t vm = __ballot_sync(0xffffffffu, lane < U && blob_of(lane) != nullptr);
                if (lane == 0) {
                    *vmask_s = vm;                                   // read after the barrier below
                    copy_h();
                }
            }
            uint64_t t_retry = 0;
            for (;;) {
                if (!bad && !mbar_wait(hbar, hpar, p.err)) bad = true;
                hpar ^= 1u;
                const bool miss = group_sums(hh, U, I, ngI, gsum_s) && !bad;
                if (!__syncthreads_or(miss)) break;
                // rare: copy again (bounded like every wait; the generic reads of
                // the old copy are ordered before it by the barrier above)
                if (tid == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (t_retry == 0) t_retry = now;
                    if (now - t_retry > lim || ld_relaxed(abortw) != 0u) {
                        atomicExch(abortw, 1u);
                        set_error(p.err, SMOE_DEV_TIMEOUT);
                        *giveup_s = 1;
                    } else {
                        __nanosleep(100);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        copy_h();
                    }
                }
                __syncthreads();
                if (*giveup_s) {
                    bad = true;
                    break;
                }
            }
            const uint32_t vmask = *vmask_s;
            const int na = U * ngI, nj = (na - warp + kStkWarps - 1) / kStkWarps;   // this warp's atoms
            for (int j = 0; j < nj; j += 2) {
                const bool two = j + 1 < nj;
                const int a0 = warp + kStkWarps * j, a1 = two ? a0 + kStkWarps : a0;
                const int u0 = a0 / ngI, u1 = a1 / ngI;
                if (!bad && !mbar_wait(&dbar[u0], par, p.err)) bad = true;
                if (two && !bad && !mbar_wait(&dbar[u1], par, p.err)) bad = true;
                uint4 h[4];                                          // atom 0: h0 h1, atom 1: h0 h1
#pragma unroll
                for (int q = 0; q < 4; ++q) h[q] = make_uint4(0, 0, 0, 0);
                if (lane < 8) {                  // B columns 0 (high parts, lanes 0..3) and 1 (low parts, 4..7)
                    const int part = lane >> 2, t4 = lane & 3;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int a = q < 2 ? a0 : a1;
                        h[q] = *reinterpret_cast<const uint4 *>(hh + (size_t(part) * U + a / ngI) * I +
                                                                (a % ngI) * kGroup + 16 * t4 + 8 * (q & 1));
                    }
                }
                // both atoms unconditionally (the second repeats the first when this
                // warp has an odd count; a result not needed is dropped), so the two
                // chains always overlap
                float2 y0 = down_atom<BITS>(wdn + size_t(u0) * wbytes + (a0 % ngI) * AB, h[0], h[1], gsum_s[a0], lane);
                float2 y1 = down_atom<BITS>(wdn + size_t(u1) * wbytes + (a1 % ngI) * AB, h[2], h[3], gsum_s[a1], lane);
                if (!(vmask >> u0 & 1u) || bad) y0 = make_float2(0.f, 0.f);
                if (!(vmask >> u1 & 1u) || bad) y1 = make_float2(0.f, 0.f);
                if ((lane & 3) == 0) {
                    yd[a0 * 16 + (lane >> 2)] = y0.x;
                    yd[a0 * 16 + (lane >> 2) + 8] = y0.y;
                    if (two) {
                        yd[a1 * 16 + (lane >> 2)] = y1.x;
                        yd[a1 * 16 + (lane >> 2) + 8] = y1.y;
                    }
                }
            }
            __syncthreads();
            if (!kRing && tid == 0 && l + 1 < p.n_layers) {         // the shared down rows are read
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_shared_down(l + 1);
            }
            if (tid < U * 16) {                                      // expert u, row r: its groups in order
                const int u = tid >> 4, r = tid & 15;
                float s = 0.f;
                for (int kb = 0; kb < ngI; ++kb) s += yd[(u * ngI + kb) * 16 + r];
                ysum[tid] = s;
            }
            __syncthreads();
            if (tid < 16) {
                const int row = 16 * c + tid;
                float acc = 0.f;
                for (int j = 0; j < k; ++j) acc = fmaf(w_s[j], ysum[(j + 1) * 16 + tid], acc);
                acc = fmaf(*gate_s, ysum[tid], acc);
                acc += __uint_as_float(uint32_t(x_s[row]) << 16);
                const uint16_t o = f32_to_bf16_bits(acc);
                p.xs[size_t(l + 1) * H + row] = o;
                st_relaxed_u16(p.xe + size_t(l + 1) * H + row, canon16(o));
            }
        }
        // the next layer's copies overwrite regions read through the generic proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
    }
}

// ---------------------------------------------------------------------- host

template <int BITS>
static const void *stack_kernel_for(int ngI)
{
    switch (ngI) {
    case 1: return reinterpret_cast<const void *>(&decode_stack_kernel<1, BITS>);
    case 2: return reinterpret_cast<const void *>(&decode_stack_kernel<2, BITS>);
    case 4: return reinterpret_cast<const void *>(&decode_stack_kernel<4, BITS>);
    default: return reinterpret_cast<const void *>(&decode_stack_kernel<8, BITS>);
    }
}

cudaError_t stack_config(smoe_ctx *ctx)
{
    StackCfg &c = ctx->stack;
    c = StackCfg();
    const smoe_shape &s = ctx->shape;
    int coop = 0, max_smem = 0;
    cudaError_t e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, ctx->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device);
    if (e != cudaSuccess) return e;
    c.grid = ctx->num_sms;
    c.U = s.k + 1;
    c.nr = (s.E + 1 + c.grid - 1) / c.grid;
    c.nu = (s.k * (s.I / 8) + c.grid - 1) / c.grid;
    // most units (routed, plus the shared one where the CTA has it) of one CTA,
    // with the kernel's order of the routed units
    const int nD = s.H / 16, nrb = s.I / 8, R = s.k * nrb;
    c.nslot = 0;
    for (int b = 0; b < c.grid; ++b) {
        const int ord = b >= nD ? b - nD : (nD - 1 - b) + (c.grid - nD);
        const int n = (ord < R ? (R - 1 - ord) / c.grid + 1 : 0) + (b < nrb ? 1 : 0);
        if (n > c.nslot) c.nslot = n;
    }
    c.smem = stk_smem(s.H, s.E, s.I, c.U, c.nr, c.nu, s.bits, c.nslot).total;
    const int ngI = s.I / kGroup;
    const bool ngi_ok = ngI == 1 || ngI == 2 || ngI == 4 || ngI == 8;
    c.ok = coop && ngi_ok && c.grid >= s.H / 16 && c.grid >= s.I / 8 && s.E % 4 == 0 && s.E <= kStkMaxE &&
           c.nu <= kStkWarps && c.smem <= max_smem && (s.bits == 4 || s.bits == 8);
    if (!c.ok) return cudaSuccess;
    const void *kern = s.bits == 8 ? stack_kernel_for<8>(ngI) : stack_kernel_for<4>(ngI);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, c.smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStkThreads, c.smem);
    if (e != cudaSuccess) return e;
    c.ok = per_sm >= 1;
    return cudaSuccess;
}

cudaError_t launch_stack(const smoe_ctx *ctx, const StackParams &p, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(p.sync, 0, p.sync_bytes, st);
    if (e == cudaSuccess) e = prof_record(ctx->nprof > 0 ? ctx->prof[0] : nullptr, st);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(ctx->stack.grid);
    lc.blockDim = dim3(kStkThreads);
    lc.dynamicSmemBytes = ctx->stack.smem;
    lc.stream = st;
    lc.attrs = at;
    lc.numAttrs = 1;
    const int ngI = p.I / kGroup;
    if (ctx->shape.bits == 8) {
        if (ngI == 1) e = cudaLaunchKernelEx(&lc, decode_stack_kernel<1, 8>, p);
        else if (ngI == 2) e = cudaLaunchKernelEx(&lc, decode_stack_kernel<2, 8>, p);
        else if (ngI == 4) e = cudaLaunchKernelEx(&lc, decode_stack_kernel<4, 8>, p);
        else e = cudaLaunchKernelEx(&lc, decode_stack_kernel<8, 8>, p);
    } else {
        if (ngI == 1) e = cudaLaunchKernelEx(&lc, decode_stack_kernel<1, 4>, p);
        else if (ngI == 2) e = cudaLaunchKernelEx(&lc, decode_stack_kernel<2, 4>, p);
        else if (ngI == 4) e = cudaLaunchKernelEx(&lc, decode_stack_kernel<4, 4>, p);
        else e = cudaLaunchKernelEx(&lc, decode_stack_kernel<8, 4>, p);
    }
    if (e == cudaSuccess) e = prof_record(ctx->nprof > 1 ? ctx->prof[1] : nullptr, st);
    return e;
}

}  // namespace smoe
