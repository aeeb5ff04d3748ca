// decode_stack.cu -- one decode step (one token) through a stack of MoE
// layers in a single persistent, cooperative launch: one CTA per SM for the
// whole step, the layers separated by three grid-wide arrival counters each
// instead of kernel boundaries. Per layer l:
//   1. x_l and this CTA's router rows (rows c, c + G, ...; row E is the
//      shared-gate vector) are bulk-copied into shared memory; the CTA's
//      logits go to the workspace; counter A.
//   2. Every CTA reads all E + 1 logits and computes the same top-k (by rank
//      among the few logits that can be chosen), renormalised weights and
//      shared gate (route_common.cuh's arithmetic); CTA 0 also writes them out.
//   3. Gate/up: work units (expert u, 16-row block rb: intermediates
//      8 rb .. 8 rb + 7, 32 contiguous atoms, one bulk copy) are spread over
//      all CTAs; SwiGLU values go to the workspace as bf16 high and low
//      parts with each unit's sum of them; counter B.
//   4. Down and combine: CTA c < H/16 owns output rows 16 c .. 16 c + 15. Its
//      down atoms of every expert were requested in step 3, so they stream in
//      with the gate/up weights; after counter B it reads all h, computes the
//      rows for every expert and writes x_{l+1} = bf16(x_l + sum_j w_j y_j
//      (route order) + gate y_shared); counter C.
// While layer l computes, layer l + 1's router rows and shared-expert blob
// are prefetched into L2. The per-atom arithmetic is the decode kernel's
// (bf16 (128 + q) fragments on m16n8k16 tensor-core steps, s and b - 128 s
// per group, h as bf16 hi + lo). Every wait is bounded: a grid-wide wait gives
// up after two seconds and raises an abort word that ends the others' waits.
// Pages: the per-token expert stream of a decode step and its fixed-stride
// blobs (xix.ai article, paragraphs on how it works); the shared expert and
// its gate (agentlenshq article, how expert streaming works).
#include "decode_common.cuh"
#include "route_common.cuh"

namespace smoe {

constexpr int kStkWarps = 16;
constexpr int kStkThreads = kStkWarps * 32;

struct StkSmem {
    int x_s, xsum, rows, zs, table, units, wdn, hps, hh, hl, hsum, yp, red, cand, ints, bars, total;
};

__host__ __device__ inline StkSmem stk_smem(int H, int E, int I, int U, int nr, int nu)
{
    StkSmem L;
    int o = 0;
    L.x_s = o;   o = align128(o + 2 * H + 16);
    L.xsum = o;  o = align128(o + (H / kGroup) * 4);
    L.rows = o;  o = align128(o + nr * H * 2);
    L.zs = o;    o = align128(o + (E + 1) * 4);
    L.table = o; o = align128(o + E * 4);
    L.units = o; o = align128(o + nu * (H / kGroup) * kAtomBytes);
    L.wdn = o;   o = align128(o + U * (I / kGroup) * kAtomBytes);
    L.hps = o;   o = align128(o + U * (I / 8) * 4);
    L.hh = o;    o = align128(o + U * (I + 8) * 2);
    L.hl = o;    o = align128(o + U * (I + 8) * 2);
    L.hsum = o;  o = align128(o + U * (I / kGroup) * kDecodeMaxT * 4);
    L.yp = o;    o = align128(o + U * 2 * 16 * 4);
    L.red = o;   o = align128(o + nu * kStkWarps * 8 * 8);
    L.cand = o;  o = align128(o + (2 * E + 2 * 16 + 2 * 16) * 4);
    L.ints = o;  o = align128(o + 64 * 4);
    L.bars = o;  o = align128(o + (nu + U + 3) * 8);
    L.total = o;
    return L;
}

__device__ __forceinline__ void bulk_nohint(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void prefetch_l2_bytes(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Thread 0 waits until *ctr >= target (limit_ns at most, two seconds by default, or until another
// CTA raised the abort word), then the CTA synchronises. The counter is polled
// with relaxed loads, one in flight at a time and spaced by a short sleep (the
// abort word and the clock every 16 polls), and an acquire fence then orders what the arrivals
// released before this CTA's reads. Returns false if the wait gave up; the
// results of the step are then garbage and the error word says so, but every
// CTA still runs to the end.
__device__ bool grid_wait(const uint32_t *ctr, uint32_t target, uint32_t *abortw, int32_t *err, int *flag_s,
                          uint64_t limit_ns)
{
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint64_t t0 = global_ns();
        for (uint32_t it = 1; ld_relaxed(ctr) < target; ++it) {
            __nanosleep(32);                     // polls spaced out: the arrivals hit the same line
            if ((it & 15) == 0) {
                if (ld_relaxed(abortw)) { ok = 0; break; }
                if (global_ns() - t0 > limit_ns) {
                    atomicExch(abortw, 1u);
                    set_error(err, SMOE_DEV_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        asm volatile("fence.proxy.async.global;" ::: "memory");   // later bulk copies read what we acquired
        *flag_s = ok;
    }
    __syncthreads();
    return *flag_s != 0;
}

// Composite order of the routing keys: larger key first, equal keys by lower id.
__device__ __forceinline__ bool key_before(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(kStkThreads, 1) decode_stack_kernel(const __grid_constant__ StackParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = p.H, E = p.E, k = p.k, I = p.I, U = p.U;
    const int ngH = H / kGroup, ngI = I / kGroup, nrb = I / 8, nrbB = H / 16;
    const uint32_t ubytes = uint32_t(ngH * kAtomBytes), wbytes = uint32_t(ngI * kAtomBytes);
    const uint64_t down_off = uint64_t(I / 8) * ngH * kAtomBytes;
    const StkSmem L = stk_smem(H, E, I, U, p.nr, p.nu);
    uint16_t *x_s = reinterpret_cast<uint16_t *>(smem + L.x_s);
    float *xsum = reinterpret_cast<float *>(smem + L.xsum);
    uint16_t *rows = reinterpret_cast<uint16_t *>(smem + L.rows);
    float *zs = reinterpret_cast<float *>(smem + L.zs);
    int *table = reinterpret_cast<int *>(smem + L.table);
    uint8_t *units = smem + L.units;
    uint8_t *wdn = smem + L.wdn;
    float *hps = reinterpret_cast<float *>(smem + L.hps);
    uint16_t *hh = reinterpret_cast<uint16_t *>(smem + L.hh);
    uint16_t *hl = reinterpret_cast<uint16_t *>(smem + L.hl);
    float *hsum = reinterpret_cast<float *>(smem + L.hsum);
    float *yp = reinterpret_cast<float *>(smem + L.yp);
    float2 *red = reinterpret_cast<float2 *>(smem + L.red);     // [nu][warps][8] gate/up partial sums
    uint32_t *cand_k = reinterpret_cast<uint32_t *>(smem + L.cand);   // [E] candidates
    int32_t *cand_i = reinterpret_cast<int32_t *>(cand_k + E);
    uint32_t *mx_k = reinterpret_cast<uint32_t *>(cand_i + E);        // [16] slice maxima
    int32_t *mx_i = reinterpret_cast<int32_t *>(mx_k + 16);
    uint32_t *sel_k = reinterpret_cast<uint32_t *>(mx_i + 16);        // [16] chosen, in route order
    int32_t *sel_i = reinterpret_cast<int32_t *>(sel_k + 16);
    int *ints = reinterpret_cast<int *>(smem + L.ints);
    int *ids_s = ints;                  // [16] route order
    float *w_s = reinterpret_cast<float *>(ints + 16);   // [16]
    float *gate_s = reinterpret_cast<float *>(ints + 32);
    int *flag_s = ints + 33;
    int *ncand = ints + 34;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *ubar = bars, *dbar = bars + p.nu, *xbar = dbar + U, *rbar = xbar + 1, *hbar = rbar + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int G = int(gridDim.x), c = int(blockIdx.x);
    uint32_t *abortw = p.sync + 3 * p.n_layers;
    const int nr_mine = c <= E ? (E - c) / G + 1 : 0;           // router rows c, c + G, ... <= E

    if (tid == 0) {
        for (int i = 0; i < p.nu + U + 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    bool bad = false;                    // this thread's bounded mbarrier wait gave up

    for (int l = 0; l < p.n_layers; ++l) {
        const uint32_t par = uint32_t(l & 1);
        uint32_t *cnt = p.sync + 3 * l;
        const uint8_t *shared = p.shared[l];
        auto blob_of = [&](int u) -> const uint8_t * {
            if (u == 0) return shared;
            const int64_t slot = table[ids_s[u - 1]];
            if (slot < 0 || slot >= p.n_slots) return nullptr;
            return p.pool + uint64_t(slot) * p.stride;
        };

        // ---- 1. x_l, router rows, slot table row; logits of this CTA's rows
        if (l > 0) grid_wait(p.sync + 3 * (l - 1) + 2, uint32_t(nrbB), abortw, p.err, flag_s, p.wait_ns);
        if (tid == 0) {
            mbar_arrive_expect_tx(xbar, uint32_t(H * 2));
            bulk_nohint(x_s, p.xs + size_t(l) * H, uint32_t(H * 2), xbar);
            mbar_arrive_expect_tx(rbar, uint32_t(nr_mine * H * 2 + E * 4));
            for (int j = 0; j < nr_mine; ++j) {
                const int r = c + j * G;
                bulk_nohint(rows + size_t(j) * H, r < E ? p.Wr[l] + size_t(r) * H : p.ws[l], uint32_t(H * 2), rbar);
            }
            bulk_nohint(table, p.table + size_t(l) * E, uint32_t(E * 4), rbar);
        }
        if (!bad && !mbar_wait(xbar, par, p.err)) bad = true;
        if (!bad && !mbar_wait(rbar, par, p.err)) bad = true;
        for (int j = warp; j < nr_mine; j += kStkWarps) {
            const float z = router_dot(rows + size_t(j) * H, x_s, H, lane);
            if (lane == 0) __stcg(p.logits + size_t(l) * (E + 1) + c + j * G, z);
        }
        for (int grp = warp; grp < ngH; grp += kStkWarps) {          // per-group sums of x (bias term)
            const uint32_t v = *reinterpret_cast<const uint32_t *>(x_s + grp * kGroup + 2 * lane);
            float s = bf16lo(v) + bf16hi(v);
            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) xsum[grp] = s;
        }
        __syncthreads();
        if (tid == 0) ticket_add(&cnt[0], 1u);

        // ---- 2. routing, redundantly in every CTA. Warp w holds the keys of slice
        // w (E / 16 logits); the k-th largest of the 16 slice maxima bounds the
        // k-th largest key from below (k distinct keys reach it), so only keys at
        // or above it can be chosen. Each such candidate's rank among the
        // candidates (larger key first, ties to the lower id) is its place in
        // route order.
        // (the failure-detection test hook asks for one arrival more than there are CTAs)
        grid_wait(&cnt[0], uint32_t(G) + (l == p.stall_layer ? 1u : 0u), abortw, p.err, flag_s, p.wait_ns);
        for (int e = tid; e <= E; e += kStkThreads) zs[e] = __ldcg(p.logits + size_t(l) * (E + 1) + e);
        if (tid == 0) *ncand = 0;
        __syncthreads();
        {
            const int spw = (E + kStkWarps - 1) / kStkWarps;        // keys per slice (<= 64)
            uint32_t kk[2];
            int32_t ki[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int j = lane + 32 * h2, e = warp * spw + j;
                const bool in = j < spw && e < E;
                kk[h2] = in ? fkey(zs[e] + (p.bias ? p.bias[e] : 0.f)) : 0u;
                ki[h2] = in ? e : 0x7fffffff;
            }
            const bool second = key_before(kk[1], ki[1], kk[0], ki[0]);
            const uint32_t bk = second ? kk[1] : kk[0];
            const int32_t bi = second ? ki[1] : ki[0];
            const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
            const int32_t mi = int32_t(__reduce_min_sync(0xffffffffu, uint32_t(bk == mk ? bi : 0x7fffffff)));
            if (lane == 0) {
                mx_k[warp] = mk;
                mx_i[warp] = mi;
            }
            __syncthreads();
            // the k-th largest slice maximum (k <= 16 slices): the one with rank k - 1
            int rank = 0;
            if (lane < kStkWarps)
                for (int j = 0; j < kStkWarps; ++j) rank += key_before(mx_k[j], mx_i[j], mx_k[lane], mx_i[lane]);
            // (fewer than k slices with keys: no such rank; then every key is a candidate)
            const int tl = __ffs(__ballot_sync(0xffffffffu, lane < kStkWarps && rank == k - 1)) - 1;
            const uint32_t t_k = tl >= 0 ? mx_k[tl] : 0u;
            const int32_t t_i = tl >= 0 ? mx_i[tl] : 0x7fffffff;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
                if (kk[h2] != 0u && !key_before(t_k, t_i, kk[h2], ki[h2])) {
                    const int pos = atomicAdd(ncand, 1);
                    cand_k[pos] = kk[h2];
                    cand_i[pos] = ki[h2];
                }
            __syncthreads();
            const int n = *ncand;
            for (int q = tid; q < n; q += kStkThreads) {
                const uint32_t ck = cand_k[q];
                const int32_t ci = cand_i[q];
                int r = 0;
                for (int j = 0; j < n; ++j) r += key_before(cand_k[j], cand_i[j], ck, ci);
                if (r < k) {
                    sel_k[r] = ck;
                    sel_i[r] = ci;
                }
            }
            __syncthreads();
        }
        if (warp == 0) {
            const float wl = choice_weight(sel_k, k, lane);
            if (lane < k) {
                ids_s[lane] = sel_i[lane];
                w_s[lane] = wl;
                if (c == 0) {
                    p.ids[size_t(l) * k + lane] = sel_i[lane];
                    p.w[size_t(l) * k + lane] = wl;
                }
            }
            if (lane == 0) {
                *gate_s = shared_gate(zs[E]);
                if (c == 0) p.gate[l] = *gate_s;
            }
        }
        __syncthreads();

        // ---- 3. request this layer's weights (one bulk copy per lane 0 of a warp,
        // so the copies issue in parallel); prefetch the next layer's fixed ones into L2
        if (lane == 0) {
            const int nd = c < nrbB ? U : 0;
            for (int it = warp; it < p.nu + nd; it += kStkWarps) {
                if (it < p.nu) {
                    const int q = c + it * G, u = q / nrb;
                    if (u >= U) continue;
                    const uint8_t *blob = blob_of(u);
                    if (blob) {
                        mbar_arrive_expect_tx(&ubar[it], ubytes);
                        bulk_g2s(units + size_t(it) * ubytes, blob + size_t(q % nrb) * ubytes, ubytes, &ubar[it], pol);
                    } else {
                        set_error(p.err, SMOE_DEV_BAD_SLOT);
                        mbar_arrive(&ubar[it]);
                    }
                } else {
                    const int u = it - p.nu;
                    const uint8_t *blob = blob_of(u);
                    if (blob) {
                        mbar_arrive_expect_tx(&dbar[u], wbytes);
                        bulk_g2s(wdn + size_t(u) * wbytes, blob + down_off + size_t(c) * wbytes, wbytes, &dbar[u], pol);
                    } else {
                        mbar_arrive(&dbar[u]);
                    }
                }
            }
            if (warp == kStkWarps - 1 && l + 1 < p.n_layers) {
                for (int j = 0; j < nr_mine; ++j) {
                    const int r = c + j * G;
                    prefetch_l2_bytes(r < E ? p.Wr[l + 1] + size_t(r) * H : p.ws[l + 1], uint32_t(H * 2));
                }
                for (int i = 0; i < p.nu; ++i) {
                    const int q = c + i * G;
                    if (q < nrb) prefetch_l2_bytes(p.shared[l + 1] + size_t(q) * ubytes, ubytes);
                }
                if (c < nrbB) prefetch_l2_bytes(p.shared[l + 1] + down_off + size_t(c) * wbytes, wbytes);
            }
        }

        // ---- 4. gate/up units -> h. Each warp takes atoms kb = warp, warp + 16, ...
        // of the CTA's units one after another, with no CTA barrier between units.
        // The token is MMA column 0, so lanes 4 g (t4 = 0) hold the partial sums of
        // rows g (gate) and g + 8 (up); they go to red[unit][warp][g]. After one
        // barrier warp i reduces unit i over the warps in order.
        int n_mine = 0;                                             // this CTA's units (uniform)
        for (int i = 0; i < p.nu; ++i) {
            const int q = c + i * G, u = q / nrb;
            if (u >= U) break;                                      // uniform
            ++n_mine;
            const bool valid = blob_of(u) != nullptr;               // uniform
            if (!bad && !mbar_wait(&ubar[i], par, p.err)) bad = true;
            float aG = 0.f, aU = 0.f;
            if (valid && !bad) {
                const uint8_t *ubase = units + size_t(i) * ubytes;
                for (int kb = warp; kb < ngH; kb += kStkWarps) {
                    const uint8_t *atom = ubase + kb * kAtomBytes;
                    const uint4 A = *reinterpret_cast<const uint4 *>(atom + 16 * lane);
                    const uint2 SB = *reinterpret_cast<const uint2 *>(atom + kAtomQBytes + 8 * g);
                    const int col = kb * kGroup + 16 * t4;
                    uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
                    if (g == 0) {                                   // the token is MMA column 0
                        xa = *reinterpret_cast<const uint4 *>(x_s + col);
                        xb = *reinterpret_cast<const uint4 *>(x_s + col + 8);
                    }
                    const uint32_t xl[4] = {xa.x, xa.y, xa.z, xa.w}, xr[4] = {xb.x, xb.y, xb.z, xb.w};
                    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int m = 0; m < 4; m += 2) {
                        const uint32_t a0[4] = {nib_pair(A.x, m), nib_pair(A.z, m), nib_pair(A.y, m), nib_pair(A.w, m)};
                        const uint32_t a1[4] = {nib_pair(A.x, m + 1), nib_pair(A.z, m + 1), nib_pair(A.y, m + 1),
                                                nib_pair(A.w, m + 1)};
                        mma_bf16(acc, a0, xl[m], xr[m]);
                        mma_bf16(acc2, a1, xl[m + 1], xr[m + 1]);
                    }
                    float sg, bpg, su, bpu;
                    scale_bias(SB.x, sg, bpg);
                    scale_bias(SB.y, su, bpu);
                    aG += fmaf(sg, acc[0] + acc2[0], bpg * xsum[kb]);
                    aU += fmaf(su, acc[2] + acc2[2], bpu * xsum[kb]);
                }
            }
            if (t4 == 0) red[(i * kStkWarps + warp) * 8 + g] = make_float2(aG, aU);
        }
        __syncthreads();
        if (warp < n_mine) {
            const int i = warp, q = c + i * G, u = q / nrb, rb = q % nrb;
            const bool valid = blob_of(u) != nullptr;
            const float2 *ri = red + i * kStkWarps * 8 + g;
            float aG = ri[0].x, aU = ri[0].y;
#pragma unroll
            for (int w = 1; w < kStkWarps; ++w) {
                const float2 v = ri[w * 8];
                aG += v.x;
                aU += v.y;
            }
            // intermediate 8 rb + g (the four lanes of a g hold the same sums). h goes
            // out as bf16 hi and lo = bf16(h - hi), with the unit's sum of hi + lo over
            // its 8 intermediates (the down rows' bias term)
            const float hv = (valid && !bad) ? silu(aG) * aU : 0.f;
            const uint16_t hi = f32_to_bf16_bits(hv);
            const uint16_t lo = f32_to_bf16_bits(hv - __uint_as_float(uint32_t(hi) << 16));
            float sum = __uint_as_float(uint32_t(hi) << 16) + __uint_as_float(uint32_t(lo) << 16);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            uint16_t *hrow = p.h + (size_t(l) * 2 * U + u) * I;
            if (t4 == 0) {
                __stcg(hrow + 8 * rb + g, hi);
                __stcg(hrow + size_t(U) * I + 8 * rb + g, lo);
            }
            if (lane == 0) __stcg(p.hps + (size_t(l) * U + u) * nrb + rb, sum);
        }
        __syncthreads();
        if (tid == 0) ticket_add(&cnt[1], 1u);

        // ---- 5. down rows of every expert for rows 16 c .. 16 c + 15, combine
        if (c < nrbB) {
            grid_wait(&cnt[1], uint32_t(G), abortw, p.err, flag_s, p.wait_ns);
            // h rows of every expert (hi, lo; padded rows), and the unit sums: one bulk
            // copy per lane of warp 0
            if (warp == 0) {
                if (lane == 0) mbar_arrive_expect_tx(hbar, uint32_t(U * I * 4 + U * nrb * 4));
                __syncwarp();
                const uint16_t *hl_src = p.h + size_t(l) * 2 * U * I;
                for (int j = lane; j < 2 * U + 1; j += 32) {
                    if (j < U)
                        bulk_nohint(hh + j * (I + 8), hl_src + size_t(j) * I, uint32_t(I * 2), hbar);
                    else if (j < 2 * U)
                        bulk_nohint(hl + (j - U) * (I + 8), hl_src + size_t(U + (j - U)) * I, uint32_t(I * 2), hbar);
                    else
                        bulk_nohint(hps, p.hps + size_t(l) * U * nrb, uint32_t(U * nrb * 4), hbar);
                }
            }
            if (!bad && !mbar_wait(hbar, par, p.err)) bad = true;
            for (int it = tid; it < U * ngI; it += kStkThreads) {   // group sums: the 8 unit sums in order
                const float *ps = hps + it * 8;
                float s2 = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) s2 += ps[j];
                hsum[it * kDecodeMaxT] = s2;
            }
            __syncthreads();
            const int nkh = ngI >= 2 ? 2 : 1;
            for (int it = warp; it < U * nkh; it += kStkWarps) {
                const int u = it / nkh, kh = it % nkh;
                const int kbeg = kh * (ngI / nkh), kend = kh + 1 == nkh ? ngI : kbeg + ngI / nkh;
                const bool valid = blob_of(u) != nullptr;
                float y[4] = {0.f, 0.f, 0.f, 0.f};
                if (!bad && !mbar_wait(&dbar[u], par, p.err)) bad = true;
                if (valid && !bad)
                    down_rows(wdn + size_t(u) * wbytes, 0, ngI, kbeg, kend, hh + u * (I + 8), hl + u * (I + 8),
                              hsum + u * ngI * kDecodeMaxT, I, 1, lane, y);
                if (t4 == 0) {                                       // token = column 0
                    yp[(u * 2 + kh) * 16 + g] = y[0];
                    yp[(u * 2 + kh) * 16 + g + 8] = y[2];
                }
            }
            if (nkh == 1)
                for (int i = tid; i < U * 16; i += kStkThreads) yp[((i / 16) * 2 + 1) * 16 + i % 16] = 0.f;
            __syncthreads();
            if (tid < 16) {
                const int row = 16 * c + tid;
                auto yv = [&](int u) { return yp[(u * 2) * 16 + tid] + yp[(u * 2 + 1) * 16 + tid]; };
                float acc = 0.f;
                for (int j = 0; j < k; ++j) acc = fmaf(w_s[j], yv(j + 1), acc);
                acc = fmaf(*gate_s, yv(0), acc);
                acc += __uint_as_float(uint32_t(x_s[row]) << 16);
                p.xs[size_t(l + 1) * H + row] = f32_to_bf16_bits(acc);
            }
            __syncthreads();
            if (tid == 0) ticket_add(&cnt[2], 1u);
        }
    }
}

// ---------------------------------------------------------------------- host

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
    c.nu = (c.U * (s.I / 8) + c.grid - 1) / c.grid;
    c.smem = stk_smem(s.H, s.E, s.I, c.U, c.nr, c.nu).total;
    c.ok = coop && c.grid >= s.H / 16 && s.E % 4 == 0 && c.nu <= kStkWarps && c.smem <= max_smem;
    if (!c.ok) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_stack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, c.smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_stack_kernel, kStkThreads, c.smem);
    if (e != cudaSuccess) return e;
    c.ok = per_sm >= 1;
    return cudaSuccess;
}

cudaError_t launch_stack(const smoe_ctx *ctx, const StackParams &p, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(p.sync, 0, size_t(3 * p.n_layers + 1) * 4, st);
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
    e = cudaLaunchKernelEx(&lc, decode_stack_kernel, p);
    if (e == cudaSuccess) e = prof_record(ctx->nprof > 1 ? ctx->prof[1] : nullptr, st);
    return e;
}

}  // namespace smoe
