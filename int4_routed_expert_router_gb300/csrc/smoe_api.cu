// smoe_api.cu -- the C ABI declared in include/smoe.h: blob layout, packing of
// MLX triples into fixed-stride blobs, context and slot table, workspace
// carving, and dispatch of the router / expert kernels.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "smoe_dev.cuh"
#include "smoe_internal.h"

using namespace smoe;

namespace smoe {

// ------------------------------------------------------------------ packing
// Blob word for MLX word mw (columns c0..c0+7 of one row, column c0+j in bits
// 4j..4j+3): column c0+2m goes to bits 4m.., column c0+2m+1 to bits 16+4m..
__host__ __device__ inline uint32_t blob_word(uint32_t mw)
{
    uint32_t out = 0;
    for (int m = 0; m < 4; ++m) {
        out |= ((mw >> (8 * m)) & 0xFu) << (4 * m);
        out |= ((mw >> (8 * m + 4)) & 0xFu) << (16 + 4 * m);
    }
    return out;
}

// Source (matrix, row) of logical row lr (0..15) of atom row block rb.
__host__ __device__ inline void atom_row(bool down, int rb, int lr, int *mat, int *row)
{
    if (!down) {
        *mat = lr < 8 ? 0 : 1;            // gate rows then up rows
        *row = 8 * rb + (lr & 7);
    } else {
        *mat = 2;
        *row = 16 * rb + lr;
    }
}

// The 16 bytes of lane L of atom (part, rb, kb).
__host__ __device__ inline uint4 atom_lane(const smoe_expert_src &src, int H, int I, bool down, int rb, int kb,
                                           int L)
{
    const int g = L >> 2, t = L & 3;
    const int wpr = down ? I / 8 : H / 8;
    const int w0 = kb * 8 + 2 * t;     // MLX word of columns kb*64 + 16t ..
    uint32_t out[4];
    for (int half = 0; half < 2; ++half) {     // row g, row g+8
        int mat, row;
        atom_row(down, rb, g + 8 * half, &mat, &row);
        const uint32_t *q = src.q[mat] + size_t(row) * wpr;
        out[2 * half] = blob_word(q[w0]);
        out[2 * half + 1] = blob_word(q[w0 + 1]);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// The 8 bytes (s_g, b_g, s_g8, b_g8) of scale entry g of atom (part, rb, kb).
__host__ __device__ inline uint2 atom_sb(const smoe_expert_src &src, int H, int I, bool down, int rb, int kb, int g)
{
    const int gpr = down ? I / kGroup : H / kGroup;
    uint32_t v[2];
    for (int half = 0; half < 2; ++half) {
        int mat, row;
        atom_row(down, rb, g + 8 * half, &mat, &row);
        const size_t i = size_t(row) * gpr + kb;
        v[half] = uint32_t(src.s[mat][i]) | (uint32_t(src.b[mat][i]) << 16);
    }
    return make_uint2(v[0], v[1]);
}

void pack_host(const smoe_shape &s, const smoe_expert_src &src, uint8_t *dst)
{
    const Layout L = layout_of(s.H, s.I);
    for (int part = 0; part < 2; ++part) {
        const bool down = part == 1;
        const int nrb = down ? s.H / 16 : s.I / 8, nkb = down ? s.I / kGroup : s.H / kGroup;
        uint8_t *base = dst + (down ? L.down_off : L.gu_off);
        for (int rb = 0; rb < nrb; ++rb)
            for (int kb = 0; kb < nkb; ++kb) {
                uint8_t *atom = base + (size_t(rb) * nkb + kb) * kAtomBytes;
                for (int lane = 0; lane < 32; ++lane) {
                    const uint4 v = atom_lane(src, s.H, s.I, down, rb, kb, lane);
                    std::memcpy(atom + 16 * lane, &v, 16);
                }
                for (int g = 0; g < 8; ++g) {
                    const uint2 v = atom_sb(src, s.H, s.I, down, rb, kb, g);
                    std::memcpy(atom + kAtomQBytes + 8 * g, &v, 8);
                }
            }
    }
}

// ------------------------------------------------------ 8-bit experts (host)
// MLX's 8-bit affine format (4 values per uint32, column c of a row in bits
// 8 (c % 4) ..) packs into atoms of the same 16 rows x 64 columns that hold
// each value's low nibble in plane 0 and its high nibble in plane 1, each
// plane in the 4-bit atom's lane order, then the same 64 bytes of (s, b): so
// q = lo + 16 hi, and a kernel that reads 4-bit atoms reads each plane as
// one. The pages name int4/int8 group quantisation ("Swiftlet Packs 80B Qwen
// Into Mac...", last paragraph). The layout, the host and device packers and
// the plain debug path take 8-bit experts; the fast expert kernels do not.

Layout layout8_of(int H, int I)
{
    Layout L;
    L.gu_off = 0;
    L.gu_bytes = uint64_t(I / 8) * (H / kGroup) * kAtom8Bytes;
    L.down_off = L.gu_bytes;
    L.down_bytes = uint64_t(H / 16) * (I / kGroup) * kAtom8Bytes;
    L.blob = L.gu_bytes + L.down_bytes;
    return L;
}

// The 4-bit-format word of 8 consecutive columns (column c0 + j in bits
// 4j ..) made of one nibble plane of the 8-bit words w0 (columns c0 ..
// c0 + 3) and w1 (c0 + 4 .. c0 + 7): plane 0 the low nibbles, plane 1 the high.
__host__ __device__ inline uint32_t plane_word(uint32_t w0, uint32_t w1, int plane)
{
    uint32_t out = 0;
    for (int j = 0; j < 8; ++j) {
        const uint32_t v = ((j < 4 ? w0 : w1) >> (8 * (j & 3))) & 0xFFu;
        out |= ((v >> (4 * plane)) & 0xFu) << (4 * j);
    }
    return out;
}

// Lane L of nibble plane `plane` of 8-bit atom (part, rb, kb).
__host__ __device__ inline uint4 atom_lane8(const smoe_expert_src &src, int H, int I, bool down, int rb, int kb,
                                            int L, int plane)
{
    const int g = L >> 2, t = L & 3;
    const int wpr = down ? I / 4 : H / 4;
    const int w0 = kb * 16 + 4 * t;    // 8-bit MLX word of columns kb*64 + 16t ..
    uint32_t out[4];
    for (int half = 0; half < 2; ++half) {     // row g, row g+8
        int mat, row;
        atom_row(down, rb, g + 8 * half, &mat, &row);
        const uint32_t *q = src.q[mat] + size_t(row) * wpr;
        out[2 * half] = blob_word(plane_word(q[w0], q[w0 + 1], plane));
        out[2 * half + 1] = blob_word(plane_word(q[w0 + 2], q[w0 + 3], plane));
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

void pack_host8(const smoe_shape &s, const smoe_expert_src &src, uint8_t *dst)
{
    const Layout L = layout8_of(s.H, s.I);
    for (int part = 0; part < 2; ++part) {
        const bool down = part == 1;
        const int nrb = down ? s.H / 16 : s.I / 8, nkb = down ? s.I / kGroup : s.H / kGroup;
        uint8_t *base = dst + (down ? L.down_off : L.gu_off);
        for (int rb = 0; rb < nrb; ++rb)
            for (int kb = 0; kb < nkb; ++kb) {
                uint8_t *atom = base + (size_t(rb) * nkb + kb) * kAtom8Bytes;
                for (int plane = 0; plane < 2; ++plane)
                    for (int lane = 0; lane < 32; ++lane) {
                        const uint4 v = atom_lane8(src, s.H, s.I, down, rb, kb, lane, plane);
                        std::memcpy(atom + kAtomQBytes * plane + 16 * lane, &v, 16);
                    }
                for (int g = 0; g < 8; ++g) {
                    const uint2 v = atom_sb(src, s.H, s.I, down, rb, kb, g);
                    std::memcpy(atom + 2 * kAtomQBytes + 8 * g, &v, 8);
                }
            }
    }
}

// One thread per (atom, lane): 16 bytes of nibbles, and for lanes < 8 the 8
// bytes of scales/biases.
__global__ void pack_kernel(const smoe_expert_src src, int H, int I, uint8_t *dst, uint64_t down_off,
                            long long n_gu_atoms, long long n_atoms)
{
    const long long total = n_atoms * 32;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long a = i >> 5;
        const int lane = int(i & 31);
        const bool down = a >= n_gu_atoms;
        const long long ai = down ? a - n_gu_atoms : a;
        const int nkb = down ? I / kGroup : H / kGroup;
        const int rb = int(ai / nkb), kb = int(ai % nkb);
        uint8_t *atom = dst + (down ? down_off : 0) + ai * kAtomBytes;
        *reinterpret_cast<uint4 *>(atom + 16 * lane) = atom_lane(src, H, I, down, rb, kb, lane);
        if (lane < 8) *reinterpret_cast<uint2 *>(atom + kAtomQBytes + 8 * lane) = atom_sb(src, H, I, down, rb, kb, lane);
    }
}

// 8-bit: one thread per (atom, plane, lane): 16 bytes of that plane's
// nibbles, and for plane 0, lanes < 8 the 8 bytes of scales/biases.
__global__ void pack_kernel8(const smoe_expert_src src, int H, int I, uint8_t *dst, uint64_t down_off,
                             long long n_gu_atoms, long long n_atoms)
{
    const long long total = n_atoms * 64;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long a = i >> 6;
        const int plane = int((i >> 5) & 1), lane = int(i & 31);
        const bool down = a >= n_gu_atoms;
        const long long ai = down ? a - n_gu_atoms : a;
        const int nkb = down ? I / kGroup : H / kGroup;
        const int rb = int(ai / nkb), kb = int(ai % nkb);
        uint8_t *atom = dst + (down ? down_off : 0) + ai * kAtom8Bytes;
        *reinterpret_cast<uint4 *>(atom + kAtomQBytes * plane + 16 * lane) =
            atom_lane8(src, H, I, down, rb, kb, lane, plane);
        if (plane == 0 && lane < 8)
            *reinterpret_cast<uint2 *>(atom + 2 * kAtomQBytes + 8 * lane) = atom_sb(src, H, I, down, rb, kb, lane);
    }
}

cudaError_t launch_pack_device(const smoe_shape &s, const smoe_expert_src &src, uint8_t *dst, cudaStream_t st)
{
    if (s.bits == 8) {
        const Layout L8 = layout8_of(s.H, s.I);
        const long long ngu = (long long)(s.I / 8) * (s.H / kGroup);
        const long long nd = (long long)(s.H / 16) * (s.I / kGroup);
        const long long threads = (ngu + nd) * 64;
        const long long grid = (threads + 255) / 256;
        pack_kernel8<<<unsigned(grid < 65535 ? grid : 65535), 256, 0, st>>>(src, s.H, s.I, dst, L8.down_off, ngu,
                                                                            ngu + nd);
        return cudaGetLastError();
    }
    const Layout L = layout_of(s.H, s.I);
    const long long ngu = (long long)(s.I / 8) * (s.H / kGroup);
    const long long nd = (long long)(s.H / 16) * (s.I / kGroup);
    const long long threads = (ngu + nd) * 32;
    const int block = 256;
    const long long grid = (threads + block - 1) / block;
    pack_kernel<<<unsigned(grid < 65535 ? grid : 65535), block, 0, st>>>(src, s.H, s.I, dst, L.down_off, ngu,
                                                                         ngu + nd);
    return cudaGetLastError();
}

Workspace workspace_layout(const smoe_shape &s, int T)
{
    auto al = [](uint64_t v) { return (v + 255) & ~uint64_t(255); };
    Workspace w = {};
    uint64_t o = 0;
    w.route_counter = o; o = al(o + 64);
    w.fwd_counters = o;  o = al(o + 64 * 4);
    w.logits = o;        o = al(o + uint64_t(T) * (s.E + 1) * 4);
    if (T <= kDecodeMaxT) {
        const uint64_t umax = uint64_t(s.E < T * s.k ? s.E : T * s.k) + 1;
        w.ypair = o;     o = al(o + umax * T * s.H * 4);
    } else {
        const uint64_t P = uint64_t(T) * s.k, nch = (uint64_t(T) + bucket_tok(T) - 1) / bucket_tok(T);
        w.counts = o;     o = al(o + nch * s.E * 4);
        w.chunk_base = o; o = al(o + nch * s.E * 4);
        w.offsets = o;    o = al(o + (uint64_t(s.E) + 1) * 4);
        w.tiles = o;      o = al(o + uint64_t(prefill_max_tiles(T, s.k, s.E)) * sizeof(PfTile));
        w.ntiles = o;     o = al(o + 4);
        w.pair_token = o; o = al(o + P * 4);
        w.pair_pos = o;   o = al(o + P * 4);
        w.hbuf = o;       o = al(o + (P + T) * s.I * 2);
        w.ybuf = o;       o = al(o + (P + T) * s.H * 2);
        w.xt = o;         o = al(o + uint64_t(T) * s.H * 2);
    }
    w.total = o;
    return w;
}

}  // namespace smoe

// ====================================================================== C ABI
// allow8: the 8-bit format is accepted (layout, packing and contexts)
static int shape_check(const smoe_shape *s, bool allow8 = false)
{
    if (!s) return SMOE_EINVAL;
    if (s->group != 64 || !(s->bits == 4 || (allow8 && s->bits == 8))) return SMOE_ENOTSUP;
    if (s->H <= 0 || s->E <= 0 || s->k <= 0 || s->I <= 0) return SMOE_EINVAL;
    if (s->H % 256 || s->H > 2048) return SMOE_ENOTSUP;
    if (s->I % 64 || s->I < 64 || s->I > 512 || s->I_shared != s->I) return SMOE_ENOTSUP;
    if (s->k > 16 || s->k > s->E || s->E > 1024) return SMOE_ENOTSUP;
    return SMOE_OK;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? SMOE_OK : SMOE_ECUDA; }

extern "C" int smoe_layout_of(const smoe_shape *shape, smoe_layout *out)
{
    int rc = shape_check(shape, true);
    if (rc) return rc;
    if (!out) return SMOE_EINVAL;
    const bool b8 = shape->bits == 8;
    const Layout L = b8 ? layout8_of(shape->H, shape->I) : layout_of(shape->H, shape->I);
    out->blob_bytes = L.blob;
    out->gu_offset = L.gu_off;
    out->gu_bytes = L.gu_bytes;
    out->down_offset = L.down_off;
    out->down_bytes = L.down_bytes;
    out->atom_bytes = b8 ? kAtom8Bytes : kAtomBytes;
    out->atom_rows = kAtomRows;
    out->group = kGroup;
    out->reserved = 0;
    return SMOE_OK;
}

extern "C" int pack_experts(const smoe_shape *shape, const smoe_expert_src *src, int32_t n,
                            const int64_t *dst_slots, void *pool, uint64_t pool_bytes, int32_t where,
                            void *stream)
{
    int rc = shape_check(shape, true);
    if (rc) return rc;
    if (n < 0 || (n > 0 && (!src || !dst_slots || !pool))) return SMOE_EINVAL;
    if (where != SMOE_HOST && where != SMOE_DEVICE) return SMOE_EINVAL;
    const bool b8 = shape->bits == 8;
    const Layout L = b8 ? layout8_of(shape->H, shape->I) : layout_of(shape->H, shape->I);
    // the device packer stores 16-byte lanes at pool + slot * stride (the stride is a
    // whole number of 16-byte lanes); both packers read q as uint32 and s, b as fp16
    if (where == SMOE_DEVICE && (reinterpret_cast<uintptr_t>(pool) & 15)) return SMOE_EINVAL;
    for (int i = 0; i < n; ++i) {
        for (int m = 0; m < 3; ++m) {
            if (!src[i].q[m] || !src[i].s[m] || !src[i].b[m]) return SMOE_EINVAL;
            if ((reinterpret_cast<uintptr_t>(src[i].q[m]) & 3) || (reinterpret_cast<uintptr_t>(src[i].s[m]) & 1) ||
                (reinterpret_cast<uintptr_t>(src[i].b[m]) & 1))
                return SMOE_EINVAL;
        }
        if (dst_slots[i] < 0) return SMOE_ERANGE;
        const uint64_t end = (uint64_t(dst_slots[i]) + 1) * L.blob;
        if (end / L.blob != uint64_t(dst_slots[i]) + 1 || end > pool_bytes) return SMOE_ENOMEM;
    }
    uint8_t *base = static_cast<uint8_t *>(pool);
    for (int i = 0; i < n; ++i) {
        uint8_t *dst = base + uint64_t(dst_slots[i]) * L.blob;
        if (where == SMOE_HOST) {
            if (b8) pack_host8(*shape, src[i], dst);
            else pack_host(*shape, src[i], dst);
        } else {
            cudaError_t e = launch_pack_device(*shape, src[i], dst, static_cast<cudaStream_t>(stream));
            if (e != cudaSuccess) return SMOE_ECUDA;
        }
    }
    return SMOE_OK;
}

extern "C" int smoe_ctx_create(const smoe_shape *shape, int32_t n_layers, int64_t n_slots, int32_t *table_dev,
                               smoe_ctx **out)
{
    int rc = shape_check(shape, true);
    if (rc) return rc;
    if (!out || n_layers <= 0 || n_slots <= 0 || !table_dev) return SMOE_EINVAL;
    *out = nullptr;
    smoe_ctx *c = new (std::nothrow) smoe_ctx();
    if (!c) return SMOE_ENOMEM;
    c->shape = *shape;
    c->layout = shape->bits == 8 ? layout8_of(shape->H, shape->I) : layout_of(shape->H, shape->I);
    c->n_layers = n_layers;
    c->n_slots = n_slots;
    c->table_dev = table_dev;
    c->cs = shape->I / kSlice;
    c->stack_wait_ns = 0;
    c->stack_stall_layer = -1;
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e == cudaSuccess) e = route_config();
    if (e == cudaSuccess) e = prefill_config();
    if (e == cudaSuccess) e = decode_config(c);
    if (e == cudaSuccess) e = stack_config(c);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return e == cudaErrorInvalidConfiguration || e == cudaErrorInvalidValue ? SMOE_ENOTSUP : SMOE_ECUDA;
    }
    *out = c;
    return SMOE_OK;
}

extern "C" int smoe_ctx_destroy(smoe_ctx *ctx)
{
    delete ctx;
    return SMOE_OK;
}

extern "C" int set_slot_table(smoe_ctx *ctx, int32_t layer, const int32_t *host_table, void *stream)
{
    if (!ctx || !host_table || layer < 0 || layer >= ctx->n_layers) return SMOE_EINVAL;
    const int E = ctx->shape.E;
    std::vector<int32_t> tmp(host_table, host_table + E);
    for (int e = 0; e < E; ++e)
        if (tmp[e] < 0 || tmp[e] >= ctx->n_slots) return SMOE_ERANGE;
    std::qsort(tmp.data(), tmp.size(), sizeof(int32_t), [](const void *a, const void *b) {
        const int32_t x = *static_cast<const int32_t *>(a), y = *static_cast<const int32_t *>(b);
        return (x > y) - (x < y);
    });
    for (size_t i = 1; i < tmp.size(); ++i)
        if (tmp[i] == tmp[i - 1]) return SMOE_ERANGE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(ctx->table_dev + size_t(layer) * E, host_table, sizeof(int32_t) * E,
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

extern "C" uint64_t smoe_workspace_bytes(const smoe_ctx *ctx, int32_t T)
{
    if (!ctx || T <= 0 || T > SMOE_MAX_TOKENS) return 0;
    return workspace_layout(ctx->shape, T).total;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

extern "C" int moe_route(const smoe_ctx *ctx, const uint16_t *W_r, const uint16_t *w_s, const uint16_t *x,
                         int32_t T, const float *logit_bias, int32_t *ids, float *w, float *gate, void *workspace,
                         uint64_t workspace_bytes, void *stream)
{
    if (!ctx || T < 0 || T > SMOE_MAX_TOKENS) return SMOE_EINVAL;
    if (T == 0) return SMOE_OK;                      // nothing to do; the buffers may be null
    if (!W_r || !w_s || !x || !ids || !w || !gate || !workspace) return SMOE_EINVAL;
    if (!aligned16(W_r) || !aligned16(w_s) || !aligned16(x) || !aligned16(workspace)) return SMOE_EINVAL;
    const Workspace W = workspace_layout(ctx->shape, T);
    if (workspace_bytes < W.total) return SMOE_ENOMEM;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    RouteParams p = {};
    p.Wr = W_r;
    p.ws = w_s;
    p.x = x;
    p.bias = logit_bias;
    p.logits = reinterpret_cast<float *>(ws + W.logits);
    p.ids = ids;
    p.w = w;
    p.gate = gate;
    p.counter = reinterpret_cast<uint32_t *>(ws + W.route_counter);
    p.err = nullptr;
    p.T = T;
    p.H = ctx->shape.H;
    p.E = ctx->shape.E;
    p.k = ctx->shape.k;
    return cuda_status(launch_route(p, static_cast<cudaStream_t>(stream)));
}

extern "C" int moe_forward(const smoe_ctx *ctx, int32_t layer, const uint16_t *x, int32_t T, const int32_t *ids,
                           const float *w, const float *gate, const void *pool, uint64_t pool_bytes,
                           const void *shared_blob, const uint16_t *residual, uint16_t *out, void *workspace,
                           uint64_t workspace_bytes, int32_t *err, void *stream)
{
    if (!ctx || T < 0 || T > SMOE_MAX_TOKENS) return SMOE_EINVAL;
    if (layer < 0 || layer >= ctx->n_layers) return SMOE_EINVAL;
    // 8-bit experts: the bucketed path for T > 8, the T <= 8 kernel where it fits
    if (ctx->shape.bits != 4 && T <= kDecodeMaxT && !ctx->decode_ok) return SMOE_ENOTSUP;
    if (T == 0) return SMOE_OK;                      // nothing to do; the buffers may be null
    if (!x || !ids || !w || !gate || !pool || !shared_blob || !out || !workspace || !err) return SMOE_EINVAL;
    if (!aligned16(x) || !aligned16(pool) || !aligned16(shared_blob) || !aligned16(workspace) || !aligned16(out) ||
        (residual && !aligned16(residual)))
        return SMOE_EINVAL;
    if (pool_bytes < uint64_t(ctx->n_slots) * ctx->layout.blob) return SMOE_ENOMEM;
    const Workspace W = workspace_layout(ctx->shape, T);
    if (workspace_bytes < W.total) return SMOE_ENOMEM;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T > kDecodeMaxT) {
        PrefillParams q = {};
        q.ids = ids;
        q.counts = reinterpret_cast<int32_t *>(ws + W.counts);
        q.chunk_base = reinterpret_cast<int32_t *>(ws + W.chunk_base);
        q.ticket = reinterpret_cast<uint32_t *>(ws + W.fwd_counters);   // unused by the T <= 8 path of this call
        q.offsets = reinterpret_cast<int32_t *>(ws + W.offsets);
        q.tiles = reinterpret_cast<PfTile *>(ws + W.tiles);
        q.ntiles = reinterpret_cast<int32_t *>(ws + W.ntiles);
        q.table_row = ctx->table_dev + size_t(layer) * ctx->shape.E;
        q.n_slots = ctx->n_slots;
        q.pair_token = reinterpret_cast<int32_t *>(ws + W.pair_token);
        q.w = w;
        q.gate = gate;
        q.pair_pos = reinterpret_cast<int32_t *>(ws + W.pair_pos);
        q.ypair = reinterpret_cast<const uint16_t *>(ws + W.ybuf);
        q.residual = residual;
        q.out = out;
        q.err = err;
        q.T = T;
        q.H = ctx->shape.H;
        q.E = ctx->shape.E;
        q.k = ctx->shape.k;
        q.P = T * ctx->shape.k;
        GemmParams g = {};
        g.pool = static_cast<const uint8_t *>(pool);
        g.shared_blob = static_cast<const uint8_t *>(shared_blob);
        g.table_row = ctx->table_dev + size_t(layer) * ctx->shape.E;
        g.stride = ctx->layout.blob;
        g.n_slots = ctx->n_slots;
        g.x = reinterpret_cast<const uint16_t *>(ws + W.xt);
        g.x_bf16 = x;
        g.hbuf = reinterpret_cast<uint16_t *>(ws + W.hbuf);
        g.ypair = reinterpret_cast<uint16_t *>(ws + W.ybuf);
        g.pair_token = q.pair_token;
        g.ntiles = q.ntiles;
        g.tiles = q.tiles;
        g.err = err;
        g.T = T;
        g.H = q.H;
        g.E = q.E;
        g.k = q.k;
        g.I = ctx->shape.I;
        g.P = q.P;
        g.bits = ctx->shape.bits;
        return cuda_status(launch_prefill(q, g, st, ctx->prof, ctx->nprof));
    }
    DecodeParams p = {};
    p.x = x;
    p.ids = ids;
    p.w = w;
    p.gate = gate;
    p.pool = static_cast<const uint8_t *>(pool);
    p.shared_blob = static_cast<const uint8_t *>(shared_blob);
    p.table_row = ctx->table_dev + size_t(layer) * ctx->shape.E;
    p.residual = residual;
    p.out = out;
    p.ypair = reinterpret_cast<float *>(ws + W.ypair);
    p.counters = reinterpret_cast<uint32_t *>(ws + W.fwd_counters);
    p.err = err;
    p.stride = ctx->layout.blob;
    p.n_slots = ctx->n_slots;
    p.T = T;
    p.H = ctx->shape.H;
    p.E = ctx->shape.E;
    p.k = ctx->shape.k;
    p.I = ctx->shape.I;
    cudaError_t e = prof_record(ctx->nprof > 0 ? ctx->prof[0] : nullptr, st);
    if (e == cudaSuccess) e = launch_decode(ctx, p, st);
    if (e == cudaSuccess) e = prof_record(ctx->nprof > 1 ? ctx->prof[1] : nullptr, st);
    return cuda_status(e);
}

extern "C" int smoe_check(int32_t *err_dev, int32_t *code, void *stream)
{
    if (!err_dev) return SMOE_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, err_dev, sizeof h, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && h != 0) e = cudaMemsetAsync(err_dev, 0, sizeof h, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return SMOE_ECUDA;
    if (code) *code = h;
    return h ? SMOE_EDEVICE : SMOE_OK;
}

extern "C" int smoe_set_profile_events(smoe_ctx *ctx, void *const *events, int32_t n)
{
    if (!ctx || n < 0 || n > 4 || (n > 0 && !events)) return SMOE_EINVAL;
    for (int i = 0; i < 4; ++i) ctx->prof[i] = i < n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
    ctx->nprof = n;
    return SMOE_OK;
}

// Workspace of moe_decode_stack: the arrival words and h's per-expert
// counters (zeroed at launch), the exchange region the kernel fills with its
// sentinel (logits [n][E + kStackZPad] fp32, x [n + 1][H] bf16), then h
// [n][2][U][I] bf16 (read only after its counter says it is complete).
struct StackWs {
    uint64_t sync, hcnt, zl, xe, xend, hx, total;
};

static StackWs stack_ws(const smoe_ctx *ctx, int n)
{
    auto al = [](uint64_t v) { return (v + 255) & ~uint64_t(255); };
    const smoe_shape &s = ctx->shape;
    StackWs w = {};
    uint64_t o = 0;
    w.sync = o;   o = al(o + kStackSyncBytes);
    w.hcnt = o;   o = al(o + uint64_t(n) * ctx->stack.U * kStackCntStride * 4);
    w.zl = o;     o = al(o + uint64_t(n) * (s.E + kStackZPad) * 4);
    w.xe = o;     o = al(o + (uint64_t(n) + 1) * s.H * 2);
    w.xend = o;
    w.hx = o;     o = al(o + uint64_t(n) * 2 * ctx->stack.U * s.I * 2);
    w.total = o;
    return w;
}

extern "C" uint64_t smoe_stack_workspace_bytes(const smoe_ctx *ctx, int32_t n_layers)
{
    if (!ctx || !ctx->stack.ok || n_layers < 1 || n_layers > kStackMaxLayers) return 0;
    return stack_ws(ctx, n_layers).total;
}

extern "C" int moe_decode_stack(const smoe_ctx *ctx, int32_t first_layer, int32_t n_layers,
                                const uint16_t *const *W_r, const uint16_t *const *w_s,
                                const void *const *shared_blobs, const float *logit_bias, uint16_t *xs,
                                int32_t *ids, float *w, float *gate, const void *pool, uint64_t pool_bytes,
                                void *workspace, uint64_t workspace_bytes, int32_t *err, void *stream)
{
    if (!ctx || !W_r || !w_s || !shared_blobs || !xs || !ids || !w || !gate || !pool || !workspace || !err)
        return SMOE_EINVAL;
    if (n_layers < 1 || first_layer < 0 || first_layer + n_layers > ctx->n_layers) return SMOE_EINVAL;
    if (n_layers > kStackMaxLayers || !ctx->stack.ok) return SMOE_ENOTSUP;
    if (!aligned16(xs) || !aligned16(pool) || !aligned16(workspace)) return SMOE_EINVAL;
    if (pool_bytes < uint64_t(ctx->n_slots) * ctx->layout.blob) return SMOE_ENOMEM;
    const StackWs W = stack_ws(ctx, n_layers);
    if (workspace_bytes < W.total) return SMOE_ENOMEM;
    StackParams p = {};
    for (int l = 0; l < n_layers; ++l) {
        if (!W_r[l] || !w_s[l] || !shared_blobs[l]) return SMOE_EINVAL;
        if (!aligned16(W_r[l]) || !aligned16(w_s[l]) || !aligned16(shared_blobs[l])) return SMOE_EINVAL;
        p.Wr[l] = W_r[l];
        p.ws[l] = w_s[l];
        p.shared[l] = static_cast<const uint8_t *>(shared_blobs[l]);
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.bias = logit_bias;
    p.xs = xs;
    p.ids = ids;
    p.w = w;
    p.gate = gate;
    p.pool = static_cast<const uint8_t *>(pool);
    p.table = ctx->table_dev + size_t(first_layer) * ctx->shape.E;
    p.stride = ctx->layout.blob;
    p.n_slots = ctx->n_slots;
    p.zl = reinterpret_cast<float *>(ws + W.zl);
    p.hx = reinterpret_cast<uint16_t *>(ws + W.hx);
    p.xe = reinterpret_cast<uint16_t *>(ws + W.xe);
    p.xbuf = ws + W.zl;
    p.xbuf_words16 = (W.total - W.zl) / 16;       // logits, layer outputs and h
    p.sync = reinterpret_cast<uint32_t *>(ws + W.sync);
    p.hcnt = reinterpret_cast<uint32_t *>(ws + W.hcnt);
    p.sync_bytes = W.zl;                           // the counters and arrival words, zeroed per launch
    p.err = err;
    p.wait_ns = ctx->stack_wait_ns ? ctx->stack_wait_ns : kWaitLimitNs;
    p.stall_layer = ctx->stack_stall_layer;
    p.n_layers = n_layers;
    p.H = ctx->shape.H;
    p.E = ctx->shape.E;
    p.k = ctx->shape.k;
    p.I = ctx->shape.I;
    p.U = ctx->stack.U;
    p.nr = ctx->stack.nr;
    p.nu = ctx->stack.nu;
    p.nslot = ctx->stack.nslot;
    return cuda_status(launch_stack(ctx, p, static_cast<cudaStream_t>(stream)));
}

extern "C" int smoe_set_stack_wait(smoe_ctx *ctx, uint64_t grid_wait_ns, int32_t stall_layer)
{
    if (!ctx || stall_layer < -1 || stall_layer >= kStackMaxLayers) return SMOE_EINVAL;
    ctx->stack_wait_ns = grid_wait_ns;
    ctx->stack_stall_layer = stall_layer;
    return SMOE_OK;
}

extern "C" int smoe_ctx_describe(const smoe_ctx *ctx, char *buf, int32_t len)
{
    if (!ctx || !buf || len <= 0) return SMOE_EINVAL;
    int o = std::snprintf(buf, size_t(len), "sms=%d decode: cluster=%d", ctx->num_sms, ctx->cs);
    for (int T = 1; T <= kDecodeMaxT && o < len; ++T)
        o += std::snprintf(buf + o, size_t(len - o), " T%d:{slots=%d smem=%d/%d clusters=%d/%d}", T,
                           ctx->decode[T].nst, ctx->decode[T].smem, ctx->decode[T].smem16,
                           ctx->decode[T].max_clusters, ctx->decode[T].max_clusters16);
    if (o < len)
        std::snprintf(buf + o, size_t(len - o), " stack:{ok=%d grid=%d rows=%d units=%d smem=%d}", int(ctx->stack.ok),
                      ctx->stack.grid, ctx->stack.nr, ctx->stack.nu, ctx->stack.smem);
    return SMOE_OK;
}

extern "C" const char *smoe_status_string(int status)
{
    switch (status) {
    case SMOE_OK: return "ok";
    case SMOE_EINVAL: return "invalid argument";
    case SMOE_ERANGE: return "slot or expert id out of range";
    case SMOE_ENOMEM: return "pool or workspace too small";
    case SMOE_ECUDA: return "CUDA runtime error";
    case SMOE_EDEVICE: return "kernel reported an error";
    case SMOE_ENOTSUP: return "shape not supported";
    default: return "unknown status";
    }
}
