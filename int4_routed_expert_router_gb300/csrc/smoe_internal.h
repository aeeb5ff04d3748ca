// smoe_internal.h -- library-internal definitions shared by the host code and
// the kernels (blob format constants, context, kernel parameter blocks).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/smoe.h"

namespace smoe {

constexpr int kGroup = 64;          // quantisation group along the input dim
constexpr int kAtomRows = 16;       // rows per atom
constexpr int kAtomQBytes = 512;    // packed nibbles of one atom
constexpr int kAtomBytes = 576;     // nibbles + 16 (s, b) fp16 pairs
constexpr int kAtom8Bytes = 2 * kAtomQBytes + 64;   // 8-bit atom: two nibble planes, then the (s, b) pairs

// Decode kernel (fused experts, T <= kDecodeMaxT).
constexpr int kDecodeMaxT = 8;
constexpr int kBucketTok = 32;     // most tokens per bucketing chunk (T > kDecodeMaxT path)
// tokens per bucketing chunk for T tokens: small chunks (more warps in the
// ordered scatter) when T is small
inline __host__ __device__ int bucket_tok(int T) { return T <= 1024 ? 8 : kBucketTok; }
constexpr int kRouteGemvMaxT = 512; // T > kDecodeMaxT up to this: logits by the GEMV kernel, else tcgen05
constexpr int kSlice = 32;                        // intermediates per CTA
constexpr int kChunkCols = 256;                   // H columns per streamed chunk
constexpr int kRowBlocksA = kSlice / 8;           // gate/up row blocks per CTA
constexpr int kChunkBytes = kRowBlocksA * (kChunkCols / kGroup) * kAtomBytes;   // 9216

struct Layout {
    uint64_t blob, gu_off, gu_bytes, down_off, down_bytes;
};

inline Layout layout_of(int H, int I)
{
    Layout L;
    L.gu_off = 0;
    L.gu_bytes = uint64_t(I / 8) * (H / kGroup) * kAtomBytes;
    L.down_off = L.gu_bytes;
    L.down_bytes = uint64_t(H / 16) * (I / kGroup) * kAtomBytes;
    L.blob = L.gu_bytes + L.down_bytes;
    return L;
}

struct DecodeCfg {
    int nst = 0;              // ring slots
    int smem = 0;             // dynamic shared memory bytes, 8 consumer warps
    int max_clusters = 0;     // co-resident clusters, 8 consumer warps
    int smem16 = 0;           // the same with 16 consumer warps
    int max_clusters16 = 0;
};

// Multi-layer decode step (decode_stack.cu), one token.
constexpr int kStackMaxLayers = 64;
constexpr int kStackSyncBytes = 64;         // start-of-launch arrival counter, abort word
constexpr int kStackCntStride = 32;         // words between two experts' arrival counters (one 128-byte line)
constexpr int kStackZPad = 8;               // a logit row holds E + kStackZPad words (E % 4 == 0)

struct StackCfg {
    bool ok = false;          // cooperative launch available and the shared memory fits
    int grid = 0;             // CTAs (one per SM)
    int U = 0;                // experts per layer: k routed + the shared expert
    int nr = 0;               // most router rows of one CTA
    int nu = 0;               // most routed gate/up units of one CTA
    int nslot = 0;            // most gate/up units (routed + shared) of one CTA: 8-bit ring slots
    int smem = 0;
};

struct StackParams {
    const uint16_t *Wr[kStackMaxLayers];       // router rows of each layer [E][H] bf16
    const uint16_t *ws[kStackMaxLayers];       // shared-gate vector of each layer [H]
    const uint8_t *shared[kStackMaxLayers];    // shared-expert blob of each layer
    const float *bias;                         // [E] logit offsets or nullptr
    uint16_t *xs;                              // [(n_layers + 1)][H] bf16: input, then each layer's output
    int32_t *ids;                              // [n_layers][k]
    float *w;                                  // [n_layers][k]
    float *gate;                               // [n_layers]
    const uint8_t *pool;
    const int32_t *table;                      // slot table rows of the layers [n_layers][E]
    uint64_t stride;
    int64_t n_slots;
    // exchange buffers, one region filled with the all-ones sentinel at launch:
    float *zl;                                 // [n_layers][E + kStackZPad] logits (word E: shared gate)
    uint16_t *hx;                              // [n_layers][2][U][I] bf16: h's high part, then h - high
                                               // (not part of the filled region: guarded by hcnt)
    uint16_t *xe;                              // [n_layers + 1][H] bf16: each layer's output
    void *xbuf;                                // the region (16-byte aligned)
    uint64_t xbuf_words16;                     // its size in 16-byte words
    uint32_t *sync;                            // kStackSyncBytes: [0] start arrivals, [1] abort word
    uint32_t *hcnt;                            // [n_layers][U][kStackCntStride] arrival counters of h (zeroed)
    uint64_t sync_bytes;                       // bytes from sync zeroed at launch (sync and hcnt)
    int32_t *err;
    uint64_t wait_ns;                          // limit of a grid-wide wait
    int stall_layer;                           // test hook: this layer's first grid-wide wait never completes (-1: off)
    int n_layers, H, E, k, I, U, nr, nu, nslot;
};

}  // namespace smoe

struct smoe_ctx {
    smoe_shape shape;
    smoe::Layout layout;
    int32_t n_layers;
    int64_t n_slots;
    int32_t *table_dev;
    int device;
    int num_sms;
    int cs;                                  // cluster size of the decode kernel = I / kSlice
    cudaEvent_t prof[4];                     // profiling hook (smoe_set_profile_events)
    int nprof;
    smoe::DecodeCfg decode[smoe::kDecodeMaxT + 1];
    smoe::StackCfg stack;
    bool decode_ok;                          // the T <= 8 expert kernel runs this shape's experts
    uint64_t stack_wait_ns;                  // grid-wide wait limit of moe_decode_stack (smoe_set_stack_wait)
    int32_t stack_stall_layer;               // -1, or the layer whose first grid-wide wait is made to run out
};

namespace smoe {

struct RouteParams {
    const uint16_t *Wr;
    const uint16_t *ws;
    const uint16_t *x;
    const float *bias;
    float *logits;          // [T][E+1] (column E: shared-gate logit)
    int32_t *ids;
    float *w;
    float *gate;
    uint32_t *counter;
    int32_t *err;
    int T, H, E, k;
    int fused_topk;
    int gate_in_logits;     // logits[t][E] holds the shared-gate logit (GEMV path)
};

struct DecodeParams {
    const uint16_t *x;
    const int32_t *ids;
    const float *w;
    const float *gate;
    const uint8_t *pool;
    const uint8_t *shared_blob;
    const int32_t *table_row;   // slot table row of this layer
    const uint16_t *residual;
    uint16_t *out;
    float *ypair;               // [(U_max + 1)][T][H] fp32, expert outputs (unweighted)
    uint32_t *counters;         // [cs] arrival tickets per row chunk
    int32_t *err;
    uint64_t stride;
    int64_t n_slots;
    int T, H, E, k, I;
    int cs, nst;
};

struct PfTile {
    int32_t kind;     // 0: run of an expert's pairs; 1: run of tokens for the shared expert
    int32_t slot;     // pool slot of the expert (kind 0; -1 if the slot table entry is out of range), else 0
    int32_t p0;       // first pair (kind 0) or first token (kind 1)
    int32_t n;        // rows in the run (1 .. 192)
};

// Token-bucketed path (T > 8): bucketing and combine.
struct PrefillParams {
    const int32_t *ids;
    int32_t *counts;       // [E][chunks]
    int32_t *chunk_base;   // [E][chunks]
    uint32_t *ticket;      // arrival ticket of the scan (zero between calls)
    int32_t *offsets;      // [E + 1]
    PfTile *tiles;         // [max tiles]
    int32_t *ntiles;
    const int32_t *table_row;  // the layer's slot table row [E]
    int64_t n_slots;
    int32_t *pair_token;   // [T*k]
    const float *w;        // [T][k] routing weights
    const float *gate;     // [T] shared-expert gates
    int32_t *pair_pos;     // [T*k] position of pair (t, j) in expert order, -1 if invalid
    const uint16_t *ypair; // [(T*k + T)][H] fp16 expert outputs (unweighted)
    const uint16_t *residual;
    uint16_t *out;
    int32_t *err;
    int T, H, E, k, P;     // P = T*k (rows of routed pairs; shared rows follow)
};

struct GemmParams {
    int mode;              // 0 gate/up, 1 down, 2 router logits
    const uint8_t *pool;
    const uint8_t *shared_blob;
    const int32_t *table_row;
    uint64_t stride;
    int64_t n_slots;
    const uint16_t *x;     // expert GEMMs: xt [T][H] fp16 (x in the MMA K order); router: x [T][H] bf16
    const uint16_t *x_bf16;  // the caller's bf16 x (converted into xt by the path)
    uint16_t *hbuf;        // [(P + T)][I] fp16
    uint16_t *ypair;       // [(P + T)][H] fp16 expert outputs (unweighted)
    const int32_t *pair_token;
    const int32_t *ntiles;
    const PfTile *tiles;
    const uint16_t *Wr;    // router rows (mode 2)
    float *logits;         // [T][E + 1] (mode 2)
    int32_t *err;
    int T, H, E, k, I, P;
    int m_tiles;
    int bits;              // expert GEMMs: 4 or 8 (the atom format of pool and shared_blob)
};

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while its predecessor in the stream finishes; it calls pdl_wait (griddepcontrol.wait)
// before touching global memory, so it still sees all of the predecessor's work.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args)
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, static_cast<Args &&>(args)...);
}

// workspace carving (all offsets 256-byte aligned)
struct Workspace {
    uint64_t route_counter, logits, fwd_counters, ypair, total;
    // token-bucketed path (T > kDecodeMaxT)
    uint64_t counts, chunk_base, offsets, tiles, ntiles, pair_token, pair_pos, hbuf, ybuf, xt;
};

Workspace workspace_layout(const smoe_shape &s, int T);

cudaError_t route_config();
cudaError_t launch_route(const RouteParams &p, cudaStream_t st);
cudaError_t launch_decode(const smoe_ctx *ctx, const DecodeParams &p, cudaStream_t st);
cudaError_t decode_config(smoe_ctx *ctx);
cudaError_t stack_config(smoe_ctx *ctx);
cudaError_t launch_stack(const smoe_ctx *ctx, const StackParams &p, cudaStream_t st);
cudaError_t prefill_config();
int prefill_max_tiles(int T, int k, int E);
cudaError_t launch_router_gemm(const RouteParams &r, cudaStream_t st);
cudaError_t launch_prefill(const PrefillParams &p, const GemmParams &g, cudaStream_t st, const cudaEvent_t *prof,
                           int nprof);
// records ev (if any) on st as an external event
inline cudaError_t prof_record(cudaEvent_t ev, cudaStream_t st)
{
    return ev ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal) : cudaSuccess;
}
cudaError_t launch_pack_device(const smoe_shape &s, const smoe_expert_src &src, uint8_t *dst,
                               cudaStream_t st);
void pack_host(const smoe_shape &s, const smoe_expert_src &src, uint8_t *dst);

}  // namespace smoe
