/*
 * smoe.h -- C ABI of the int4 routed-expert MoE layer for one GB300 (sm_103a).
 *
 * The layer is the sparse Mixture-of-Experts block of the Qwen3-Next /
 * Qwen3.5-3.6 hybrid models that the Swiftlet runtime runs on Apple devices
 * (pages: "Swiftlet Packs 80B Qwen Into Mac With 4.3GB Memory..." on xix.ai,
 * paragraph on how it works; "Swiftletは低RAM使用量で..." on agentlenshq.com,
 * section on how expert streaming works). For each token x (bf16, length H):
 *
 *   z  = W_r x (+ optional per-expert logit offset)       router, E logits
 *   p  = softmax(z); ids = the k largest p (ties: lower id first)
 *   w_j = p_{ids_j} / sum_j' p_{ids_j'}                     renormalised
 *   f_e(x) = D_e (silu(G_e x) * (U_e x))                   SwiGLU expert
 *   out = sum_{j<k} w_j f_{ids_j}(x) + sigmoid(w_s . x) f_shared(x)
 *
 * The routed and shared experts hold MLX-style affine 4-bit weights: groups of
 * 64 along the input dimension, an fp16 scale s and bias b per group,
 * w = s*q + b (the same xix.ai page, last paragraph, names MLX-style int4 and
 * int8 group quantisation with 64-bit offsets). 8-bit experts are supported
 * for packing, routing, moe_forward at every T and the plain debug path
 * (see smoe_ctx_create). The routed experts of every layer live in
 * one pool of fixed-stride blobs, one blob per expert, reached through a slot
 * table (same page, paragraph on how it works: fixed-stride blobs, one read
 * per expert, a bounded slot pool).
 *
 * Conventions for every call:
 *  - Return value: SMOE_OK (0) or a negative SMOE_E* status. Nothing aborts,
 *    prints, or throws across this ABI.
 *  - Device memory is always owned by the caller. The library never allocates
 *    device memory; smoe_workspace_bytes() says how much scratch to pass.
 *  - "stream" is a cudaStream_t (NULL = legacy default stream). moe_route and
 *    moe_forward only enqueue work on it: they never synchronise, so they can
 *    be issued back to back and captured into a CUDA graph.
 *  - bf16 / fp16 tensors are passed as uint16_t bit patterns.
 *  - All tensors are dense and row-major (C order), 16-byte aligned.
 */
#ifndef SMOE_H
#define SMOE_H

#include <stdint.h>

#if defined(__GNUC__)
#define SMOE_API __attribute__((visibility("default")))
#else
#define SMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define SMOE_OK 0
#define SMOE_EINVAL (-1)   /* bad argument: null pointer, bad size, misaligned */
#define SMOE_ERANGE (-2)   /* slot or expert id out of range, duplicate slot */
#define SMOE_ENOMEM (-3)   /* pool or workspace smaller than required */
#define SMOE_ECUDA (-4)    /* a CUDA runtime call failed */
#define SMOE_EDEVICE (-5)  /* a kernel reported a problem in the error word */
#define SMOE_ENOTSUP (-6)  /* shape outside what the kernels support */

/* Codes a kernel may store in the device error word (first one wins). */
#define SMOE_DEV_BAD_SLOT 1     /* a selected expert's slot is < 0 or >= n_slots */
#define SMOE_DEV_BAD_EXPERT 2   /* an id in ids[] is < 0 or >= E */
#define SMOE_DEV_TIMEOUT 3      /* a bounded wait inside a kernel gave up */
#define SMOE_DEV_RANGE 4        /* T > 8 path: |x| or |h| >= 65504, or an expert output that rounds to
                                   65504 or beyond in fp16 (outside its fp16 intermediates) */

/* Most tokens of one moe_route / moe_forward call (T); larger T is
 * SMOE_EINVAL and smoe_workspace_bytes returns 0. A call with T = 0 (any
 * entry point taking T) returns SMOE_OK without touching a buffer, so its
 * buffer pointers may be null (smoe_workspace_bytes(ctx, 0) is 0). */
#define SMOE_MAX_TOKENS (1 << 20)

/* ------------------------------------------------------------------ shapes */
/* H: hidden size; E: routed experts per layer; k: experts per token;
 * I: routed expert intermediate size; I_shared: shared expert intermediate
 * size; group: quantisation group (must be 64); bits: 4, or 8 (layout,
 * packing, routing, moe_forward for T <= 8 and moe_forward_debug; see
 * smoe_ctx_create).
 * Supported: H % 256 == 0, H <= 2048, I % 64 == 0, 64 <= I <= 512, I_shared == I,
 * 1 <= k <= 16, k <= E <= 1024. Others return SMOE_ENOTSUP. */
typedef struct smoe_shape {
    int32_t H, E, k, I, I_shared, group, bits;
} smoe_shape;

/* ------------------------------------------------------------- blob layout */
/* One expert blob (fixed stride, no padding at H=2048, I=512:
 * 1,769,472 bytes = 432 * 4 KiB). It is made of 576-byte "atoms"; an atom
 * holds 16 logical rows x one group of 64 input columns:
 *   bytes [0,512): 32 lanes x 16 bytes; lane L = 4g+t (g < 8, t < 4) holds the
 *     four uint32 words (row g, cols 16t..16t+7), (row g, cols 16t+8..16t+15),
 *     (row g+8, cols 16t..16t+7), (row g+8, cols 16t+8..16t+15) of the group;
 *     a word for columns c0..c0+7 keeps column c0+2m in bits 4m..4m+3 and
 *     column c0+2m+1 in bits 16+4m..16+4m+3 (m < 4): even columns in the low
 *     half-word, odd columns in the high half-word;
 *   bytes [512,576): for g < 8, fp16 (s, b) of row g followed by (s, b) of
 *     row g+8 (8 bytes per g).
 * Gate/up part (first): atom index rb*(H/64) + kb for row block rb < I/8 and
 *   input group kb < H/64; logical row g < 8 is gate row 8rb+g and logical row
 *   g+8 is up row 8rb+g (the two rows SwiGLU multiplies sit together).
 * Down part (second, at offset down_offset): atom index rd*(I/64) + kb for
 *   row block rd < H/16 and input group kb < I/64; logical row i is down row
 *   16rd+i.
 * The 16x64 atom is the operand fragment of one 16x8x16 tensor-core step per
 * lane, so the decode kernel loads a lane's share with one 128-bit load. */
typedef struct smoe_layout {
    uint64_t blob_bytes;    /* stride between slots */
    uint64_t gu_offset;     /* 0 */
    uint64_t gu_bytes;      /* (I/8)*(H/64)*576 */
    uint64_t down_offset;   /* == gu_bytes */
    uint64_t down_bytes;    /* (H/16)*(I/64)*576 */
    uint32_t atom_bytes;    /* 576 */
    uint32_t atom_rows;     /* 16 */
    uint32_t group;         /* 64 */
    uint32_t reserved;
} smoe_layout;

/* 8-bit experts (bits = 8): the same atoms of 16 rows x 64 columns in the
 * same order, 1,088 bytes each: bytes [0,512) hold each value's low nibble
 * and bytes [512,1024) its high nibble, each plane laid out exactly as the
 * 4-bit atom's bytes [0,512) (so q = low + 16 * high), then the (s, b) bytes
 * of the 4-bit atom at [1024,1088). 3,342,336 bytes per blob at H=2048, I=512.
 * The pages name MLX int4/int8 group quantisation ("Swiftlet Packs 80B Qwen
 * Into Mac...", last paragraph). */

/* Fills *out for shape. Errors: SMOE_EINVAL (null), SMOE_ENOTSUP (shape). */
SMOE_API int smoe_layout_of(const smoe_shape *shape, smoe_layout *out);
/* (for bits = 8, atom_bytes is 1088 and the offsets count 8-bit atoms) */

/* ------------------------------------------------------- smoe_quantize_mlx */
/* MLX-style affine quantisation of one float32 matrix w [rows][cols]
 * (row-major, host memory) into the triples pack_experts reads: per group of
 * 64 columns of a row, b = the group minimum rounded down to fp16, s = (max -
 * b) / (2^bits - 1) rounded up to fp16, q = round-half-even((w - b) / s)
 * clamped to [0, 2^bits - 1] (q = 0 where s = 0), all in double precision, so
 * |w - (s q + b)| <= s / 2. Outputs (host, caller-owned): q uint32
 * [rows][cols * bits / 32] (column c in bits bits*(c % (32/bits)).. of word
 * c / (32/bits)), s and b fp16 bits [rows][cols / 64]. The pages name MLX
 * int4/int8 group quantisation with a scale and bias per group of 64 (xix.ai
 * article, last paragraph) but not the quantiser; the rounding directions are
 * this library's reading, and bit parity with MLX's own quantiser is not
 * claimed. Errors: SMOE_EINVAL (negative sizes, null buffers), SMOE_ENOTSUP
 * (bits not 4 or 8, cols % 64), SMOE_ERANGE (a value or a group's span that
 * fp16 cannot hold: non-finite or above 65504). */
SMOE_API int smoe_quantize_mlx(const float *w, int32_t rows, int32_t cols, int32_t bits, uint32_t *q,
                               uint16_t *s, uint16_t *b);

/* ------------------------------------------------------------ pack_experts */
/* MLX triples of one expert (as produced by MLX's affine quantisation):
 * q[0] gate uint32 [I][H/8], q[1] up [I][H/8], q[2] down [H][I/8], column c of
 * a row in bits 4*(c%8).. of word c/8; s[m], b[m] fp16 bits [rows][cols/64].
 * With bits = 8: q[0], q[1] [I][H/4], q[2] [H][I/4], column c in bits
 * 8*(c%4).. of word c/4. */
typedef struct smoe_expert_src {
    const uint32_t *q[3];
    const uint16_t *s[3];
    const uint16_t *b[3];
} smoe_expert_src;

#define SMOE_HOST 0     /* src triples and pool are host memory; runs on the CPU */
#define SMOE_DEVICE 1   /* src triples and pool are device memory; a kernel on stream */

/* Writes expert i's blob at pool + dst_slots[i] * layout.blob_bytes (64-bit
 * offsets; the pool may span tens of GB) for i < n. src and dst_slots are
 * host arrays of n entries; the pointers inside src point to memory of kind
 * `where`. The pool must hold at least (max slot + 1) * blob_bytes bytes
 * (pool_bytes). With SMOE_DEVICE the copies are enqueued on stream and the
 * triples must stay valid until they complete. Corresponds to the pages'
 * repack step ("swiftlet-repack" builds fixed-stride containers from MLX
 * checkpoints), done in memory.
 * 8-bit experts pack with either kind. q words must start on a 4-byte and s,
 * b on a 2-byte boundary, and a device pool on a 16-byte boundary (else
 * SMOE_EINVAL before any work).
 * Errors: SMOE_EINVAL, SMOE_ENOTSUP, SMOE_ERANGE (slot < 0), SMOE_ENOMEM
 * (slot past pool_bytes), SMOE_ECUDA. */
SMOE_API int pack_experts(const smoe_shape *shape, const smoe_expert_src *src, int32_t n,
                 const int64_t *dst_slots, void *pool, uint64_t pool_bytes,
                 int32_t where, void *stream);

/* ---------------------------------------------------------------- context */
typedef struct smoe_ctx smoe_ctx;

/* Creates a host-side context on the current CUDA device for shape, a stack
 * of n_layers layers and a pool of n_slots slots. table_dev is caller-owned
 * device memory of n_layers*E int32 (the slot table; filled by
 * set_slot_table). The context allocates no device memory. A context of
 * 8-bit experts (shape.bits = 8) serves every call (the T <= 8 kernel, the
 * bucketed expert GEMMs and the stack kernel all read the two nibble
 * planes); a shape whose 8-bit T <= 8 kernel does not fit the GPU makes
 * moe_forward (T <= 8) and moe_forward_noalloc return SMOE_ENOTSUP.
 * Errors: SMOE_EINVAL, SMOE_ENOTSUP, SMOE_ECUDA. */
SMOE_API int smoe_ctx_create(const smoe_shape *shape, int32_t n_layers, int64_t n_slots,
                    int32_t *table_dev, smoe_ctx **out);
SMOE_API int smoe_ctx_destroy(smoe_ctx *ctx);

/* ---------------------------------------------------------- set_slot_table */
/* Sets layer's row of the slot table: expert e of that layer lives in slot
 * host_table[e] (host array of E int32). Every entry must be in [0, n_slots)
 * and the E entries distinct; else SMOE_ERANGE and nothing is written. The
 * copy is enqueued on stream and this call waits for it, so host_table may be
 * reused on return. Corresponds to the pages' slot pool: which slot holds
 * which expert. Changing the table never changes results (bit-identical). */
SMOE_API int set_slot_table(smoe_ctx *ctx, int32_t layer, const int32_t *host_table, void *stream);

/* Bytes of scratch that moe_route / moe_forward need for T tokens. The caller
 * allocates it on the device and zero-fills it once before first use; every
 * call leaves its counters at zero again, so it can be reused without
 * clearing. Calls that use the same workspace must not overlap on the GPU. */
SMOE_API uint64_t smoe_workspace_bytes(const smoe_ctx *ctx, int32_t T);

/* --------------------------------------------------------------- moe_route */
/* Router for T tokens: logits z = W_r x (+ logit_bias), softmax, top-k with
 * ties to the lower id, renormalised weights, and the shared-expert gate.
 * The pages: every layer routes each token to 10 of 512 experts (80B model)
 * or 8 of 256 (35B model), with the router kept resident (xix.ai article,
 * paragraph on how it works; agentlenshq article, section on how expert
 * streaming works). The softmax, the renormalisation over the chosen k, the
 * tie rule and the sigmoid gate of the shared expert are this library's
 * reading; the pages do not spell them out.
 *   W_r   bf16 [E][H] device   router rows
 *   w_s   bf16 [H]    device   shared-expert gate vector
 *   x     bf16 [T][H] device   token activations
 *   logit_bias fp32 [E] device or NULL, added to the logits
 *   ids   int32 [T][k] device  out: chosen experts, descending probability
 *   w     fp32  [T][k] device  out: renormalised weights (sum to 1 per token)
 *   gate  fp32  [T]    device  out: sigmoid(w_s . x)
 * Logits are accumulated in fp32. Errors: SMOE_EINVAL, SMOE_ENOMEM
 * (workspace), SMOE_ECUDA (launch). */
SMOE_API int moe_route(const smoe_ctx *ctx, const uint16_t *W_r, const uint16_t *w_s,
              const uint16_t *x, int32_t T, const float *logit_bias,
              int32_t *ids, float *w, float *gate,
              void *workspace, uint64_t workspace_bytes, void *stream);

/* ------------------------------------------------------------- moe_forward */
/* The expert part of the layer for T tokens given their routing (the pages:
 * each chosen routed expert is fetched whole from a fixed-size slot, one read
 * per expert, while the shared experts stay resident; an expert read from the
 * cache or from storage gives exactly the same answer -- xix.ai article,
 * paragraphs on how it works and on correctness; agentlenshq article, section
 * on how expert streaming works):
 *   out[t] = sum_{j<k} w[t][j] f_{ids[t][j]}(x_t) + gate[t] f_shared(x_t)
 *            (+ residual[t] if residual != NULL), rounded once to bf16.
 * Routed expert e of `layer` is read from pool + table[layer][e] * blob_bytes;
 * the shared expert from shared_blob (one blob of the same layout).
 *   x        bf16 [T][H] device
 *   ids, w, gate   as written by moe_route (device)
 *   pool     device, pool_bytes >= n_slots * blob_bytes
 *   residual bf16 [T][H] device or NULL
 *   out      bf16 [T][H] device (may alias residual, not x)
 *   err      int32 device error word; the first device-side problem stores a
 *            SMOE_DEV_* code there (the expert concerned contributes zero) and
 *            nothing traps. Read it with smoe_check().
 * Partial sums are fp32 and are combined in a fixed order (route order for
 * each token, then the shared term), so the result does not depend on
 * scheduling, slot placement or run: bit-identical across runs and slot
 * permutations. T <= 8 takes the fused decode kernel (weights exact, fp32
 * intermediates); larger T the token-bucketed path, whose tensor-core GEMMs
 * take fp16 operands (dequantised weights, x, h) and stores each expert's
 * output in fp16 before the weighted combine, so it needs |x| < 65504 (else
 * SMOE_DEV_RANGE in the error word). Errors: SMOE_EINVAL, SMOE_ENOMEM,
 * SMOE_ECUDA. */
SMOE_API int moe_forward(const smoe_ctx *ctx, int32_t layer, const uint16_t *x, int32_t T,
                const int32_t *ids, const float *w, const float *gate,
                const void *pool, uint64_t pool_bytes, const void *shared_blob,
                const uint16_t *residual, uint16_t *out,
                void *workspace, uint64_t workspace_bytes, int32_t *err, void *stream);

/* -------------------------------------------------- moe_forward_noalloc */
/* moe_forward for T <= 8 without a workspace, for callers that cannot
 * allocate device memory: code handed only its input and output buffers by a
 * host framework that owns all device memory (plugin or custom-operator
 * interfaces), or loops that must never allocate because an allocation can
 * synchronise the device. The pages describe no such interface; it has no
 * counterpart there. Arguments and results are those of moe_forward minus
 * the workspace. The scratch (arrival tickets and per-expert outputs) lives
 * in one fixed 8 MiB array inside the library, which every GPU that loads the
 * library holds until the process exits; a call needing more than that
 * ((min(E, T*k) + 1) * T * H * 4 bytes plus 256) returns SMOE_ENOMEM, and
 * T > 8 returns SMOE_ENOTSUP. The first call on a device looks up the
 * array's device address (make that first call before any stream capture);
 * every call clears the tickets on `stream` before launching. All calls share
 * the one array, so calls that overlap on the GPU (other streams, other
 * threads) race and give wrong results: serialise them. */
SMOE_API int moe_forward_noalloc(const smoe_ctx *ctx, int32_t layer, const uint16_t *x, int32_t T,
                                 const int32_t *ids, const float *w, const float *gate,
                                 const void *pool, uint64_t pool_bytes, const void *shared_blob,
                                 const uint16_t *residual, uint16_t *out, int32_t *err, void *stream);

/* ----------------------------------------------------- moe_decode_stack */
/* One decode step for ONE token through n_layers consecutive layers
 * (first_layer .. first_layer + n_layers - 1 of the context), each layer being
 * moe_route followed by moe_forward with the residual added:
 *   x_{l+1} = bf16(x_l + sum_j w_j f_{ids_j}(x_l) + gate f_shared(x_l)),
 * the residual stacking of a decode step (the layers run one after the
 * other for each new token: xix.ai article, paragraph on how it works). The
 * whole step is one persistent launch (one CTA per SM, cooperative) instead of
 * kernel boundaries: per layer the CTAs exchange the router logits, the
 * SwiGLU values and the layer's output through the workspace, each value
 * polled where it is needed. The routing rule and its fp32 arithmetic are
 * moe_route's, so ids, w and gate equal what moe_route returns for the same
 * x_l.
 *   W_r, w_s      HOST arrays of n_layers device pointers: each layer's router
 *                 rows (bf16 [E][H]) and shared-gate vector (bf16 [H]); the
 *                 pointers are copied into the launch, the arrays may be
 *                 freed when the call returns
 *   shared_blobs  HOST array of n_layers device pointers to the layers'
 *                 shared-expert blobs
 *   logit_bias    fp32 [E] device or NULL (the same for every layer)
 *   xs            bf16 [n_layers + 1][H] device: xs[0] is the input (read),
 *                 xs[l + 1] receives layer l's output
 *   ids, w        int32 / fp32 [n_layers][k] device, out: each layer's routing
 *   gate          fp32 [n_layers] device, out
 *   pool          as for moe_forward
 *   workspace     device, >= smoe_stack_workspace_bytes(ctx, n_layers) bytes;
 *                 the call initialises it itself (no clearing needed)
 *   err           device error word as for moe_forward; a wait for other
 *                 CTAs' results that gives up (2 s) stores SMOE_DEV_TIMEOUT
 * Expert arithmetic is the decode kernel's (exact weights, fp32 partials, h
 * as bf16 hi + lo); the partial sums are combined in a fixed order, so the
 * step is bit-identical across runs. A result whose bits are all ones (a
 * NaN) is stored as the canonical NaN 0x7FFF. Needs E % 4 == 0, E <= 512,
 * 1 <= n_layers <= 64 and a GPU with cooperative launch and enough shared
 * memory (see
 * smoe_ctx_describe); otherwise SMOE_ENOTSUP. Errors: SMOE_EINVAL,
 * SMOE_ENOMEM, SMOE_ENOTSUP, SMOE_ECUDA. The pages describe one MoE layer at a
 * time; running a step's layers in one launch is this library's. */
SMOE_API int moe_decode_stack(const smoe_ctx *ctx, int32_t first_layer, int32_t n_layers,
                              const uint16_t *const *W_r, const uint16_t *const *w_s,
                              const void *const *shared_blobs, const float *logit_bias,
                              uint16_t *xs, int32_t *ids, float *w, float *gate,
                              const void *pool, uint64_t pool_bytes,
                              void *workspace, uint64_t workspace_bytes, int32_t *err, void *stream);

/* Workspace bytes moe_decode_stack needs for n_layers layers (0 if the
 * context cannot run it). */
SMOE_API uint64_t smoe_stack_workspace_bytes(const smoe_ctx *ctx, int32_t n_layers);

/* Failure-detection hook (for tests; both settings are off by default).
 * grid_wait_ns sets how long a wait of moe_decode_stack for other CTAs'
 * results (router logits, SwiGLU values, a layer's output) may last on this
 * context before it gives up (0: the default two seconds). With
 * stall_layer >= 0, the wait for that layer's router logits (the layer
 * counted from the call's first_layer) also asks for a word that nothing
 * writes, so its limit runs out: the CTA that gives up first stores
 * SMOE_DEV_TIMEOUT in the error word and raises the step's abort word, the
 * other CTAs' waits end on it, every CTA still waits for its own bulk copies
 * (their limit stays at two seconds) and the launch ends normally; the
 * step's outputs from that layer on are undefined. stall_layer = -1 turns
 * the stall off. Affects calls made after it. The pages describe no such
 * hook. Errors: SMOE_EINVAL. */
SMOE_API int smoe_set_stack_wait(smoe_ctx *ctx, uint64_t grid_wait_ns, int32_t stall_layer);

/* Waits for stream, reads the error word (then clears it to 0) and returns
 * SMOE_OK, SMOE_EDEVICE if a kernel stored a code (copied to *code if
 * non-NULL), or SMOE_ECUDA. Not for use inside graph capture. */
SMOE_API int smoe_check(int32_t *err_dev, int32_t *code, void *stream);

/* Writes a one-line description of the kernel configuration the context
 * chose (cluster size, ring stages, shared memory, co-resident clusters) into
 * buf (NUL-terminated, at most len bytes). Errors: SMOE_EINVAL. */
SMOE_API int smoe_ctx_describe(const smoe_ctx *ctx, char *buf, int32_t len);

/* Profiling hook. events: up to 4 caller-created cudaEvent_t (as void*), or
 * NULL/n = 0 to turn it off. While set, each moe_forward on this context
 * records them on its stream (as external events, so they also become event
 * nodes when the stream is being captured): events[0] before the dominant
 * kernel, events[1] after it -- the fused decode kernel for T <= 8, the
 * grouped gate/up GEMM otherwise -- and, for T > 8, events[2] after the
 * grouped down GEMM; moe_decode_stack records events[0] and events[1]
 * around its one kernel. The library keeps the pointers, not the events.
 * Errors: SMOE_EINVAL. */
SMOE_API int smoe_set_profile_events(smoe_ctx *ctx, void *const *events, int32_t n);

/* The same layer as moe_forward, computed plainly for checking the fast
 * kernels on the device: one CTA per token, each weight decoded on its own
 * from the blob (s * q + b in fp32), fp32 dot products, the routed experts in
 * route order then the shared expert, one bf16 rounding. Slow (about a
 * millisecond per token at H = 2048); no workspace. Arguments and errors as
 * for moe_forward (bad ids and slots set the error word and are skipped). */
SMOE_API int moe_forward_debug(const smoe_ctx *ctx, int32_t layer, const uint16_t *x, int32_t T,
                               const int32_t *ids, const float *w, const float *gate, const void *pool,
                               uint64_t pool_bytes, const void *shared_blob, const uint16_t *residual,
                               uint16_t *out, int32_t *err, void *stream);

/* ------------------------------------------------------- streaming slot pool */
/* A cache of experts: the context's n_slots device slots hold a changing
 * subset of all n_layers * E experts, whose packed blobs (pack_experts layout,
 * one stride each) sit in host memory in [layer][expert] order; pinned host
 * memory lets the copies run at the link's rate. The cache owns the context's
 * slot table from creation on: entries of experts that are not resident are
 * -1, so a moe_forward that names one sets SMOE_DEV_BAD_SLOT instead of
 * reading another expert's weights. Results are bit-identical to a fully
 * resident pool (they do not depend on slot placement). Use per layer:
 * moe_route, read its ids to the host (which waits for the stream), then
 * smoe_cache_prepare, then moe_forward on the same stream. The pages' slot
 * pool fed from storage with an LFU + recency cache (xix.ai article, how it
 * works; agentlenshq article, how expert streaming works). */
typedef struct smoe_cache smoe_cache;

/* host_store: host, >= n_layers * E * stride bytes; pool: device, the
 * context's n_slots slots (>= n_slots * stride bytes), both caller-owned and
 * outliving the cache. Clears the context's slot table (asynchronously on
 * stream). Errors: SMOE_EINVAL, SMOE_ENOMEM, SMOE_ECUDA. */
SMOE_API int smoe_cache_create(smoe_ctx *ctx, const void *host_store, uint64_t host_bytes, void *pool,
                               uint64_t pool_bytes, void *stream, smoe_cache **out);
SMOE_API int smoe_cache_destroy(smoe_cache *cache);

/* Makes experts ids[0..n) (host memory, any order, repeats allowed) of `layer`
 * resident. A miss takes a free slot, else evicts the resident expert used
 * least often, ties to the one used least recently, never one named by this
 * request; its blob is copied host -> device (one cudaMemcpyAsync per blob,
 * on up to four internal streams that start after the work already queued on
 * stream and that stream waits for) and the changed slot-table rows are
 * rewritten, all asynchronously with respect to the host. The host mirror of the table is reused by the next call, so call
 * again only after the stream has passed this call's copies (reading the next
 * layer's ids to the host ensures it). hits/misses (nullable): this call's
 * counts, one per entry of ids. Errors: SMOE_EINVAL (layer or an id out of
 * range), SMOE_ENOMEM (more distinct experts than slots), SMOE_ECUDA. */
SMOE_API int smoe_cache_prepare(smoe_cache *cache, int32_t layer, const int32_t *ids, int32_t n, void *stream,
                                int32_t *hits, int32_t *misses);

/* Totals since creation: entries found resident, entries copied in, bytes copied. */
SMOE_API int smoe_cache_stats(const smoe_cache *cache, uint64_t *hits, uint64_t *misses, uint64_t *bytes_copied);

/* The replacement policy alone, on the host (no device, no copies): runs
 * n_requests records [layer, n, id_0 .. id_{n-1}] (concatenated in requests)
 * through a fresh policy with n_slots slots and writes the slot of every
 * requested id, in order, to out_slots; hits/misses totals (nullable).
 * Errors: SMOE_EINVAL, SMOE_ENOMEM. */
SMOE_API int smoe_cache_simulate(int32_t n_layers, int32_t E, int64_t n_slots, const int32_t *requests,
                                 int32_t n_requests, int32_t *out_slots, int64_t *hits, int64_t *misses);

/* Shape of a Gated DeltaNet layer: n_k query/key heads and n_v value heads
 * (n_v a multiple of n_k; value head h reads query/key head h / (n_v / n_k)),
 * key width d_k and value width d_v. */
typedef struct smoe_gdn_shape {
    int32_t nk, nv, dk, dv;
} smoe_gdn_shape;

/* T recurrence steps of a Gated DeltaNet layer for B sequences, in order,
 * on a state held in device memory (the linear-attention layers that make up
 * three quarters of the hybrid model and keep a fixed-size state instead of a
 * growing KV cache: xix.ai article, paragraph on the forward pass; agentlenshq
 * article, section on how expert streaming works). The pages do not spell the
 * rule out; this is the gated delta rule with L2-normalised q and k. Per
 * sequence b, value head h, token t, with S = state[b][h] (d_v x d_k):
 *   k^ = k / sqrt(sum k^2 + 1e-6),  q^ = scale * q / sqrt(sum q^2 + 1e-6),
 *   S <- exp(g) S + beta (v - exp(g) S k^) k^T,  o = S q^.
 * All device pointers, 16-byte aligned, row-major:
 *   q, k  bf16 [T][B][n_k][d_k];   v, out  bf16 [T][B][n_v][d_v];
 *   g, beta  fp32 [T][B][n_v] (g the log decay, beta the write strength);
 *   state  fp32 [B][n_v][d_v][d_k], read and updated in place (caller-owned).
 * scale <= 0 means 1 / sqrt(d_k). Arithmetic is fp32; out is rounded to bf16.
 * Supported: d_k in {32, 64, 128}, d_v a multiple of 4 up to 1024; others
 * return SMOE_ENOTSUP. B = 0 or T = 0 does nothing. Asynchronous on stream.
 * Errors: SMOE_EINVAL (null, misaligned, n_v not a multiple of n_k),
 * SMOE_ENOTSUP, SMOE_ECUDA. */
SMOE_API int gdn_step(const smoe_gdn_shape *shape, int32_t B, int32_t T, const uint16_t *q, const uint16_t *k,
                      const uint16_t *v, const float *g, const float *beta, float scale, float *state,
                      uint16_t *out, void *stream);

/* Short English text for a status code (static storage). */
SMOE_API const char *smoe_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* SMOE_H */
