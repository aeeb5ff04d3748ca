// noalloc.cu -- moe_forward_noalloc: the decode path of moe_forward for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that is handed only its input and
// output buffers by a host framework that owns all device memory (plugin or
// custom-operator interfaces of serving engines), and loops that must never
// allocate because an allocation can synchronise the device and stall them.
// For those callers this entry point takes the fused decode kernel's scratch
// (per-expert outputs and arrival tickets) from a fixed array compiled into
// the library instead of from a caller-provided workspace.
#include <mutex>

#include "smoe_dev.cuh"
#include "smoe_internal.h"

using namespace smoe;

namespace {

// Scratch for the decode kernel: 256 bytes of arrival tickets, then the
// per-expert outputs. Every GPU that loads the library holds it until exit.
constexpr uint64_t kNoAllocScratchBytes = 8ull << 20;   // 8 MiB
constexpr uint64_t kTicketBytes = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device

// In host code g_noalloc_scratch names a host-side stand-in, not device
// memory; the kernel must be given the address the runtime reports for the
// current device. Looked up once per device, on that device's first call.
int scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMOE_ECUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SMOE_ECUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SMOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int moe_forward_noalloc(const smoe_ctx *ctx, int32_t layer, const uint16_t *x, int32_t T,
                                   const int32_t *ids, const float *w, const float *gate, const void *pool,
                                   uint64_t pool_bytes, const void *shared_blob, const uint16_t *residual,
                                   uint16_t *out, int32_t *err, void *stream)
{
    if (!ctx || T < 0) return SMOE_EINVAL;
    if (layer < 0 || layer >= ctx->n_layers) return SMOE_EINVAL;
    if (!ctx->decode_ok) return SMOE_ENOTSUP;        // no T <= 8 kernel for this shape's atoms
    if (T == 0) return SMOE_OK;                      // nothing to do; the buffers may be null
    if (!x || !ids || !w || !gate || !pool || !shared_blob || !out || !err) return SMOE_EINVAL;
    if (T > kDecodeMaxT) return SMOE_ENOTSUP;
    if (!aligned16(x) || !aligned16(pool) || !aligned16(shared_blob) || !aligned16(out) ||
        (residual && !aligned16(residual)))
        return SMOE_EINVAL;
    if (pool_bytes < uint64_t(ctx->n_slots) * ctx->layout.blob) return SMOE_ENOMEM;
    const smoe_shape &s = ctx->shape;
    const uint64_t umax = uint64_t(s.E < T * s.k ? s.E : T * s.k) + 1;
    const uint64_t need = kTicketBytes + umax * uint64_t(T) * s.H * 4;
    if (need > kNoAllocScratchBytes) return SMOE_ENOMEM;    // the fixed scratch is too small for this call
    void *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the tickets must start at zero; the array keeps whatever the last call left
    if (cudaMemsetAsync(scratch, 0, kTicketBytes, st) != cudaSuccess) return SMOE_ECUDA;
    DecodeParams p = {};
    p.x = x;
    p.ids = ids;
    p.w = w;
    p.gate = gate;
    p.pool = static_cast<const uint8_t *>(pool);
    p.shared_blob = static_cast<const uint8_t *>(shared_blob);
    p.table_row = ctx->table_dev + size_t(layer) * s.E;
    p.residual = residual;
    p.out = out;
    p.counters = static_cast<uint32_t *>(scratch);
    p.ypair = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + kTicketBytes);
    p.err = err;
    p.stride = ctx->layout.blob;
    p.n_slots = ctx->n_slots;
    p.T = T;
    p.H = s.H;
    p.E = s.E;
    p.k = s.k;
    p.I = s.I;
    return launch_decode(ctx, p, st) == cudaSuccess ? SMOE_OK : SMOE_ECUDA;
}
