// synth.cu -- device side of the seeded input generator (see synthetic/__init__.py).
//
// Produces the MLX affine 4-bit (or 8-bit) triples of many experts directly in device
// memory with the same counter-based recipe as the numpy generator, so the
// tens-of-GB expert pools never cross PCIe/C2C. Holds none of the MoE layer's
// arithmetic: only the SplitMix64 output mix (Steele, Lea, Flood, OOPSLA 2014)
// and round-to-nearest-even conversion of a double to fp16.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t stream_key(uint64_t seed, int tid, int layer, int code)
{
    const uint64_t tag = (uint64_t(tid) << 52) | (uint64_t(layer) << 26) | uint64_t(code);
    return mix64((seed * kGolden) ^ tag);
}

__device__ __forceinline__ uint64_t value(uint64_t key, uint64_t i) { return mix64(key + kGolden * (i + 1)); }

// IEEE binary64 -> binary16, nearest with ties to even (finite inputs).
__device__ uint16_t f64_to_f16(double v)
{
    const uint64_t bits = uint64_t(__double_as_longlong(v));
    const uint16_t sign = uint16_t((bits >> 63) << 15);
    const int e = int((bits >> 52) & 0x7ff) - 1023;
    const uint64_t mant = bits & ((1ull << 52) - 1);
    if (e > 15) return sign | 0x7c00;
    uint64_t sig;
    int shift;
    uint16_t ebits;
    if (e >= -14) {            // normal result
        sig = mant;
        shift = 42;
        ebits = uint16_t(e + 15);
    } else {                   // subnormal result: quantum 2^-24
        if (e < -25) return sign;
        sig = mant | (1ull << 52);
        shift = 42 + (-14 - e);
        ebits = 0;
    }
    uint64_t m = sig >> shift;
    const uint64_t rem = sig & ((1ull << shift) - 1), half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (m & 1))) ++m;
    uint32_t out = (uint32_t(ebits) << 10) + uint32_t(m);   // carry into the exponent is correct
    if (out >= 0x7c00) return sign | 0x7c00;
    return sign | uint16_t(out);
}

__device__ __forceinline__ double f16_to_f64(uint16_t h)
{
    const int e = (h >> 10) & 31, m = h & 1023;
    double v = e == 0 ? ldexp(double(m), -24) : ldexp(1.0 + m / 1024.0, e - 15);
    return (h & 0x8000) ? -v : v;
}

struct Job {
    uint32_t *q[3];
    uint16_t *s[3];
    uint16_t *b[3];
};

__global__ void q_kernel(uint64_t seed, int layer, int code0, int n, int H, int I, int bits, Job job)
{
    const int per = 32 / bits;                       // values per word: 8 (4-bit) or 4 (8-bit)
    const int wq[3] = {I * (H / per), I * (H / per), H * (I / per)};
    for (int ex = 0; ex < n; ++ex)
        for (int m = 0; m < 3; ++m) {
            const uint64_t key = stream_key(seed, 1 + 2 * m, layer, code0 + ex);
            uint32_t *q = job.q[m] + size_t(ex) * wq[m];
            const long long npair = wq[m] / 2;
            for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < npair;
                 i += (long long)gridDim.x * blockDim.x) {
                const uint64_t v = value(key, uint64_t(i));
                reinterpret_cast<uint2 *>(q)[i] = make_uint2(uint32_t(v), uint32_t(v >> 32));
            }
        }
}

__global__ void sb_kernel(uint64_t seed, int layer, int code0, int n, int H, int I, int bits, Job job)
{
    const int ng[3] = {I * (H / 64), I * (H / 64), H * (I / 64)};
    for (int ex = 0; ex < n; ++ex)
        for (int m = 0; m < 3; ++m) {
            const uint64_t key = stream_key(seed, 2 + 2 * m, layer, code0 + ex);
            uint16_t *s = job.s[m] + size_t(ex) * ng[m];
            uint16_t *b = job.b[m] + size_t(ex) * ng[m];
            for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < ng[m];
                 i += (long long)gridDim.x * blockDim.x) {
                const uint64_t v = value(key, uint64_t(i));
                const double u = double(v >> 40) / 16777216.0;
                double s64 = __dadd_rn(0.002, __dmul_rn(0.004, u));
                if (bits == 8) s64 = __ddiv_rn(s64, 17.0);   // the 8-bit recipe's scale
                const uint16_t sh = f64_to_f16(s64);
                s[i] = sh;
                b[i] = f64_to_f16(__dmul_rn(bits == 8 ? -127.5 : -7.5, f16_to_f64(sh)));
            }
        }
}

}  // namespace

// Triples of experts code0 .. code0+n-1 of `layer` (code 2^26-1 = shared
// expert). Output arrays hold the n experts back to back, each in MLX layout:
// q[0], q[1] [I][H/8], q[2] [H][I/8] (8 bits: [I][H/4], [H][I/4]);
// s/b[0..1] [I][H/64], s/b[2] [H][I/64]. bits: 4 or 8. Returns 0 or a cudaError_t.
extern "C" int synth_expert_triples_bits(uint64_t seed, int layer, int code0, int n, int H, int I, int bits,
                                         uint32_t *gq, uint16_t *gs, uint16_t *gb, uint32_t *uq, uint16_t *us,
                                         uint16_t *ub, uint32_t *dq, uint16_t *ds, uint16_t *db, void *stream)
{
    if (bits != 4 && bits != 8) return int(cudaErrorInvalidValue);
    Job job = {{gq, uq, dq}, {gs, us, ds}, {gb, ub, db}};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    q_kernel<<<1024, 256, 0, st>>>(seed, layer, code0, n, H, I, bits, job);
    sb_kernel<<<256, 256, 0, st>>>(seed, layer, code0, n, H, I, bits, job);
    return int(cudaGetLastError());
}

extern "C" int synth_expert_triples(uint64_t seed, int layer, int code0, int n, int H, int I, uint32_t *gq,
                                    uint16_t *gs, uint16_t *gb, uint32_t *uq, uint16_t *us, uint16_t *ub,
                                    uint32_t *dq, uint16_t *ds, uint16_t *db, void *stream)
{
    return synth_expert_triples_bits(seed, layer, code0, n, H, I, 4, gq, gs, gb, uq, us, ub, dq, ds, db, stream);
}
