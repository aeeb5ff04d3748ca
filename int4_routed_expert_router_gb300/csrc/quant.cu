// quant.cu -- smoe_quantize_mlx: float weights -> MLX-style affine triples
// (q, s, b) in the layout pack_experts reads, on the host.
//
// Per group of 64 consecutive columns of a row: b = the group minimum rounded
// down to fp16, s = (maximum - b) / (2^bits - 1) rounded up to fp16, so that
// [b, b + (2^bits - 1) s] holds the group; q = (w - b) / s rounded to the
// nearest integer (ties to even), clamped to [0, 2^bits - 1]; a group of one
// value gets s = 0 and q = 0. Every step is in double precision. The pages
// name MLX int4 and int8 group quantisation with a scale and a bias per group
// of 64 (xix.ai article, last paragraph) but do not define the quantiser; the
// rounding directions are this library's reading (dequantisation error at
// most s / 2).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "smoe.h"

namespace {

// The fp16 value next to v in direction dir (-1: the largest fp16 <= v,
// +1: the smallest fp16 >= v), as bits; v finite with |v| <= 65504.
uint16_t fp16_directed(double v, int dir)
{
    if (v == 0.0) return 0;
    int e2 = 0;
    std::frexp(std::fabs(v), &e2);          // |v| in [2^(e2 - 1), 2^e2)
    int ex = e2 - 1;
    if (ex < -14) ex = -14;                 // below the normal range the spacing stays 2^-24
    const double ulp = std::ldexp(1.0, ex - 10);
    const double m = v / ulp;               // exact: a power-of-two scaling
    const double r = dir < 0 ? std::floor(m) : std::ceil(m);
    const bool neg = r < 0.0;
    double a = std::fabs(r);
    if (a >= 2048.0) {                      // rounded up into the next binade
        a /= 2.0;
        ex += 1;
    }
    if (a == 0.0) return neg ? 0x8000 : 0;
    const uint32_t ai = uint32_t(a);
    const uint16_t bits = ai >= 1024 ? uint16_t((uint32_t(ex + 15) << 10) | (ai - 1024)) : uint16_t(ai);
    return neg ? uint16_t(bits | 0x8000) : bits;
}

double fp16_value(uint16_t h)
{
    const int ex = (h >> 10) & 31, man = h & 1023;
    const double mag = ex == 0 ? std::ldexp(double(man), -24) : std::ldexp(double(1024 + man), ex - 25);
    return (h & 0x8000) ? -mag : mag;
}

}  // namespace

extern "C" int smoe_quantize_mlx(const float *w, int32_t rows, int32_t cols, int32_t bits, uint32_t *q, uint16_t *s,
                                 uint16_t *b)
{
    if (rows < 0 || cols < 0) return SMOE_EINVAL;
    if (bits != 4 && bits != 8) return SMOE_ENOTSUP;
    if (cols % 64) return SMOE_ENOTSUP;
    if (rows == 0 || cols == 0) return SMOE_OK;
    if (!w || !q || !s || !b) return SMOE_EINVAL;
    const int per_word = 32 / bits;                      // values per uint32
    const double top = double((1 << bits) - 1);
    const size_t wpr = size_t(cols) / per_word, gpr = size_t(cols) / 64;
    for (int32_t r = 0; r < rows; ++r) {
        const float *row = w + size_t(r) * cols;
        for (size_t g = 0; g < gpr; ++g) {
            const float *v = row + g * 64;
            double lo = v[0], hi = v[0];
            for (int c = 1; c < 64; ++c) {
                lo = std::fmin(lo, double(v[c]));
                hi = std::fmax(hi, double(v[c]));
            }
            if (!std::isfinite(lo) || !std::isfinite(hi) || std::fabs(lo) > 65504.0 || std::fabs(hi) > 65504.0)
                return SMOE_ERANGE;                          // outside what an fp16 bias and scale can cover
            const uint16_t bb = fp16_directed(lo, -1);
            const double bv = fp16_value(bb);
            const double span = (hi - bv) / top;
            if (span > 65504.0) return SMOE_ERANGE;
            const uint16_t sb = fp16_directed(span, +1);
            const double sv = fp16_value(sb);
            s[size_t(r) * gpr + g] = sb;
            b[size_t(r) * gpr + g] = bb;
            uint32_t *out = q + size_t(r) * wpr + g * (64 / per_word);
            for (int wd = 0; wd < 64 / per_word; ++wd) {
                uint32_t word = 0;
                for (int j = 0; j < per_word; ++j) {
                    double t = sv > 0.0 ? std::nearbyint((double(v[wd * per_word + j]) - bv) / sv) : 0.0;
                    t = t < 0.0 ? 0.0 : (t > top ? top : t);
                    word |= uint32_t(t) << (bits * j);
                }
                out[wd] = word;
            }
        }
    }
    return SMOE_OK;
}
