/*
 * smoe_oracle.c -- CPU oracle for the int4 routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do. It is deliberately plain, slow and single-threaded: every
 * value is computed in double precision (fp64) in the order the definition
 * states, so that a reader can check it against the pages by eye. It shares
 * no code, header, table or constant with the CUDA library.
 *
 * What it computes (the sparse MoE layer of the Qwen3-Next / Qwen3.5-3.6
 * hybrid models that Swiftlet runs):
 *   - "Swiftlet Packs 80B Qwen Into Mac..." (xix.ai), paragraph on how it works:
 *     each layer routes each token to 10 of 512 experts (80B) or 8 of 256 (35B);
 *     the router and the shared experts stay resident at 4 bits; routed experts
 *     are fixed-stride blobs read one per expert into a bounded slot pool.
 *   - same page, last paragraph: MLX-style int4/int8 group quantisation with
 *     byte-addressable kernels and 64-bit offsets.
 *   - "Swiftletは低RAM使用量で..." (agentlenshq.com), section on correctness:
 *     kernels are checked against an exact CPU reference, and an expert read
 *     from the cache or from disk gives the same answer.
 * The pages leave the following open; the readings taken here are:
 *   - routing: p = softmax(z) over all E logits, the k largest p are chosen
 *     (ties to the lower expert id), and their weights are renormalised to sum
 *     to one;
 *   - experts: SwiGLU MLP  y = D (silu(G x) * (U x)),  silu(v) = v / (1 + e^-v);
 *   - shared expert: same MLP, scaled by sigmoid(w_s . x), a scalar per token;
 *   - quantisation: MLX affine 4-bit, group 64 along the input dimension,
 *     fp16 scale s and bias b per group, w = s*q + b, 8 nibbles per uint32 with
 *     column c of a row in bits 4*(c%8)..4*(c%8)+3 of word c/8;
 *   - output: out = sum_j w_j y_{e_j} (j in route order) + gate * y_shared,
 *     rounded once to bf16 (nearest, ties to even).
 * The dequantised weight s*q + b is exact in fp64 (an 11-bit significand times
 * a 4-bit integer plus an 11-bit significand), so no rounding is introduced
 * before the dot products.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_GROUP 64

/* ------------------------------------------------------------ conversions */

/* bf16 bits -> value: bf16 is the upper half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp16 bits -> value, from the IEEE binary16 definition. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Round v to a binary format with `mant` stored mantissa bits and minimum
 * normal exponent `emin`, nearest with ties to even; returns the rounded value
 * (possibly +-inf). */
static double round_to_format(double v, int mant, int emin, double maxfinite)
{
    if (v == 0.0 || isnan(v) || isinf(v))
        return v;
    int ex;
    frexp(v, &ex);                 /* |v| = f * 2^ex, 0.5 <= f < 1 */
    int lead = ex - 1;             /* exponent of the leading bit */
    if (lead < emin)
        lead = emin;               /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, lead - mant);
    double r = nearbyint(v / quantum) * quantum;   /* default mode: ties-to-even */
    if (fabs(r) > maxfinite)
        return v > 0 ? INFINITY : -INFINITY;
    return r;
}

uint16_t orc_f64_to_bf16(double v)
{
    double r = round_to_format(v, 7, -126, 0x1.fep127);
    float f = (float)r;            /* exact: r is representable in bf16 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(v))
        return 0x7fc0;
    return (uint16_t)(u >> 16);
}

uint16_t orc_f64_to_f16(double v)
{
    if (isnan(v))
        return 0x7e00;
    double r = round_to_format(v, 10, -14, 65504.0);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isinf(a))
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    if (a < ldexp(1.0, -14))
        return sign | (uint16_t)(a / ldexp(1.0, -24));       /* subnormal */
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    uint16_t m = (uint16_t)((a / ldexp(1.0, e) - 1.0) * 1024.0);
    return sign | (uint16_t)((e + 15) << 10) | m;
}

/* --------------------------------------------------------- dequantisation */

/* W[r][c] = s[r][c/64] * q + b[r][c/64], q = nibble c%8 of word q[r][c/8]. */
void orc_dequant_mlx(const uint32_t *q, const uint16_t *s, const uint16_t *b,
                     int rows, int cols, double *W)
{
    int wpr = cols / 8, gpr = cols / ORC_GROUP;
    for (int r = 0; r < rows; r++)
        for (int c = 0; c < cols; c++) {
            uint32_t word = q[(size_t)r * wpr + c / 8];
            unsigned nib = (word >> (4 * (c % 8))) & 15u;
            double sc = orc_f16_to_f64(s[(size_t)r * gpr + c / ORC_GROUP]);
            double bi = orc_f16_to_f64(b[(size_t)r * gpr + c / ORC_GROUP]);
            W[(size_t)r * cols + c] = sc * (double)nib + bi;
        }
}

/* MLX-style affine quantiser (reading taken; bit parity with MLX unpinned):
 * per group of 64, b = fp16 rounded down of min, s = fp16 rounded up of
 * (max - b)/15, q = clamp(round_half_even((w - b)/s), 0, 15). The covered range
 * [b, b + 15 s] contains [min, max], so |w - (s q + b)| <= s/2. */
static uint16_t f16_round_dir(double v, int up)
{
    uint16_t h = orc_f64_to_f16(v);
    double hv = orc_f16_to_f64(h);
    if (up && hv < v)
        h = (h & 0x8000) ? (uint16_t)(h - 1) : (uint16_t)(h + 1);
    else if (!up && hv > v)
        h = (h & 0x8000) ? (uint16_t)(h + 1) : (h == 0 ? 0x8001 : (uint16_t)(h - 1));
    return h;
}

void orc_quantize_mlx(const double *W, int rows, int cols,
                      uint32_t *q, uint16_t *s, uint16_t *b)
{
    int wpr = cols / 8, gpr = cols / ORC_GROUP;
    memset(q, 0, sizeof(uint32_t) * (size_t)rows * wpr);
    for (int r = 0; r < rows; r++)
        for (int g = 0; g < gpr; g++) {
            const double *w = W + (size_t)r * cols + g * ORC_GROUP;
            double lo = w[0], hi = w[0];
            for (int c = 1; c < ORC_GROUP; c++) {
                if (w[c] < lo) lo = w[c];
                if (w[c] > hi) hi = w[c];
            }
            uint16_t bb = f16_round_dir(lo, 0);
            double bv = orc_f16_to_f64(bb);
            uint16_t ss = f16_round_dir((hi - bv) / 15.0, 1);
            double sv = orc_f16_to_f64(ss);
            s[(size_t)r * gpr + g] = ss;
            b[(size_t)r * gpr + g] = bb;
            for (int c = 0; c < ORC_GROUP; c++) {
                double t = sv > 0 ? nearbyint((w[c] - bv) / sv) : 0.0;
                if (t < 0) t = 0;
                if (t > 15) t = 15;
                int col = g * ORC_GROUP + c;
                q[(size_t)r * wpr + col / 8] |= (uint32_t)t << (4 * (col % 8));
            }
        }
}

/* ----------------------------------------------------------------- routing */

/* For each token t: z_e = sum_h x[t][h] W_r[e][h] (+ bias_e), p = softmax(z),
 * ids = the k largest p in descending order (ties: lower e first),
 * w_j = p_{ids_j} / sum_{j'} p_{ids_j'}, gate = 1 / (1 + exp(-(w_s . x))).
 * probs (nullable) receives p [T][E]. */
void orc_route(const uint16_t *x, int T, int H, const uint16_t *Wr,
               const uint16_t *ws, int E, const float *bias, int k,
               int32_t *ids, double *w, double *gate, double *probs)
{
    double *z = malloc(sizeof(double) * E);
    double *p = malloc(sizeof(double) * E);
    char *taken = malloc((size_t)E);
    for (int t = 0; t < T; t++) {
        const uint16_t *xt = x + (size_t)t * H;
        double zmax = -INFINITY;
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int h = 0; h < H; h++)
                acc += orc_bf16_to_f64(xt[h]) * orc_bf16_to_f64(Wr[(size_t)e * H + h]);
            if (bias)
                acc += (double)bias[e];
            z[e] = acc;
            if (acc > zmax) zmax = acc;
        }
        double sum = 0.0;
        for (int e = 0; e < E; e++) {
            p[e] = exp(z[e] - zmax);
            sum += p[e];
        }
        for (int e = 0; e < E; e++)
            p[e] /= sum;
        if (probs)
            memcpy(probs + (size_t)t * E, p, sizeof(double) * E);
        memset(taken, 0, (size_t)E);
        double psum = 0.0;
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || p[e] > p[best]))
                    best = e;            /* strict '>' keeps the lower id on ties */
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
            psum += p[best];
        }
        for (int j = 0; j < k; j++)
            w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]] / psum;
        double gs = 0.0;
        for (int h = 0; h < H; h++)
            gs += orc_bf16_to_f64(xt[h]) * orc_bf16_to_f64(ws[h]);
        gate[t] = 1.0 / (1.0 + exp(-gs));
    }
    free(z);
    free(p);
    free(taken);
}

/* ------------------------------------------------------------------ experts */

/* One expert in MLX triples form. */
typedef struct orc_expert {
    const uint32_t *q[3];          /* gate [I][H/8], up [I][H/8], down [H][I/8] */
    const uint16_t *s[3];          /* fp16 bits, [rows][cols/64] */
    const uint16_t *b[3];
} orc_expert;

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* y = D (silu(G x) * (U x)) for one token, all in fp64. */
static void expert_mlp(const double *G, const double *U, const double *D,
                       int H, int I, const double *x, double *hbuf, double *y)
{
    for (int i = 0; i < I; i++) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; c++) {
            g += G[(size_t)i * H + c] * x[c];
            u += U[(size_t)i * H + c] * x[c];
        }
        hbuf[i] = silu(g) * u;
    }
    for (int o = 0; o < H; o++) {
        double acc = 0.0;
        for (int i = 0; i < I; i++)
            acc += D[(size_t)o * I + i] * hbuf[i];
        y[o] = acc;
    }
}

typedef struct dense_expert { double *G, *U, *D; } dense_expert;

static int dense_of(const orc_expert *ex, int H, int I, dense_expert *d)
{
    for (int m = 0; m < 3; m++)
        if (!ex->q[m] || !ex->s[m] || !ex->b[m])
            return -1;
    d->G = malloc(sizeof(double) * (size_t)I * H);
    d->U = malloc(sizeof(double) * (size_t)I * H);
    d->D = malloc(sizeof(double) * (size_t)H * I);
    orc_dequant_mlx(ex->q[0], ex->s[0], ex->b[0], I, H, d->G);
    orc_dequant_mlx(ex->q[1], ex->s[1], ex->b[1], I, H, d->U);
    orc_dequant_mlx(ex->q[2], ex->s[2], ex->b[2], H, I, d->D);
    return 0;
}

static void dense_free(dense_expert *d)
{
    free(d->G);
    free(d->U);
    free(d->D);
    d->G = d->U = d->D = NULL;
}

/* The full layer given the routing: for each token t,
 *   out64[t] = sum_{j=0..k-1} w[t][j] * f_{ids[t][j]}(x_t) + gate[t] * f_shared(x_t)
 * summed in route order j = 0..k-1, then the shared term; out_bf16 is out64
 * rounded once to bf16. experts[e] must hold every routed expert that ids
 * names (others may be all-NULL). Returns 0, or -1 if a needed expert is
 * missing. */
int orc_moe_combine(int T, int H, int k, int I, int Is,
                    const uint16_t *x, const int32_t *ids, const double *w,
                    const double *gate, const orc_expert *experts, int E,
                    const orc_expert *shared, double *out64, uint16_t *out_bf16)
{
    double *xt = malloc(sizeof(double) * H);
    double *y = malloc(sizeof(double) * H);
    double *hb = malloc(sizeof(double) * (I > Is ? I : Is));
    dense_expert *cache = calloc((size_t)E, sizeof(dense_expert));
    dense_expert sh = {0};
    int rc = 0;
    if (dense_of(shared, H, Is, &sh)) { rc = -1; goto done; }
    for (int t = 0; t < T && rc == 0; t++) {
        for (int c = 0; c < H; c++)
            xt[c] = orc_bf16_to_f64(x[(size_t)t * H + c]);
        double *o = out64 + (size_t)t * H;
        for (int c = 0; c < H; c++)
            o[c] = 0.0;
        for (int j = 0; j < k; j++) {
            int e = ids[(size_t)t * k + j];
            if (e < 0 || e >= E) { rc = -1; break; }
            if (!cache[e].G && dense_of(&experts[e], H, I, &cache[e])) { rc = -1; break; }
            expert_mlp(cache[e].G, cache[e].U, cache[e].D, H, I, xt, hb, y);
            for (int c = 0; c < H; c++)
                o[c] += w[(size_t)t * k + j] * y[c];
        }
        if (rc) break;
        expert_mlp(sh.G, sh.U, sh.D, H, Is, xt, hb, y);
        for (int c = 0; c < H; c++) {
            o[c] += gate[t] * y[c];
            if (out_bf16)
                out_bf16[(size_t)t * H + c] = orc_f64_to_bf16(o[c]);
        }
    }
done:
    for (int e = 0; e < E; e++)
        dense_free(&cache[e]);
    dense_free(&sh);
    free(cache);
    free(xt);
    free(y);
    free(hb);
    return rc;
}

/* x_next = bf16(x + y) elementwise (residual chaining of a layer stack). */
void orc_residual_bf16(const uint16_t *x, const double *y, size_t n, uint16_t *x_next)
{
    for (size_t i = 0; i < n; i++)
        x_next[i] = orc_f64_to_bf16(orc_bf16_to_f64(x[i]) + y[i]);
}

/* ------------------------------------------------------ expert blob format */

/* The oracle's own reader of the fixed-stride expert blob written by the
 * library's pack_experts (format spelled out in the library header and the
 * design notes). One blob = gate/up part then down part, both made of
 * 576-byte atoms; an atom holds 16 logical rows x one 64-column group:
 *   bytes [0,512): lane L = 4g+t (g<8, t<4) owns 16 bytes = four words
 *       (row g cols 16t..16t+7), (row g cols 16t+8..16t+15),
 *       (row g+8 cols 16t..16t+7), (row g+8 cols 16t+8..16t+15);
 *       a word for columns c0..c0+7 keeps column c0+2m in nibble m and column
 *       c0+2m+1 in nibble m+4 (m < 4): even columns low half, odd high half;
 *   bytes [512,576): for g<8, fp16 (s,b) of row g then (s,b) of row g+8.
 * gate/up atoms: index rb*(H/64)+kb for row block rb < I/8 and group kb;
 *   logical row g<8 is gate row 8rb+g, row g+8 is up row 8rb+g.
 * down atoms (after all gate/up atoms): index rd*(I/64)+kb, rd < H/16;
 *   logical row i is down row 16rd+i. */
#define ATOM 576

static unsigned blob_nibble(const uint8_t *atom, int row, int col)
{
    int g = row & 7, hi = row >> 3;                  /* hi: rows 8..15 */
    int t = col / 16, half = (col / 8) & 1, c0 = col & 7;
    int lane = 4 * g + t;
    int widx = 2 * hi + half;
    uint32_t word;
    memcpy(&word, atom + 16 * lane + 4 * widx, 4);
    int slot = (c0 & 1) ? 4 + c0 / 2 : c0 / 2;
    return (word >> (4 * slot)) & 15u;
}

static void blob_sb(const uint8_t *atom, int row, uint16_t *s, uint16_t *b)
{
    int g = row & 7, hi = row >> 3;
    const uint8_t *e = atom + 512 + 8 * g + 4 * hi;
    memcpy(s, e, 2);
    memcpy(b, e + 2, 2);
}

uint64_t orc_blob_bytes(int H, int I)
{
    return (uint64_t)(I / 8) * (H / ORC_GROUP) * ATOM +
           (uint64_t)(H / 16) * (I / ORC_GROUP) * ATOM;
}

/* Parse one blob into MLX triples (the 9 output arrays as in orc_expert). */
void orc_blob_to_mlx(const uint8_t *blob, int H, int I,
                     uint32_t *gq, uint16_t *gs, uint16_t *gb,
                     uint32_t *uq, uint16_t *us, uint16_t *ub,
                     uint32_t *dq, uint16_t *ds, uint16_t *db)
{
    int kbH = H / ORC_GROUP, kbI = I / ORC_GROUP;
    memset(gq, 0, sizeof(uint32_t) * (size_t)I * (H / 8));
    memset(uq, 0, sizeof(uint32_t) * (size_t)I * (H / 8));
    memset(dq, 0, sizeof(uint32_t) * (size_t)H * (I / 8));
    for (int i = 0; i < I; i++)
        for (int kb = 0; kb < kbH; kb++) {
            const uint8_t *atom = blob + ((size_t)(i / 8) * kbH + kb) * ATOM;
            for (int which = 0; which < 2; which++) {
                int row = (i % 8) + 8 * which;       /* gate: g, up: g+8 */
                uint32_t *q = which ? uq : gq;
                uint16_t *s = which ? us : gs, *b = which ? ub : gb;
                for (int c = 0; c < ORC_GROUP; c++) {
                    int col = kb * ORC_GROUP + c;
                    q[(size_t)i * (H / 8) + col / 8] |=
                        (uint32_t)blob_nibble(atom, row, c) << (4 * (col % 8));
                }
                blob_sb(atom, row, &s[(size_t)i * kbH + kb], &b[(size_t)i * kbH + kb]);
            }
        }
    const uint8_t *down = blob + (size_t)(I / 8) * kbH * ATOM;
    for (int o = 0; o < H; o++)
        for (int kb = 0; kb < kbI; kb++) {
            const uint8_t *atom = down + ((size_t)(o / 16) * kbI + kb) * ATOM;
            int row = o % 16;
            for (int c = 0; c < ORC_GROUP; c++) {
                int col = kb * ORC_GROUP + c;
                dq[(size_t)o * (I / 8) + col / 8] |=
                    (uint32_t)blob_nibble(atom, row, c) << (4 * (col % 8));
            }
            blob_sb(atom, row, &ds[(size_t)o * kbI + kb], &db[(size_t)o * kbI + kb]);
        }
}

/* The layer read through a slot table: routed expert e of this layer lives in
 * blob pool + table[e] * stride (64-bit offsets); the shared expert in its own
 * blob. Routing (ids, w, gate) comes from orc_route. Returns 0, -1 on a
 * missing/invalid slot. */
int orc_moe_combine_pool(int T, int H, int k, int I, int E,
                         const uint16_t *x, const int32_t *ids, const double *w,
                         const double *gate, const uint8_t *pool, uint64_t stride,
                         int64_t n_slots, const int32_t *table, const uint8_t *shared_blob,
                         double *out64, uint16_t *out_bf16)
{
    size_t nq_gu = (size_t)I * (H / 8), ns_gu = (size_t)I * (H / ORC_GROUP);
    size_t nq_d = (size_t)H * (I / 8), ns_d = (size_t)H * (I / ORC_GROUP);
    size_t per = 4 * (2 * nq_gu + nq_d) + 2 * 2 * (2 * ns_gu + ns_d);
    orc_expert *ex = calloc((size_t)E + 1, sizeof(orc_expert));
    uint8_t **mem = calloc((size_t)E + 1, sizeof(uint8_t *));
    int rc = 0;
    for (int n = 0; n < T * k + 1 && rc == 0; n++) {
        int e = n < T * k ? ids[n] : E;             /* E stands for the shared expert */
        if (e < 0 || e > E) { rc = -1; break; }
        if (mem[e]) continue;
        const uint8_t *blob;
        if (e == E) {
            blob = shared_blob;
        } else {
            int64_t slot = table[e];
            if (slot < 0 || slot >= n_slots) { rc = -1; break; }
            blob = pool + (uint64_t)slot * stride;
        }
        uint8_t *m = mem[e] = malloc(per);
        uint32_t *gq = (uint32_t *)m, *uq = gq + nq_gu, *dq = uq + nq_gu;
        uint16_t *gs = (uint16_t *)(dq + nq_d), *gb = gs + ns_gu, *us = gb + ns_gu,
                 *ub = us + ns_gu, *ds = ub + ns_gu, *db = ds + ns_d;
        orc_blob_to_mlx(blob, H, I, gq, gs, gb, uq, us, ub, dq, ds, db);
        orc_expert v = {{gq, uq, dq}, {gs, us, ds}, {gb, ub, db}};
        ex[e] = v;
    }
    if (rc == 0)
        rc = orc_moe_combine(T, H, k, I, I, x, ids, w, gate, ex, E, &ex[E], out64, out_bf16);
    for (int e = 0; e <= E; e++)
        free(mem[e]);
    free(mem);
    free(ex);
    return rc;
}

/* ============================================================ 8-bit experts
 * The pages name MLX-style int4/int8 group quantisation ("Swiftlet Packs 80B
 * Qwen Into Mac...", last paragraph; agentlenshq article, relation to
 * TurboFieldfare) and an 8-bit 80B run (paper-digest page, Core Mechanics).
 * Reading taken: MLX's 8-bit affine format, the same group of 64 and fp16 s,
 * b per group, w = s*q + b with q in 0..255, 4 values per uint32 (column c of
 * a row in bits 8*(c%4)..8*(c%4)+7 of word c/4). s*q + b stays exact in fp64
 * (an 11-bit significand times an 8-bit integer plus an 11-bit significand). */

void orc_dequant_mlx8(const uint32_t *q, const uint16_t *s, const uint16_t *b,
                      int rows, int cols, double *W)
{
    int wpr = cols / 4, gpr = cols / ORC_GROUP;
    for (int r = 0; r < rows; r++)
        for (int c = 0; c < cols; c++) {
            uint32_t word = q[(size_t)r * wpr + c / 4];
            unsigned byte = (word >> (8 * (c % 4))) & 255u;
            double scale = orc_f16_to_f64(s[(size_t)r * gpr + c / ORC_GROUP]);
            double bias = orc_f16_to_f64(b[(size_t)r * gpr + c / ORC_GROUP]);
            W[(size_t)r * cols + c] = scale * (double)byte + bias;
        }
}

/* The 4-bit quantiser's rule with 255 steps: b = fp16 rounded down of the
 * group min, s = fp16 rounded up of (max - b)/255, q = clamp(round_half_even(
 * (w - b)/s), 0, 255); so again |w - (s q + b)| <= s/2. */
void orc_quantize_mlx8(const double *W, int rows, int cols,
                       uint32_t *q, uint16_t *s, uint16_t *b)
{
    int wpr = cols / 4, gpr = cols / ORC_GROUP;
    memset(q, 0, sizeof(uint32_t) * (size_t)rows * wpr);
    for (int r = 0; r < rows; r++)
        for (int g = 0; g < gpr; g++) {
            const double *w = W + (size_t)r * cols + g * ORC_GROUP;
            double lo = w[0], hi = w[0];
            for (int c = 1; c < ORC_GROUP; c++) {
                if (w[c] < lo) lo = w[c];
                if (w[c] > hi) hi = w[c];
            }
            uint16_t bb = f16_round_dir(lo, 0);
            double bv = orc_f16_to_f64(bb);
            uint16_t ss = f16_round_dir((hi - bv) / 255.0, 1);
            double sv = orc_f16_to_f64(ss);
            s[(size_t)r * gpr + g] = ss;
            b[(size_t)r * gpr + g] = bb;
            for (int c = 0; c < ORC_GROUP; c++) {
                double t = sv > 0 ? nearbyint((w[c] - bv) / sv) : 0.0;
                if (t < 0) t = 0;
                if (t > 255) t = 255;
                int col = g * ORC_GROUP + c;
                q[(size_t)r * wpr + col / 4] |= (uint32_t)t << (8 * (col % 4));
            }
        }
}

/* The layer given the routing, for experts given as dense fp64 weights (any
 * width, already dequantised): the definition of orc_moe_combine, term for
 * term. G[e], U[e]: [I][H]; D[e]: [H][I]; NULL for experts that ids does not
 * name. Returns 0, or -1 if a needed expert is missing. */
int orc_moe_combine_dense(int T, int H, int k, int I, int Is,
                          const uint16_t *x, const int32_t *ids, const double *w,
                          const double *gate, const double *const *G, const double *const *U,
                          const double *const *D, int E, const double *Gs, const double *Us,
                          const double *Ds, double *out64, uint16_t *out_bf16)
{
    double *xt = malloc(sizeof(double) * H);
    double *y = malloc(sizeof(double) * H);
    double *hb = malloc(sizeof(double) * (I > Is ? I : Is));
    int rc = 0;
    for (int t = 0; t < T && rc == 0; t++) {
        for (int c = 0; c < H; c++)
            xt[c] = orc_bf16_to_f64(x[(size_t)t * H + c]);
        double *o = out64 + (size_t)t * H;
        for (int c = 0; c < H; c++)
            o[c] = 0.0;
        for (int j = 0; j < k; j++) {
            int e = ids[(size_t)t * k + j];
            if (e < 0 || e >= E || !G[e] || !U[e] || !D[e]) { rc = -1; break; }
            expert_mlp(G[e], U[e], D[e], H, I, xt, hb, y);
            for (int c = 0; c < H; c++)
                o[c] += w[(size_t)t * k + j] * y[c];
        }
        if (rc) break;
        expert_mlp(Gs, Us, Ds, H, Is, xt, hb, y);
        for (int c = 0; c < H; c++) {
            o[c] += y[c] * gate[t];
            if (out_bf16)
                out_bf16[(size_t)t * H + c] = orc_f64_to_bf16(o[c]);
        }
    }
    free(xt);
    free(y);
    free(hb);
    return rc;
}

/* The oracle's reader of the library's 8-bit blob: the atoms keep the 4-bit
 * atom's row and column order, but hold each value's low nibble in plane 0
 * (bytes [0,512), the 4-bit lane layout) and its high nibble in plane 1
 * (bytes [512,1024), the same layout), then the 64 bytes of fp16 (s, b) at
 * [1024,1088) in the 4-bit atom's order. Atom order as for 4 bits. */
#define ATOM8 1088

static unsigned blob8_value(const uint8_t *atom, int row, int col)
{
    return blob_nibble(atom, row, col) | (blob_nibble(atom + 512, row, col) << 4);
}

uint64_t orc_blob_bytes8(int H, int I)
{
    return (uint64_t)(I / 8) * (H / ORC_GROUP) * ATOM8 +
           (uint64_t)(H / 16) * (I / ORC_GROUP) * ATOM8;
}

/* Parse one 8-bit blob into 8-bit MLX triples (q words of 4 values). */
void orc_blob_to_mlx8(const uint8_t *blob, int H, int I,
                      uint32_t *gq, uint16_t *gs, uint16_t *gb,
                      uint32_t *uq, uint16_t *us, uint16_t *ub,
                      uint32_t *dq, uint16_t *ds, uint16_t *db)
{
    int kbH = H / ORC_GROUP, kbI = I / ORC_GROUP;
    memset(gq, 0, sizeof(uint32_t) * (size_t)I * (H / 4));
    memset(uq, 0, sizeof(uint32_t) * (size_t)I * (H / 4));
    memset(dq, 0, sizeof(uint32_t) * (size_t)H * (I / 4));
    for (int i = 0; i < I; i++)
        for (int kb = 0; kb < kbH; kb++) {
            const uint8_t *atom = blob + ((size_t)(i / 8) * kbH + kb) * ATOM8;
            for (int which = 0; which < 2; which++) {
                int row = (i % 8) + 8 * which;       /* gate: g, up: g+8 */
                uint32_t *q = which ? uq : gq;
                uint16_t *s = which ? us : gs, *b = which ? ub : gb;
                for (int c = 0; c < ORC_GROUP; c++) {
                    int col = kb * ORC_GROUP + c;
                    q[(size_t)i * (H / 4) + col / 4] |=
                        (uint32_t)blob8_value(atom, row, c) << (8 * (col % 4));
                }
                blob_sb(atom + 512, row, &s[(size_t)i * kbH + kb], &b[(size_t)i * kbH + kb]);
            }
        }
    const uint8_t *down = blob + (size_t)(I / 8) * kbH * ATOM8;
    for (int o = 0; o < H; o++)
        for (int kb = 0; kb < kbI; kb++) {
            const uint8_t *atom = down + ((size_t)(o / 16) * kbI + kb) * ATOM8;
            int row = o % 16;
            for (int c = 0; c < ORC_GROUP; c++) {
                int col = kb * ORC_GROUP + c;
                dq[(size_t)o * (I / 4) + col / 4] |=
                    (uint32_t)blob8_value(atom, row, c) << (8 * (col % 4));
            }
            blob_sb(atom + 512, row, &ds[(size_t)o * kbI + kb], &db[(size_t)o * kbI + kb]);
        }
}
