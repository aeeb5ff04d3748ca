/*
 * gdn_oracle.c -- CPU oracle of one Gated DeltaNet recurrence step
 * (fp64, single-threaded, plain loops). TEST INFRASTRUCTURE: only tests/,
 * the smoke check and the benchmark's CPU baseline use it; the CUDA library
 * shares no code with it.
 *
 * The pages say that three quarters of the hybrid model's layers are Gated
 * DeltaNet linear attention with a fixed-size recurrent state, so no KV
 * cache grows with the context (xix.ai article, paragraph on the forward
 * pass; agentlenshq article, section on how expert streaming works). They do
 * not spell out the recurrence. The reading taken is the gated delta rule as
 * published for Gated DeltaNet (Yang, Kautz and Hatamizadeh, "Gated Delta
 * Networks: Improving Mamba2 with Delta Rule", ICLR 2025), with the L2
 * normalisation of queries and keys used there. Per sequence and value
 * head, with state S (d_v rows x d_k columns) and one token:
 *
 *   k^ = k / sqrt(sum k^2 + 1e-6),  q^ = scale * q / sqrt(sum q^2 + 1e-6)
 *   alpha = exp(g)                  (g <= 0: the gate's log decay)
 *   u  = S k^                       (what the state holds for k^)
 *   S' = alpha S + beta (v - alpha u) k^T
 *   o  = S' q^
 *
 * which equals S' = alpha S (I - beta k^ k^T) + beta v k^T. A query/key
 * head serves n_v / n_k consecutive value heads (grouped value heads).
 *
 * Tokens t = 0 .. T-1 run one after the other on the same state.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

double orc_bf16_to_f64(uint16_t h);

/* Unit-norm copy of a bf16 vector of n values (times `mul`), in fp64. */
static void normalise(const uint16_t *src, int n, double mul, double *dst)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++) {
        double a = orc_bf16_to_f64(src[i]);
        ss += a * a;
    }
    double inv = mul / sqrt(ss + 1e-6);
    for (int i = 0; i < n; i++)
        dst[i] = orc_bf16_to_f64(src[i]) * inv;
}

/*
 * q, k: bf16 [T][B][n_k][d_k]; v: bf16 [T][B][n_v][d_v];
 * g, beta: fp64 [T][B][n_v]; state: fp64 [B][n_v][d_v][d_k], updated in place;
 * out: fp64 [T][B][n_v][d_v]. Returns 0, or -1 for a bad shape.
 */
int orc_gdn_step(int T, int B, int nk, int nv, int dk, int dv, const uint16_t *q, const uint16_t *k,
                 const uint16_t *v, const double *g, const double *beta, double scale, double *state,
                 double *out)
{
    if (T < 0 || B < 0 || nk <= 0 || nv <= 0 || nv % nk || dk <= 0 || dv <= 0 || dk > 1024)
        return -1;
    double kn[1024], qn[1024];
    for (int t = 0; t < T; t++)
        for (int b = 0; b < B; b++)
            for (int h = 0; h < nv; h++) {
                int hk = h / (nv / nk);
                size_t kq = (((size_t)t * B + b) * nk + hk) * dk;
                normalise(k + kq, dk, 1.0, kn);
                normalise(q + kq, dk, scale, qn);
                size_t gi = ((size_t)t * B + b) * nv + h;
                double alpha = exp(g[gi]), bt = beta[gi];
                double *S = state + ((size_t)b * nv + h) * dv * dk;
                const uint16_t *vv = v + gi * dv;
                double *o = out + gi * dv;
                for (int i = 0; i < dv; i++) {
                    double *row = S + (size_t)i * dk;
                    double u = 0.0;
                    for (int j = 0; j < dk; j++)
                        u += row[j] * kn[j];
                    double c = bt * (orc_bf16_to_f64(vv[i]) - alpha * u);
                    double oi = 0.0;
                    for (int j = 0; j < dk; j++) {
                        row[j] = alpha * row[j] + c * kn[j];
                        oi += row[j] * qn[j];
                    }
                    o[i] = oi;
                }
            }
    return 0;
}
