/*
 * CPU oracle for the chunked gated delta-rule output.
 *
 * TEST INFRASTRUCTURE ONLY.  Like attn_oracle.c, this is the slow, obviously
 * correct reference the CUDA path is checked against; only the test suite,
 * the smoke check and the benchmark's CPU legs load it, and it shares no
 * code with the product.
 *
 * What it computes follows atrex-bench "chunk_delta_rule_output" (page #004,
 * reference.py, Model.forward).  Tokens are cut into chunks of cs (64); the
 * token count is padded to whole chunks with zero q, k, v and g, and padded
 * rows are dropped from the output.  Value head hd reads query/key head
 * qh = min(hd / max(H / Hq, 1), Hq - 1).  For chunk c of batch b and value
 * head hd, with r, j the rows of the chunk (t = c * cs + r):
 *
 *   o_state[r,:] = exp(g[r]) * sum_k q[r,k] h[c][k,:]
 *   a[r,j]       = (q[r] . k[j]) * exp(g[r] - g[j])   if j <= r and g[r] <= g[j]
 *                = 0                                   otherwise
 *   out[r,:]     = scale * (o_state[r,:] + sum_j bf16(a[r,j]) * v[j,:])
 *
 * where bf16() rounds to bfloat16 (nearest even) as the page does before the
 * value product, and scale = key_dim^-1/2 unless given.  q, k, v, h are bf16
 * bit patterns, g is float32; everything else is IEEE double.
 *
 * Layouts: q, k [B, T, Hq, K]; v [B, T, H, V]; h [B, NC, H, K, V] with
 * NC = ceil(T / cs); g [B, T, H]; out [B, T, H, V] doubles.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif
#define CMUT(n) (ORACLE_MUTATION == (n))

static double bf16v(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> nearest bfloat16 value (ties to even), returned as a double.
 * A bfloat16 keeps 8 significant bits: round the significand of x to 8 bits. */
static double round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    const double m = frexp(x, &e);          /* x = m * 2^e, 0.5 <= |m| < 1 */
    const double s = ldexp(m, 8);            /* 8 significant bits before the point */
    double r = nearbyint(s);                 /* default rounding: to nearest, ties to even */
    return ldexp(r, e - 8);
}

int oracle_chunk_o(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* h,
                   const float* g, int B, int T, int Hq, int H, int K, int V, int cs,
                   double scale, double* out) {
    if (B < 0 || T < 0 || Hq <= 0 || H <= 0 || K <= 0 || V <= 0 || cs <= 0) return -1;
    const int NC = (T + cs - 1) / cs;
    int hpq = H / Hq;
    if (hpq < 1) hpq = 1;
    if (!(scale > 0.0)) scale = 1.0 / sqrt((double)K);
    if (CMUT(30)) scale = 1.0;
    for (int b = 0; b < B; ++b)
        for (int hd = 0; hd < H; ++hd) {
            int qh = hd / hpq;
            if (qh > Hq - 1) qh = Hq - 1;
            if (CMUT(34)) qh = hd % Hq;
            for (int t = 0; t < T; ++t) {
                const int c = t / cs, r = t % cs;
                const uint16_t* qr = q + (((int64_t)b * T + t) * Hq + qh) * K;
                const double gr = g[((int64_t)b * T + t) * H + hd];
                double* o = out + (((int64_t)b * T + t) * H + hd) * V;
                const uint16_t* hc = h + ((((int64_t)b * NC + c) * H + hd) * K) * V;
                /* state part */
                for (int x = 0; x < V; ++x) {
                    double acc = 0.0;
                    for (int kk = 0; kk < K; ++kk) acc += bf16v(qr[kk]) * bf16v(hc[(int64_t)kk * V + x]);
                    o[x] = acc * exp(gr);
                }
                /* intra-chunk part: keys j of the same chunk, j <= r (padded keys are zero) */
                const int jmax = CMUT(33) ? cs - 1 : r;
                for (int j = 0; j <= jmax; ++j) {
                    const int tj = c * cs + j;
                    if (tj >= T) break;
                    const double gj = g[((int64_t)b * T + tj) * H + hd];
                    const double gd = gr - gj;
                    const int keep = CMUT(32) ? gd >= 0.0 : gd <= 0.0;
                    if (!keep) continue;
                    const uint16_t* kr = k + (((int64_t)b * T + tj) * Hq + qh) * K;
                    double dot = 0.0;
                    for (int kk = 0; kk < K; ++kk) dot += bf16v(qr[kk]) * bf16v(kr[kk]);
                    double a = dot * exp(gd);
                    if (!CMUT(31)) a = round_bf16(a);
                    const uint16_t* vr = v + (((int64_t)b * T + tj) * H + hd) * V;
                    for (int x = 0; x < V; ++x) o[x] += a * bf16v(vr[x]);
                }
                for (int x = 0; x < V; ++x) o[x] *= scale;
            }
        }
    return 0;
}
