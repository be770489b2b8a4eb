/*
 * CPU oracle for single-query paged attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Like attn_oracle.c, this is the slow, obviously
 * correct reference the CUDA path is checked against; only the test suite,
 * the smoke check and the benchmark's CPU legs load it, and it shares no
 * code with the product.
 *
 * What it computes follows atrex-bench "paged_attention_decode" (page #024,
 * reference.py, Model.forward).  Sequence i has one query row per query head
 * and ctx_len = seq_lens[i] context tokens.  Token t (0 <= t < ctx_len) lives
 * in physical block b = block_tables[i][t / block_size] at position
 * p = t % block_size, where
 *
 *     key[d]   = k_cache[b][g][d / x][p][d % x]     (x = 8 elements = 16 bytes)
 *     value[d] = v_cache[b][g][d][p]
 *
 * for KV head g.  Query head h reads KV head g = h / (Hq / Hkv) (the page
 * repeats every KV head Hq / Hkv times, consecutively).  With
 * scale = head_size^-1/2, per (i, h):
 *
 *     s_t = (sum_d q[i,h,d] * key_t[d]) * scale,  m = max_t s_t,
 *     w_t = exp(s_t - m),  o[i,h,:] = sum_t w_t value_t[:] / sum_t w_t.
 *
 * A sequence with ctx_len <= 0 gets zero rows (the page starts from zeros
 * and skips it).  Inputs are bf16 or IEEE half bit patterns widened exactly
 * to double; the arithmetic is IEEE double with libm exp.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif
#define PMUT(n) (ORACLE_MUTATION == (n))

static double bf16_bits(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_bits(uint16_t b) {
    const int sign = (b >> 15) & 1;
    const int e = (b >> 10) & 0x1f;
    const int f = b & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* zero and subnormals: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -v : v;
}

static double elem(uint16_t b, int is_fp16) {
    return (is_fp16 && !PMUT(23)) ? f16_bits(b) : bf16_bits(b);
}

/*
 * out [num_seqs, Hq, D] doubles.  Returns 0, -1 on a bad argument, -2 when
 * out of memory.
 */
int oracle_paged_decode(const uint16_t* query, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                        int Hq, int Hkv, int D, int block_size, int max_blocks, int is_fp16,
                        double* out) {
    const int x = 8;
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || D % x || block_size <= 0)
        return -1;
    const int qpk = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)D);
    for (int i = 0; i < num_seqs; ++i) {
        const int64_t L = seq_lens[i];
        for (int h = 0; h < Hq; ++h) {
            double* o = out + ((int64_t)i * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (L <= 0) continue;
            const int g = PMUT(20) ? h % Hkv : h / qpk;
            const uint16_t* q = query + ((int64_t)i * Hq + h) * D;
            double* s = (double*)malloc(sizeof(double) * (size_t)L);
            if (!s) return -2;
            for (int64_t t = 0; t < L; ++t) {
                int64_t b = block_tables[(int64_t)i * max_blocks + t / block_size];
                int64_t p = t % block_size;
                if (PMUT(21)) {          /* planted: flat index without the table */
                    b = t / block_size;
                }
                double acc = 0.0;
                for (int d = 0; d < D; ++d) {
                    int64_t kidx;
                    if (PMUT(22))        /* planted: keys read in the value layout */
                        kidx = (((b * Hkv + g) * D + d) * block_size) + p;
                    else
                        kidx = ((((b * Hkv + g) * (D / x) + d / x) * block_size + p) * x) + d % x;
                    acc += elem(q[d], is_fp16) * elem(k_cache[kidx], is_fp16);
                }
                s[t] = acc * scale;
            }
            double m = s[0];
            for (int64_t t = 1; t < L; ++t) if (s[t] > m) m = s[t];
            double denom = 0.0;
            for (int64_t t = 0; t < L; ++t) {
                s[t] = exp(s[t] - m);
                denom += s[t];
            }
            for (int64_t t = 0; t < L; ++t) {
                const int64_t b = PMUT(21) ? t / block_size
                                           : block_tables[(int64_t)i * max_blocks + t / block_size];
                const int64_t p = t % block_size;
                const uint16_t* vb = v_cache + ((b * Hkv + g) * D) * block_size + p;
                for (int d = 0; d < D; ++d) o[d] += s[t] * elem(vb[(int64_t)d * block_size], is_fp16);
            }
            for (int d = 0; d < D; ++d) o[d] /= denom;
            free(s);
        }
    }
    return 0;
}
