/*
 * CPU oracle for packed variable-length, non-causal attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * reference that the CUDA path is checked against.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never calls it and shares no code with it.
 *
 * What it computes follows atrex-bench "attention_forward" (page #001,
 * reference.py, Model.forward): for every sequence i whose query slice
 * [cu_seqlens_q[i], cu_seqlens_q[i+1]) is non-empty, and for every head h,
 * the output rows of that slice are
 *
 *     softmax(Q_i,h . K_i,h^T * scale) . V_i,h ,   scale = head_dim^-1/2
 *
 * where K_i and V_i are the rows [cu_seqlens_k[i], cu_seqlens_k[i+1]).  The
 * page calls scaled_dot_product_attention with is_causal=False and no scale
 * argument, so the scale is the library default 1/sqrt(head_dim), with the
 * true head_dim.  Written out per output row r of head h:
 *
 *     s_j = (sum_d q[r,h,d] * k[j,h,d]) * scale          for each key j
 *     m   = max_j s_j
 *     w_j = exp(s_j - m)
 *     o[r,h,:] = (sum_j w_j * v[j,h,:]) / (sum_j w_j)
 *
 * Inputs are bf16 bit patterns widened exactly to double; all arithmetic is
 * IEEE double with libm exp.  There is no tiling, no exp2 and no online
 * rescaling: the max is found first, then the weights, then the weighted sum.
 *
 * Causal variant (not on the page, which is non-causal; offered as the
 * common prefill neighbour): query row r of a sequence (0-based within its
 * slice) sees only keys j <= r + (L_k - L_q), i.e. the mask is aligned to the
 * bottom-right corner, so that the last query row sees every key (the
 * convention of prefill after a cached prefix; for L_q = L_k it is the usual
 * lower triangle).  A row that sees no key gets a zero row, like an empty key
 * slice.
 *
 * Readings where the page is silent:
 *  - a sequence with an empty (or negative) query slice is skipped, and its
 *    output rows are not written (the page's loop skips it);
 *  - a non-empty query slice with an empty (or negative) key slice gets zero
 *    output rows (the weighted sum over an empty key set);
 *  - rows outside every query slice are not written.
 *
 * Layout: q, out [total_q, H, D]; k, v [total_k, H, D], row-major, token-major.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Keys visible to row r (0-based in its query slice) of a sequence with Lq
 * queries and Lk keys: all Lk, or with the causal mask min(Lk, r + 1 + Lk - Lq). */
static int64_t visible_keys(int64_t r, int64_t Lq, int64_t Lk, int causal);

/* Plant-a-mistake hook for the oracle's own pin tests: the tests build a
 * separate copy of this file with -DORACLE_MUTATION=n and check that the pins
 * catch each mistake.  The normal build defines nothing and every MUT(n) is 0. */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif
#define MUT(n) (ORACLE_MUTATION == (n))

static int64_t visible_keys(int64_t r, int64_t Lq, int64_t Lk, int causal) {
    if (!causal) return Lk;
    int64_t lim;
    if (MUT(11)) lim = r + Lk - Lq;          /* planted: the diagonal key dropped */
    else if (MUT(12)) lim = r + 1;           /* planted: top-left alignment */
    else lim = r + 1 + Lk - Lq;
    if (lim > Lk) lim = Lk;
    return lim > 0 ? lim : 0;
}

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One output row: query token t (global row), head h, keys [k0, k0+Lk). */
static void attend_row(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       int64_t t, int64_t k0, int64_t Lk, int H, int D, int h,
                       double* o, double* s /* scratch, >= Lk */) {
    const double scale = MUT(1) ? 1.0 / (double)D : 1.0 / sqrt((double)D);
    const int64_t row = (int64_t)H * D;
    int64_t keys = MUT(6) ? Lk - 1 : Lk;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (keys <= 0) {
        if (MUT(10)) for (int d = 0; d < D; ++d) o[d] = NAN;
        return;
    }
    const uint16_t* qr = q + t * row + (int64_t)h * D;
    for (int64_t j = 0; j < keys; ++j) {
        const uint16_t* kr = MUT(5) ? k + (k0 + j) * row + h
                                    : k + (k0 + j) * row + (int64_t)h * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) {
            double kd = MUT(5) ? bf16_to_double(kr[(int64_t)d * H])
                               : bf16_to_double(kr[d]);
            acc += bf16_to_double(qr[d]) * kd;
        }
        s[j] = acc * scale;
    }
    double m = s[0];
    for (int64_t j = 1; j < keys; ++j) if (s[j] > m) m = s[j];
    double denom = 0.0;
    for (int64_t j = 0; j < keys; ++j) {
        double w = MUT(9) ? exp(m - s[j]) : exp(s[j] - m);
        s[j] = w;
        denom += w;
    }
    for (int64_t j = 0; j < keys; ++j) {
        int64_t vj = MUT(7) ? t : k0 + j;
        const uint16_t* vr = v + vj * row + (int64_t)h * D;
        for (int d = 0; d < D; ++d) o[d] += s[j] * bf16_to_double(vr[d]);
    }
    if (!MUT(3))
        for (int d = 0; d < D; ++d) o[d] /= denom;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads an OpenMP parallel region would use (1 without OpenMP). */
int oracle_max_threads(int nthreads) {
#ifdef _OPENMP
    set_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Every output row of every non-empty sequence.  out has [total_q, H, D]
 * doubles; rows outside the query slices are left as the caller set them.
 * Returns 0, or -1 on a bad argument, -2 when out of memory.
 */
int oracle_attn_varlen(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const int32_t* cu_q, const int32_t* cu_k, int num_seqs,
                       int H, int D, int causal, double* out, int nthreads) {
    if (num_seqs < 0 || H <= 0 || D <= 0) return -1;
    set_threads(nthreads);
    int err = 0;
    for (int i = 0; i < num_seqs; ++i) {
        int64_t q0 = cu_q[i], Lq = (int64_t)cu_q[i + 1] - cu_q[i];
        int64_t k0 = MUT(4) ? cu_q[i] : cu_k[i];
        int64_t Lk = (int64_t)cu_k[i + 1] - cu_k[i];
        if (MUT(13)) {  /* planted: a backwards slice read as the reversed range */
            if (Lq < 0) { q0 = cu_q[i + 1]; Lq = -Lq; }
            if (Lk < 0) { k0 = cu_k[i + 1]; Lk = -Lk; }
        }
        if (Lq <= 0) continue;
        if (Lk < 0) Lk = 0;
        int64_t n = Lq * H;
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
            if (!s) {
#pragma omp atomic write
                err = -2;
            } else {
#pragma omp for schedule(dynamic, 16)
                for (int64_t idx = 0; idx < n; ++idx) {
                    int64_t t = q0 + idx / H;
                    int h = (int)(idx % H);
                    attend_row(q, k, v, t, k0, visible_keys(t - q0, Lq, Lk, causal), H, D, h,
                               out + t * (int64_t)H * D + (int64_t)h * D, s);
                }
                free(s);
            }
        }
        if (err) return err;
    }
    return 0;
}

/*
 * Selected output rows only: rows[2*n] = (token, head) pairs, out [n, D].
 * A token outside every non-empty query slice returns -3.
 */
int oracle_attn_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const int32_t* cu_q, const int32_t* cu_k, int num_seqs,
                     int H, int D, int causal, const int64_t* rows, int64_t n_rows,
                     double* out, int nthreads) {
    if (num_seqs < 0 || H <= 0 || D <= 0 || n_rows < 0) return -1;
    set_threads(nthreads);
    int64_t max_lk = 1;
    for (int i = 0; i < num_seqs; ++i) {
        int64_t Lk = (int64_t)cu_k[i + 1] - cu_k[i];
        if (Lk > max_lk) max_lk = Lk;
    }
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)max_lk);
        if (!s) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n_rows; ++r) {
                int64_t t = rows[2 * r];
                int h = (int)rows[2 * r + 1];
                int found = -1;
                for (int i = 0; i < num_seqs; ++i)
                    if (cu_q[i + 1] > cu_q[i] && t >= cu_q[i] && t < cu_q[i + 1]) {
                        found = i;
                        break;
                    }
                if (found < 0 || h < 0 || h >= H) {
#pragma omp atomic write
                    err = -3;
                    continue;
                }
                int64_t k0 = MUT(4) ? cu_q[found] : cu_k[found];
                int64_t Lk = (int64_t)cu_k[found + 1] - cu_k[found];
                if (Lk < 0) Lk = 0;
                const int64_t Lq = (int64_t)cu_q[found + 1] - cu_q[found];
                attend_row(q, k, v, t, k0, visible_keys(t - cu_q[found], Lq, Lk, causal), H, D,
                           h, out + r * (int64_t)D, s);
            }
            free(s);
        }
    }
    return err;
}
