/*
 * CPU oracle for the head-sharded local attention step of Ulysses sequence
 * parallelism. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it; the library never does.
 *
 * What it computes is plain softmax attention, per head, in float64, with an
 * explicit per-pair mask predicate and no blocking, tiling or reordering:
 *
 *   s_ij   = scale * sum_d q_id k_jd                 (scale = 1/sqrt(D) by default)
 *   allowed(i,j) = seg(i) == seg(j)  and (not causal or j <= i)
 *   lse_i  = m_i + log sum_{allowed j} exp(s_ij - m_i),   m_i = max_{allowed j} s_ij
 *   P_ij   = exp(s_ij - lse_i)
 *   O_i    = sum_j P_ij v_j
 *
 * and its gradient for L = sum O * dO:
 *
 *   dP_ij  = dO_i . v_j
 *   Delta_i = sum_j P_ij dP_ij          (taken from this definition, not as dO.O)
 *   dS_ij  = P_ij (dP_ij - Delta_i)
 *   dQ_i   = scale sum_j dS_ij k_j
 *   dK_j   = scale sum_{h in group} sum_i dS^h_ij q^h_i
 *   dV_j   = sum_{h in group} sum_i P^h_ij dO^h_i
 *
 * Sources: the pages on Ulysses sequence parallelism state that attention
 * heads are independent and that each rank computes ordinary attention over
 * the full sequence for its own heads (congresoia365 article, "Cómo Funciona
 * Ulysses", steps 4 and the closing remark on independent heads); that with
 * FlashAttention the result is exact attention with O(n) memory (same article,
 * "El Desafío del Entrenamiento de Secuencias Largas"); and that packed samples
 * must not attend across their boundaries (HF Transformers "Ulysses sequence
 * parallelism" guide, "Configurar", sp_attn_implementation). Causality within a
 * sample follows the causal-LM models the pages train. The gradient formulas
 * are the textbook derivative of softmax attention.
 *
 * Query head h reads key/value head h / (hq/hkv) (contiguous GQA groups).
 * Inputs are 16-bit patterns (uint16) of bf16, or of IEEE binary16 (fp16) when the
 * call's in_f16 flag is set, converted exactly to double.
 * Layout of every activation: [heads][T][D], row-major.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: sign, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1, ex = (h >> 10) & 0x1f, man = h & 0x3ff;
    double v;
    if (ex == 0) v = ldexp((double)man, -24);                 /* zero and subnormals: man * 2^-24 */
    else if (ex == 31) v = man ? NAN : INFINITY;
    else v = ldexp((double)(man | 0x400), ex - 25);           /* 1.man * 2^(ex - 15) */
    return sign ? -v : v;
}

/* Element type of the current call's inputs (set before any parallel region). */
static int g_in_f16 = 0;

static double elem_to_double(uint16_t b) { return g_in_f16 ? f16_to_double(b) : bf16_to_double(b); }

/* The decoder on its own, so that it can be checked against other implementations. */
void oracle_decode16(const uint16_t* in, int64_t n, int f16, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f16 ? f16_to_double(in[i]) : bf16_to_double(in[i]);
}

/* seg[t] = b such that cu[b] <= t < cu[b+1]; returns 0 on success. */
static int build_segments(const int32_t* cu, int nseq, int64_t T, int32_t* seg) {
    if (cu[0] != 0 || (int64_t)cu[nseq] != T) return -1;
    for (int b = 0; b < nseq; ++b) {
        if (cu[b + 1] < cu[b]) return -1;
        for (int64_t t = cu[b]; t < cu[b + 1]; ++t) seg[t] = b;
    }
    return 0;
}

static int allowed(const int32_t* seg, int64_t i, int64_t j, int causal) {
    if (seg[i] != seg[j]) return 0;
    if (causal && j > i) return 0;
    return 1;
}

static double dot_bf16(const uint16_t* a, const uint16_t* b, int D) {
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += elem_to_double(a[d]) * elem_to_double(b[d]);
    return s;
}

/* Scores of row i against every key j (s[j] = scale * q_i.k_j), only for allowed j;
 * returns lse_i.  s must hold T doubles; entries of masked j are left untouched. */
static double row_scores_lse(const uint16_t* qi, const uint16_t* kh, const int32_t* seg,
                             int64_t i, int64_t T, int D, double scale, int causal, double* s) {
    double m = -INFINITY;
    for (int64_t j = 0; j < T; ++j) {
        if (!allowed(seg, i, j, causal)) continue;
        s[j] = scale * dot_bf16(qi, kh + j * D, D);
        if (s[j] > m) m = s[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < T; ++j) {
        if (!allowed(seg, i, j, causal)) continue;
        sum += exp(s[j] - m);
    }
    return m + log(sum);
}

/*
 * Forward.  Computes O and LSE for the listed query heads and rows.
 *   q [hq][T][D], k/v [hkv][T][D]           16-bit patterns (bf16, or fp16 with in_f16)
 *   heads[nheads] (NULL: all hq heads), rows[nrows] (NULL: all T rows)
 *   o   [nheads][nrows][D] double, lse [nheads][nrows] double (either may be NULL)
 * Returns 0, or -1 when cu_seqlens is malformed or an argument is invalid.
 */
int oracle_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* cu, int nseq, int64_t T, int hq, int hkv, int D,
                    double scale, int causal,
                    const int32_t* heads, int nheads, const int64_t* rows, int64_t nrows,
                    double* o, double* lse, int in_f16) {
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || D <= 0 || T < 0 || nseq < 0) return -1;
    g_in_f16 = in_f16 ? 1 : 0;
    int32_t* seg = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!seg) return -1;
    if (build_segments(cu, nseq, T, seg) != 0) { free(seg); return -1; }
    if (!heads) nheads = hq;
    if (!rows) nrows = T;
    const int G = hq / hkv;
    int rc = 0;
    for (int hi = 0; hi < nheads; ++hi) {
        const int h = heads ? heads[hi] : hi;
        if (h < 0 || h >= hq) { rc = -1; break; }
        const uint16_t* qh = q + (int64_t)h * T * D;
        const uint16_t* kh = k + (int64_t)(h / G) * T * D;
        const uint16_t* vh = v + (int64_t)(h / G) * T * D;
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
            double* acc = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 8)
            for (int64_t ri = 0; ri < nrows; ++ri) {
                const int64_t i = rows ? rows[ri] : ri;
                const double l = row_scores_lse(qh + i * D, kh, seg, i, T, D, scale, causal, s);
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (int64_t j = 0; j < T; ++j) {
                    if (!allowed(seg, i, j, causal)) continue;
                    const double p = exp(s[j] - l);
                    for (int d = 0; d < D; ++d) acc[d] += p * elem_to_double(vh[j * D + d]);
                }
                if (o) for (int d = 0; d < D; ++d) o[((int64_t)hi * nrows + ri) * D + d] = acc[d];
                if (lse) lse[(int64_t)hi * nrows + ri] = l;
            }
            free(s);
            free(acc);
        }
    }
    free(seg);
    return rc;
}

/*
 * Backward.
 *   q_heads[nqh] (NULL: all hq) and q_rows[nqr] (NULL: all T): rows of dQ to produce
 *   kv_heads[nkvh] (NULL: all hkv) and k_rows[nkr] (NULL: all T): rows of dK/dV to produce;
 *     each kv head sums the contributions of all hq/hkv query heads of its group.
 *   dq [nqh][nqr][D], dk/dv [nkvh][nkr][D]   double (may be NULL)
 *   lse_out / delta_out [nqh][nqr]             double (may be NULL): lse_i and Delta_i of the dQ rows
 */
int oracle_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                    const int32_t* cu, int nseq, int64_t T, int hq, int hkv, int D,
                    double scale, int causal,
                    const int32_t* q_heads, int nqh, const int64_t* q_rows, int64_t nqr,
                    const int32_t* kv_heads, int nkvh, const int64_t* k_rows, int64_t nkr,
                    double* dq, double* dk, double* dv, double* lse_out, double* delta_out, int in_f16) {
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || D <= 0 || T < 0 || nseq < 0) return -1;
    g_in_f16 = in_f16 ? 1 : 0;
    int32_t* seg = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!seg) return -1;
    if (build_segments(cu, nseq, T, seg) != 0) { free(seg); return -1; }
    if (!q_heads) nqh = hq;
    if (!q_rows) nqr = T;
    if (!kv_heads) nkvh = hkv;
    if (!k_rows) nkr = T;
    const int G = hq / hkv;
    const int64_t TT = T > 0 ? T : 1;
    int rc = 0;

    /* Per query head h and row i: lse_i and Delta_i, computed for every row that
     * some requested output depends on. */
    double* lse_all = (double*)malloc(sizeof(double) * (size_t)TT);
    double* del_all = (double*)malloc(sizeof(double) * (size_t)TT);
    unsigned char* need = (unsigned char*)malloc((size_t)TT);
    if (!lse_all || !del_all || !need) rc = -1;

    for (int pass = 0; pass < 2 && rc == 0; ++pass) {
        /* pass 0: dQ for the requested query heads; pass 1: dK/dV for the requested kv heads */
        const int nh = pass == 0 ? nqh : nkvh * G;
        for (int hi = 0; hi < nh && rc == 0; ++hi) {
            int h;
            if (pass == 0) h = q_heads ? q_heads[hi] : hi;
            else h = (kv_heads ? kv_heads[hi / G] : hi / G) * G + hi % G;
            if (h < 0 || h >= hq) { rc = -1; break; }
            const uint16_t* qh = q + (int64_t)h * T * D;
            const uint16_t* kh = k + (int64_t)(h / G) * T * D;
            const uint16_t* vh = v + (int64_t)(h / G) * T * D;
            const uint16_t* doh = dout + (int64_t)h * T * D;

            /* which rows are needed */
            for (int64_t i = 0; i < T; ++i) need[i] = 0;
            if (pass == 0) {
                for (int64_t r = 0; r < nqr; ++r) need[q_rows ? q_rows[r] : r] = 1;
            } else {
#pragma omp parallel for schedule(dynamic, 64)
                for (int64_t i = 0; i < T; ++i) {
                    for (int64_t r = 0; r < nkr && !need[i]; ++r)
                        if (allowed(seg, i, k_rows ? k_rows[r] : r, causal)) need[i] = 1;
                }
            }

#pragma omp parallel
            {
                double* s = (double*)malloc(sizeof(double) * (size_t)TT);
#pragma omp for schedule(dynamic, 8)
                for (int64_t i = 0; i < T; ++i) {
                    if (!need[i]) continue;
                    const double l = row_scores_lse(qh + i * D, kh, seg, i, T, D, scale, causal, s);
                    double delta = 0.0;
                    for (int64_t j = 0; j < T; ++j) {
                        if (!allowed(seg, i, j, causal)) continue;
                        const double p = exp(s[j] - l);
                        const double dp = dot_bf16(doh + i * D, vh + j * D, D);
                        delta += p * dp;
                    }
                    lse_all[i] = l;
                    del_all[i] = delta;
                }
                free(s);
            }

            if (pass == 0) {
#pragma omp parallel
                {
                    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 8)
                    for (int64_t ri = 0; ri < nqr; ++ri) {
                        const int64_t i = q_rows ? q_rows[ri] : ri;
                        for (int d = 0; d < D; ++d) acc[d] = 0.0;
                        for (int64_t j = 0; j < T; ++j) {
                            if (!allowed(seg, i, j, causal)) continue;
                            const double sij = scale * dot_bf16(qh + i * D, kh + j * D, D);
                            const double p = exp(sij - lse_all[i]);
                            const double dp = dot_bf16(doh + i * D, vh + j * D, D);
                            const double ds = p * (dp - del_all[i]);
                            for (int d = 0; d < D; ++d) acc[d] += ds * elem_to_double(kh[j * D + d]);
                        }
                        if (dq) for (int d = 0; d < D; ++d) dq[((int64_t)hi * nqr + ri) * D + d] = scale * acc[d];
                        if (lse_out) lse_out[(int64_t)hi * nqr + ri] = lse_all[i];
                        if (delta_out) delta_out[(int64_t)hi * nqr + ri] = del_all[i];
                    }
                    free(acc);
                }
            } else {
                const int ki = hi / G;  /* index into the kv-head list */
#pragma omp parallel
                {
                    double* ak = (double*)malloc(sizeof(double) * (size_t)D);
                    double* av = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 8)
                    for (int64_t rj = 0; rj < nkr; ++rj) {
                        const int64_t j = k_rows ? k_rows[rj] : rj;
                        for (int d = 0; d < D; ++d) { ak[d] = 0.0; av[d] = 0.0; }
                        for (int64_t i = 0; i < T; ++i) {
                            if (!allowed(seg, i, j, causal)) continue;
                            const double sij = scale * dot_bf16(qh + i * D, kh + j * D, D);
                            const double p = exp(sij - lse_all[i]);
                            const double dp = dot_bf16(doh + i * D, vh + j * D, D);
                            const double ds = p * (dp - del_all[i]);
                            for (int d = 0; d < D; ++d) {
                                ak[d] += ds * elem_to_double(qh[i * D + d]);
                                av[d] += p * elem_to_double(doh[i * D + d]);
                            }
                        }
                        /* the first query head of a group initialises, the others add */
                        for (int d = 0; d < D; ++d) {
                            const int64_t idx = ((int64_t)ki * nkr + rj) * D + d;
                            if (dk) dk[idx] = (hi % G == 0 ? 0.0 : dk[idx]) + scale * ak[d];
                            if (dv) dv[idx] = (hi % G == 0 ? 0.0 : dv[idx]) + av[d];
                        }
                    }
                    free(ak);
                    free(av);
                }
            }
        }
    }
    free(lse_all);
    free(del_all);
    free(need);
    free(seg);
    return rc;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
