/*
 * fp64 CPU oracle for exact scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the CPU-baseline leg of
 * the benchmark are the only callers.  The CUDA library shares no code, header, table or
 * helper with this file, and this file includes nothing from it.
 *
 * What it computes is the plain three-step materialising definition of attention:
 *
 *   S = scale * Q K^T          ("How FlashAttention Reduces HBM Traffic Exactly", section
 *                               "The performance problem is data movement", equations for
 *                               S, P, O; "FlashAttention and GPU Data Movement", section 1)
 *   P = softmax(S) per row,    with the row maximum subtracted ("FlashAttention and GPU Data
 *                               Movement", section 3, the three lines defining m, l and P)
 *   O = P V
 *   L = m + ln l per row       ("FlashAttention Explained", section "Why the statistics are
 *                               cheap to store")
 *
 * evaluated one query row at a time: the row of S is materialised, then the row of P, then
 * the row of O.  Nothing is blocked, fused or reordered beyond that.
 *
 * Readings where the pages are silent:
 *  - the scale is applied to the exact fp64 dot product (never pre-multiplied into Q);
 *  - causal masking is bottom-right aligned: key j is visible to query i iff
 *    j <= i + (N_kv - N_q); for N_q == N_kv this is the pages' "col <= row";
 *  - GQA maps query head h to key/value head h / (Hq / Hkv);
 *  - a row with no visible key has O = 0 and L = -inf;
 *  - decode is the same definition with one query row per (sequence, head) and the whole
 *    cache of that sequence visible ("FlashAttention and Why Attention Is a Memory-Traffic
 *    Problem", section "Prefill versus decode": S is 1 x n);
 *  - the sliding window is the pages' sliding_causal mask ("FlashAttention Explained",
 *    FlexAttention section: key kv is visible to query q iff q >= kv and q - kv <= W), with
 *    the same bottom-right alignment: j is visible to i iff 0 <= (i + N_kv - N_q) - j <= W;
 *  - a block-sparse pattern lists the (query block, key block) pairs to compute
 *    ("FlashAttention, annotated", section 3.3; the BlockMask of "FlashAttention Explained"
 *    with one pattern for every batch and head); keys outside listed blocks are invisible,
 *    and inside a listed block the causal and window rules still apply.
 *
 * Besides the definition the file holds two small pieces of the method itself, written out
 * in the pages' order, so that the pages' worked traces can pin them:
 *  - the FA-2 online recurrence over blocks of one score row ("FlashAttention and GPU Data
 *    Movement", section 3.1), and
 *  - the merge of two (m, l, o) states ("How FlashAttention Reduces HBM Traffic Exactly",
 *    section "Why softmax does not prevent tiling", merged max / normaliser / output).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* ------------------------------------------------------------------------------------ */
/* Storage-type conversions, written from the IEEE binary16 and bfloat16 layouts.         */
/* ------------------------------------------------------------------------------------ */

/* Exact value of a binary16 bit pattern: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Exact value of a bfloat16 bit pattern: the top 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 255;
    int f = h & 127;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);                /* subnormal: f * 2^-133 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

double oracle_half_to_double(uint16_t h, int dtype) {
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(h) : oracle_f16_to_double(h);
}

/* Generic round-to-nearest-even of |x| onto a binary format with `mant` fraction bits,
 * exponent bias `bias` and maximum biased exponent `emax_biased` (all-ones reserved). */
static uint16_t encode_rne(double x, int mant, int ebits) {
    int bias = (1 << (ebits - 1)) - 1;
    int emax = (1 << ebits) - 2;                   /* largest finite biased exponent */
    uint16_t sign = (uint16_t)(signbit(x) ? 1u << (mant + ebits) : 0u);
    uint16_t inf = (uint16_t)(((1u << ebits) - 1u) << mant);
    if (isnan(x)) return (uint16_t)(inf | (1u << (mant - 1)));
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    int e2;
    (void)frexp(ax, &e2);                          /* ax = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                                /* ax in [2^e, 2^(e+1)) */
    if (e < 1 - bias) {
        /* subnormal range: multiples of 2^(1-bias-mant) */
        double q = rint(ldexp(ax, -(1 - bias - mant)));
        return (uint16_t)(sign | (uint16_t)q);   /* q == 2^mant is the smallest normal: same bits */
    }
    double q = rint(ldexp(ax, -(e - mant)));       /* in [2^mant, 2^(mant+1)] */
    if (q >= ldexp(1.0, mant + 1)) {
        q = ldexp(q, -1);
        e += 1;
    }
    int be = e + bias;
    if (be > emax) return (uint16_t)(sign | inf);
    return (uint16_t)(sign | (uint16_t)(be << mant) | (uint16_t)((uint32_t)q - (1u << mant)));
}

uint16_t oracle_double_to_f16(double x) { return encode_rne(x, 10, 5); }
uint16_t oracle_double_to_bf16(double x) { return encode_rne(x, 7, 8); }

/* Lookup table of exact values for all 65536 bit patterns of one storage type. */
static double *make_table(int dtype) {
    double *t = (double *)malloc(65536 * sizeof(double));
    if (!t) return NULL;
    for (uint32_t i = 0; i < 65536; ++i) t[i] = oracle_half_to_double((uint16_t)i, dtype);
    return t;
}

/* ------------------------------------------------------------------------------------ */
/* The definition, one query row at a time.                                               */
/* ------------------------------------------------------------------------------------ */

/* Softmax of one materialised score row and the P V product.
 * s: n scores (-inf = masked), v: value rows addressed through vrow(j), o: d outputs. */
static void softmax_pv_row(const double *s, double *p, int64_t n, const double *tab,
                           const uint16_t *const *vrows, int d, double *o, double *lse) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) m = fmax(m, s[j]);
    if (m == -INFINITY) {                          /* no visible key: O = 0, L = -inf */
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
    for (int64_t j = 0; j < n; ++j) p[j] = exp(s[j] - m) / l;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        if (p[j] == 0.0) continue;
        const uint16_t *vr = vrows[j];
        for (int c = 0; c < d; ++c) o[c] += p[j] * tab[vr[c]];
    }
    *lse = m + log(l);
}

/* The same three steps with the value rows already in fp64 (v: n rows of d). */
static void softmax_pv_row_d(const double *s, double *p, int64_t n, const double *v, int d,
                             double *o, double *lse) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) m = fmax(m, s[j]);
    if (m == -INFINITY) {
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
    for (int64_t j = 0; j < n; ++j) p[j] = exp(s[j] - m) / l;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        if (p[j] == 0.0) continue;
        const double *vr = v + j * d;
        for (int c = 0; c < d; ++c) o[c] += p[j] * vr[c];
    }
    *lse = m + log(l);
}

/* Round n doubles to the storage type (nearest, ties to even), with the conversions above. */
void oracle_round_to_storage(const double *x, uint16_t *out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == ORACLE_BF16 ? oracle_double_to_bf16(x[i]) : oracle_double_to_f16(x[i]);
}

/*
 * Prefill attention for selected rows.  Layouts (contiguous, as on the CUDA side):
 *   q [B, Hq, Nq, d], k/v [B, Hkv, Nkv, d], storage bits of fp16 (dtype 0) or bf16 (1).
 * rows[r] = (b * Hq + h) * Nq + i selects query row i of head h of batch b.
 * Outputs: o[r * d + c] and lse[r] in fp64.  Returns 0, or -1 on bad arguments.
 */
int oracle_attention_rows_masked(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 int dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                                 int causal, int64_t window, const uint8_t *block_mask,
                                 int block, double scale, const int64_t *rows, int64_t n_rows,
                                 double *o, double *lse, int n_threads);

int oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                          int B, int Hq, int Hkv, int Nq, int Nkv, int d, int causal,
                          double scale, const int64_t *rows, int64_t n_rows, double *o,
                          double *lse, int n_threads) {
    return oracle_attention_rows_masked(q, k, v, dtype, B, Hq, Hkv, Nq, Nkv, d, causal, -1, NULL,
                                        0, scale, rows, n_rows, o, lse, n_threads);
}

/*
 * The same with the two masks that change the operator: a sliding window of W keys behind
 * the diagonal (window >= 0; -1 = none) and a block-sparse pattern block_mask
 * [ceil(Nq / block)][ceil(Nkv / block)] (nonzero = compute; NULL = none).
 */
int oracle_attention_rows_masked(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 int dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                                 int causal, int64_t window, const uint8_t *block_mask,
                                 int block, double scale, const int64_t *rows, int64_t n_rows,
                                 double *o, double *lse, int n_threads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq < 0 || Nkv < 0 || d <= 0)
        return -1;
    if (block_mask && block <= 0) return -1;
    const int64_t n_kvb = block_mask ? ((int64_t)Nkv + block - 1) / block : 0;
    if (n_rows == 0) return 0;
    double *tab = make_table(dtype);
    if (!tab) return -1;
    const int group = Hq / Hkv;
    const int64_t off = (int64_t)Nkv - (int64_t)Nq;
    int bad = 0;
    /* Exact fp64 copies of K and V when they fit in 4 GiB (the values are the same either way;
     * the copy only avoids converting each element once per query row). */
    const int64_t kv_elems = (int64_t)B * Hkv * Nkv * d;
    double *kd = NULL, *vd = NULL;
    if (kv_elems > 0 && kv_elems * 16 <= ((int64_t)4 << 30)) {
        kd = (double *)malloc(sizeof(double) * (size_t)kv_elems);
        vd = (double *)malloc(sizeof(double) * (size_t)kv_elems);
        if (kd && vd) {
            for (int64_t x = 0; x < kv_elems; ++x) { kd[x] = tab[k[x]]; vd[x] = tab[v[x]]; }
        } else {
            free(kd); free(vd); kd = vd = NULL;
        }
    }
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads) reduction(| : bad)
#endif
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(Nkv > 0 ? Nkv : 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !p || !vr || !qd) bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t r = 0; r < n_rows; ++r) {
            if (bad) continue;
            const int64_t row = rows[r];
            const int64_t i = row % Nq;
            const int64_t bh = row / Nq;
            const int64_t h = bh % Hq;
            const int64_t b = bh / Hq;
            if (b >= B) { bad = 1; continue; }
            const int64_t hk = h / group;
            const uint16_t *qp = q + row * d;
            const uint16_t *kp = k + (b * Hkv + hk) * (int64_t)Nkv * d;
            const uint16_t *vp = v + (b * Hkv + hk) * (int64_t)Nkv * d;
            for (int c = 0; c < d; ++c) qd[c] = tab[qp[c]];
            const int64_t plane = (b * Hkv + hk) * (int64_t)Nkv * d;
            /* step 1: the row of S (masked entries are -inf) */
            for (int64_t j = 0; j < Nkv; ++j) {
                vr[j] = vp + j * d;
                if (causal && j > i + off) { s[j] = -INFINITY; continue; }
                if (window >= 0 && (j > i + off || i + off - j > window)) {
                    s[j] = -INFINITY;
                    continue;
                }
                if (block_mask && !block_mask[(i / block) * n_kvb + j / block]) {
                    s[j] = -INFINITY;
                    continue;
                }
                double acc = 0.0;
                if (kd) {
                    const double *kr = kd + plane + j * d;
                    for (int c = 0; c < d; ++c) acc += qd[c] * kr[c];
                } else {
                    const uint16_t *kr = kp + j * d;
                    for (int c = 0; c < d; ++c) acc += qd[c] * tab[kr[c]];
                }
                s[j] = scale * acc;
            }
            /* steps 2 and 3: the row of P, then the row of O */
            if (vd)
                softmax_pv_row_d(s, p, Nkv, vd + plane, d, o + r * d, lse + r);
            else
                softmax_pv_row(s, p, Nkv, tab, vr, d, o + r * d, lse + r);
        }
        free(s); free(p); free(vr); free(qd);
    }
    free(kd); free(vd);
    free(tab);
    return bad ? -1 : 0;
}

/*
 * Decode attention for selected (sequence, head) rows with a packed cache:
 *   q [B, Hq, d]; kc/vc [T_total, Hkv, d]; sequence b owns tokens cu[b] .. cu[b+1]-1.
 * rows[r] = b * Hq + h.  Every token of the sequence is visible (one new query token).
 */
int oracle_decode_rows(const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                       const int32_t *cu, int dtype, int B, int Hq, int Hkv, int d,
                       double scale, const int64_t *rows, int64_t n_rows, double *o,
                       double *lse, int n_threads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
    if (n_rows == 0) return 0;
    int64_t maxlen = 0;
    for (int b = 0; b < B; ++b) {
        int64_t L = (int64_t)cu[b + 1] - cu[b];
        if (L < 0) return -1;
        if (L > maxlen) maxlen = L;
    }
    double *tab = make_table(dtype);
    if (!tab) return -1;
    const int group = Hq / Hkv;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads) reduction(| : bad)
#endif
    {
        size_t cap = (size_t)(maxlen > 0 ? maxlen : 1);
        double *s = (double *)malloc(sizeof(double) * cap);
        double *p = (double *)malloc(sizeof(double) * cap);
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * cap);
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !p || !vr || !qd) bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < n_rows; ++r) {
            if (bad) continue;
            const int64_t b = rows[r] / Hq;
            const int64_t h = rows[r] % Hq;
            if (b >= B) { bad = 1; continue; }
            const int64_t hk = h / group;
            const int64_t t0 = cu[b];
            const int64_t L = (int64_t)cu[b + 1] - t0;
            const uint16_t *qp = q + rows[r] * d;
            for (int c = 0; c < d; ++c) qd[c] = tab[qp[c]];
            for (int64_t j = 0; j < L; ++j) {
                const uint16_t *kr = kc + ((t0 + j) * Hkv + hk) * d;
                vr[j] = vc + ((t0 + j) * Hkv + hk) * d;
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += qd[c] * tab[kr[c]];
                s[j] = scale * acc;
            }
            softmax_pv_row(s, p, L, tab, vr, d, o + r * d, lse + r);
        }
        free(s); free(p); free(vr); free(qd);
    }
    free(tab);
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* The method's own steps, for the pages' worked traces.                                  */
/* ------------------------------------------------------------------------------------ */

/*
 * FA-2 online recurrence over one score row split into blocks ("FlashAttention and GPU
 * Data Movement", section 3.1): for each block,
 *   m_new = max(m_old, max(S_block))
 *   alpha = exp(m_old - m_new)
 *   l     = alpha * l + sum exp(S_block - m_new)
 *   a     = alpha * a + sum exp(S_block - m_new) * V_block
 * and O = a / l after the last block.  s: n scores (-inf allowed), v: n x dv values,
 * block_ends: exclusive end index of each block.  Per block the state after it is written
 * to m_tr[k], l_tr[k], alpha_tr[k], a_tr[k*dv + c].  The start state is m = -inf, l = 0,
 * a = 0; exp(-inf - m) is taken as 0, and a block that leaves m at -inf changes nothing.
 */
int oracle_online_trace(const double *s, const double *v, int n, int dv, const int *block_ends,
                        int n_blocks, double *m_tr, double *l_tr, double *alpha_tr,
                        double *a_tr, double *o_out) {
    double m = -INFINITY, l = 0.0;
    double *a = (double *)calloc((size_t)(dv > 0 ? dv : 1), sizeof(double));
    if (!a) return -1;
    int start = 0;
    for (int kb = 0; kb < n_blocks; ++kb) {
        int end = block_ends[kb];
        if (end < start || end > n) { free(a); return -1; }
        double bmax = -INFINITY;
        for (int j = start; j < end; ++j) bmax = fmax(bmax, s[j]);
        double m_new = fmax(m, bmax);
        double alpha = 1.0;
        if (m_new != -INFINITY) {
            alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
            double bsum = 0.0;
            for (int c = 0; c < dv; ++c) a[c] *= alpha;
            for (int j = start; j < end; ++j) {
                double w = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m_new);
                bsum += w;
                for (int c = 0; c < dv; ++c) a[c] += w * v[(int64_t)j * dv + c];
            }
            l = alpha * l + bsum;
            m = m_new;
        }
        m_tr[kb] = m;
        l_tr[kb] = l;
        alpha_tr[kb] = alpha;
        for (int c = 0; c < dv; ++c) a_tr[(int64_t)kb * dv + c] = a[c];
        start = end;
    }
    for (int c = 0; c < dv; ++c) o_out[c] = (l > 0.0) ? a[c] / l : 0.0;
    free(a);
    return 0;
}

/*
 * Merge of two states (m1, l1, o1) and (m2, l2, o2), o normalised within its block
 * ("How FlashAttention Reduces HBM Traffic Exactly", section "Why softmax does not prevent
 * tiling"):
 *   m = max(m1, m2);  l = e^(m1-m) l1 + e^(m2-m) l2;
 *   o = (e^(m1-m) l1 o1 + e^(m2-m) l2 o2) / l.
 * An empty state has m = -inf and l = 0 and contributes nothing.
 */
void oracle_merge_states(double m1, double l1, const double *o1, double m2, double l2,
                         const double *o2, int dv, double *m, double *l, double *o) {
    double mm = fmax(m1, m2);
    if (mm == -INFINITY) {
        *m = -INFINITY; *l = 0.0;
        for (int c = 0; c < dv; ++c) o[c] = 0.0;
        return;
    }
    double w1 = (m1 == -INFINITY) ? 0.0 : exp(m1 - mm) * l1;
    double w2 = (m2 == -INFINITY) ? 0.0 : exp(m2 - mm) * l2;
    double ll = w1 + w2;
    for (int c = 0; c < dv; ++c) o[c] = (w1 * o1[c] + w2 * o2[c]) / ll;
    *m = mm;
    *l = ll;
}

/* Summary (m, l) of one block of scores ("FlashAttention, annotated", section 3.1). */
void oracle_block_summary(const double *x, int n, double *m, double *l) {
    double mm = -INFINITY;
    for (int j = 0; j < n; ++j) mm = fmax(mm, x[j]);
    double ll = 0.0;
    if (mm != -INFINITY)
        for (int j = 0; j < n; ++j) ll += (x[j] == -INFINITY) ? 0.0 : exp(x[j] - mm);
    *m = mm;
    *l = ll;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
