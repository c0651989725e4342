/*
 * Decode-attention oracle: plain, slow, double-precision C.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (single-token decode attention, one query row per head):
 *
 *   for every batch element b and query head h, with kv = h / G,
 *   G = n_heads / n_kv_heads and L = seq_lens[b]:
 *     s_j  = scale * sum_d q[b,h,d] * K[b,j,kv,d]            j = 0 .. L-1
 *     m    = max_j s_j
 *     w_j  = exp(s_j - m),   Z = sum_j w_j
 *     out[b,h,e] = sum_j w_j * V[b,j,kv,e] / Z               e = 0 .. Dv-1
 *
 * i.e. softmax(q K^T * scale) V. Split-KV decoding computes this same
 * quantity; only the order of the floating-point additions changes
 * (Attention at 128k: Split Over Context, section 2; The Kernel Level:
 * Attention and MoE, "Decode Starves the SMs"). The two-pass stable form follows the float64 two-pass CPU
 * reference described in section 6 of the first page.
 *
 * A second entry point runs the split-KV method itself in double:
 *   - the online-softmax recurrence over blocks of length Bc inside a
 *     segment (The Kernel Level, "But Softmax Wants the Whole Row"),
 *   - the partial triple (m_s, l_s, O_s) per contiguous segment
 *     (The Kernel Level, "Decode Starves the SMs"; Attention at 128k §2),
 *   - the rescaling merge m = max m_i, l = sum l_i e^{m_i-m},
 *     acc = sum acc_i e^{m_i-m}, out = acc / l (Attention at 128k §2;
 *     aprender issue 3725 design note §2, Kernel B), or the equivalent
 *     LSE-weight form e^{LSE_s - LSE*} (The Kernel Level, same section).
 *   - empty segments are neutral: l = 0, m = -1e30 (Attention at 128k §2).
 * It exists so the tests can pin the split identity; it is not the reference
 * the GPU output is compared with (orc_attention is).
 *
 * Storage: K/V elements are read as stored (f32, f16, bf16 or f64) and
 * widened exactly to double, so storage rounding is not part of any
 * comparison (aprender issue 3725 design note §4, the f16 case).
 *
 * Negative-control switches (flags) deliberately plant the two mistakes the
 * pages warn about, for tests that must see them fail:
 *   ORC_NC_NO_MERGE_RESCALE  drop exp(m_i - m) in the merge
 *                            (Attention at 128k §6, cpu_reference_test)
 *   ORC_NC_NO_ALPHA          drop the alpha = exp(m_old - m_new) rescale in
 *                            the online recurrence (gpuflight decoder block 6)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_F64 = 3 };
enum { ORC_NC_NO_MERGE_RESCALE = 1, ORC_NC_NO_ALPHA = 2 };
enum { ORC_MERGE_ML = 0, ORC_MERGE_LSE = 1 };

typedef struct {
    int32_t batch, n_heads, n_kv_heads, head_dim, v_dim;
    int32_t kv_type;
    int64_t k_batch_stride, k_pos_stride, k_head_stride; /* in elements */
    int64_t v_batch_stride, v_pos_stride, v_head_stride; /* in elements */
    double scale;
} orc_shape_t;

/* ---- storage readers, written from the IEEE-754 binary16 and the bfloat16
 * (truncated binary32) format definitions ---------------------------------- */
static double orc_from_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* subnormal: m * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(mant | 0x400), expo - 25); /* (1.m) * 2^(e-15)    */
    return sign ? -v : v;
}

static double orc_from_bf16(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double orc_read(const void *base, int type, int64_t idx)
{
    switch (type) {
    case ORC_F32: return (double)((const float *)base)[idx];
    case ORC_F16: return orc_from_f16(((const uint16_t *)base)[idx]);
    case ORC_BF16: return orc_from_bf16(((const uint16_t *)base)[idx]);
    default: return ((const double *)base)[idx];
    }
}

static int orc_check(const orc_shape_t *s)
{
    if (!s || s->batch < 1 || s->n_heads < 1 || s->n_kv_heads < 1) return 1;
    if (s->n_heads % s->n_kv_heads) return 1;
    if (s->head_dim < 1 || s->v_dim < 1) return 1;
    if (s->kv_type < ORC_F32 || s->kv_type > ORC_F64) return 1;
    return 0;
}

/* scores s_j for one (b, h) into sc[0..L-1] */
static void orc_scores(const orc_shape_t *s, const double *q, const void *k,
                       int b, int h, int L, double *sc)
{
    int kv = h / (s->n_heads / s->n_kv_heads);
    const double *qh = q + ((int64_t)b * s->n_heads + h) * s->head_dim;
    for (int j = 0; j < L; ++j) {
        int64_t row = (int64_t)b * s->k_batch_stride + (int64_t)j * s->k_pos_stride +
                      (int64_t)kv * s->k_head_stride;
        double dot = 0.0;
        for (int d = 0; d < s->head_dim; ++d)
            dot += qh[d] * orc_read(k, s->kv_type, row + d);
        sc[j] = s->scale * dot;
    }
}

static double orc_v(const orc_shape_t *s, const void *v, int b, int j, int kv, int e)
{
    int64_t idx = (int64_t)b * s->v_batch_stride + (int64_t)j * s->v_pos_stride +
                  (int64_t)kv * s->v_head_stride + e;
    return orc_read(v, s->kv_type, idx);
}

/* The plain definition, two-pass stable softmax. */
static void orc_one(const orc_shape_t *s, const double *q, const void *k, const void *v,
                    int b, int h, int L, double *out, double *sc)
{
    int kv = h / (s->n_heads / s->n_kv_heads);
    orc_scores(s, q, k, b, h, L, sc);
    double m = sc[0];
    for (int j = 1; j < L; ++j)
        if (sc[j] > m) m = sc[j];
    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
        sc[j] = exp(sc[j] - m);
        Z += sc[j];
    }
    for (int e = 0; e < s->v_dim; ++e) {
        double acc = 0.0;
        for (int j = 0; j < L; ++j)
            acc += sc[j] * orc_v(s, v, b, j, kv, e);
        out[e] = acc / Z;
    }
}

/*
 * orc_attention: the oracle proper.
 *   q        double [batch][n_heads][head_dim]
 *   k, v     storage arrays addressed by the shape's strides
 *   seq_lens int32 [batch], each >= 1
 *   pairs    NULL for every (b, h); else n_pairs (b, h) int32 pairs
 *   out      double: [batch][n_heads][v_dim] when pairs is NULL,
 *            else [n_pairs][v_dim]
 *   n_threads  OpenMP threads (<= 0: library default)
 * Returns 0, or 1 for an invalid shape or length.
 */
int orc_attention(const orc_shape_t *s, const double *q, const void *k, const void *v,
                  const int32_t *seq_lens, const int32_t *pairs, int n_pairs,
                  double *out, int n_threads)
{
    if (orc_check(s) || !q || !k || !v || !seq_lens || !out) return 1;
    int n = pairs ? n_pairs : s->batch * s->n_heads;
    int maxL = 0;
    for (int b = 0; b < s->batch; ++b) {
        if (seq_lens[b] < 1) return 1;
        if (seq_lens[b] > maxL) maxL = seq_lens[b];
    }
    for (int i = 0; pairs && i < n; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= s->batch || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= s->n_heads)
            return 1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)maxL);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < n; ++i) {
            int b = pairs ? pairs[2 * i] : i / s->n_heads;
            int h = pairs ? pairs[2 * i + 1] : i % s->n_heads;
            orc_one(s, q, k, v, b, h, seq_lens[b], out + (int64_t)i * s->v_dim, sc);
        }
        free(sc);
    }
    (void)n_threads;
    return 0;
}

/*
 * orc_merge: merge n partial triples (m_i, l_i, O_i) of width dv, O_i
 * un-normalised. ML form: m = max m_i, w_i = e^{m_i - m}, l = sum w_i l_i,
 * out = sum w_i O_i / l. LSE form: LSE_i = m_i + log l_i,
 * LSE* = log sum_i e^{LSE_i}, out = sum_i e^{LSE_i - LSE*} O_i / l_i.
 * Partials with l_i == 0 (and m_i = -1e30) are neutral in both forms. Writes the merged m and l
 * (for the LSE form, m = LSE* and l = 1) and out. Returns 0; 1 if every
 * partial is empty (the merged row is undefined).
 */
int orc_merge(int n, const double *m, const double *l, const double *O, int dv, int form,
              int flags, double *m_out, double *l_out, double *out)
{
    int any = 0;
    for (int i = 0; i < n; ++i)
        if (l[i] > 0.0) any = 1;
    if (!any) return 1;
    for (int e = 0; e < dv; ++e) out[e] = 0.0;
    if (form == ORC_MERGE_LSE) {
        /* LSE_i = m_i + log l_i; an empty partial has LSE_i = -inf, weight 0. */
        double lse_max = -INFINITY;
        for (int i = 0; i < n; ++i)
            if (l[i] > 0.0 && m[i] + log(l[i]) > lse_max) lse_max = m[i] + log(l[i]);
        double z = 0.0;
        for (int i = 0; i < n; ++i)
            if (l[i] > 0.0) z += exp(m[i] + log(l[i]) - lse_max);
        double lse_star = lse_max + log(z);
        for (int i = 0; i < n; ++i) {
            if (l[i] <= 0.0) continue;
            double wgt = exp(m[i] + log(l[i]) - lse_star);
            for (int e = 0; e < dv; ++e) out[e] += wgt * (O[(int64_t)i * dv + e] / l[i]);
        }
        if (m_out) *m_out = lse_star;
        if (l_out) *l_out = 1.0;
        return 0;
    }
    /* ML form, as written: every partial takes part; a neutral one
     * (l = 0, m = -1e30) gets weight exp(-1e30 - M) = 0. */
    double M = m[0];
    for (int i = 1; i < n; ++i)
        if (m[i] > M) M = m[i];
    double L = 0.0;
    for (int i = 0; i < n; ++i) {
        double w = (flags & ORC_NC_NO_MERGE_RESCALE) ? 1.0 : exp(m[i] - M);
        L += w * l[i];
        for (int e = 0; e < dv; ++e) out[e] += w * O[(int64_t)i * dv + e];
    }
    for (int e = 0; e < dv; ++e) out[e] /= L;
    if (m_out) *m_out = M;
    if (l_out) *l_out = L;
    return 0;
}

/*
 * Partial triple of one contiguous segment [j0, j1) by the online-softmax
 * recurrence over blocks of bc positions: from m = -inf, l = 0, O = 0,
 *   m_i = max(m_{i-1}, rowmax(block)), l_i = l_{i-1} e^{m_{i-1}-m_i} + sum e^{s-m_i},
 *   O_i = O_{i-1} e^{m_{i-1}-m_i} + sum e^{s-m_i} v.
 * An empty segment yields the neutral triple l = 0, m = -1e30, O = 0.
 */
static void orc_segment(const orc_shape_t *s, const void *v, int b, int kv, const double *sc,
                        int j0, int j1, int bc, int flags, double *m_out, double *l_out,
                        double *O)
{
    for (int e = 0; e < s->v_dim; ++e) O[e] = 0.0;
    if (j1 <= j0) {
        *m_out = -1e30;
        *l_out = 0.0;
        return;
    }
    double m = -INFINITY, l = 0.0;
    for (int t0 = j0; t0 < j1; t0 += bc) {
        int t1 = t0 + bc < j1 ? t0 + bc : j1;
        double bm = sc[t0];
        for (int j = t0 + 1; j < t1; ++j)
            if (sc[j] > bm) bm = sc[j];
        double mn = bm > m ? bm : m;
        double alpha = (m == -INFINITY) ? 0.0 : exp(m - mn);
        if (flags & ORC_NC_NO_ALPHA) alpha = (m == -INFINITY) ? 0.0 : 1.0;
        l *= alpha;
        for (int e = 0; e < s->v_dim; ++e) O[e] *= alpha;
        for (int j = t0; j < t1; ++j) {
            double p = exp(sc[j] - mn);
            l += p;
            for (int e = 0; e < s->v_dim; ++e) O[e] += p * orc_v(s, v, b, j, kv, e);
        }
        m = mn;
    }
    *m_out = m;
    *l_out = l;
}

/*
 * orc_attention_split: the split-KV method in double. Each (b, h) row's L
 * positions are cut into n_splits contiguous segments of ceil(L / n_splits)
 * positions (trailing segments may be empty), each segment runs the online
 * recurrence with block length bc, and the partials are merged by `form`.
 * If parts_m/parts_l/parts_O are non-NULL the partial triples are also
 * returned, laid out [pair][split] (+ [v_dim] for O). Same pair/out
 * conventions as orc_attention. Returns 0, or 1 on invalid arguments.
 */
int orc_attention_split(const orc_shape_t *s, const double *q, const void *k, const void *v,
                        const int32_t *seq_lens, const int32_t *pairs, int n_pairs,
                        int n_splits, int bc, int form, int flags, double *out,
                        double *parts_m, double *parts_l, double *parts_O)
{
    if (orc_check(s) || !q || !k || !v || !seq_lens || !out || n_splits < 1 || bc < 1)
        return 1;
    int n = pairs ? n_pairs : s->batch * s->n_heads;
    int maxL = 0;
    for (int b = 0; b < s->batch; ++b) {
        if (seq_lens[b] < 1) return 1;
        if (seq_lens[b] > maxL) maxL = seq_lens[b];
    }
    int dv = s->v_dim;
    double *sc = (double *)malloc(sizeof(double) * (size_t)maxL);
    double *pm = (double *)malloc(sizeof(double) * (size_t)n_splits);
    double *pl = (double *)malloc(sizeof(double) * (size_t)n_splits);
    double *pO = (double *)malloc(sizeof(double) * (size_t)n_splits * dv);
    int rc = 0;
    for (int i = 0; i < n && !rc; ++i) {
        int b = pairs ? pairs[2 * i] : i / s->n_heads;
        int h = pairs ? pairs[2 * i + 1] : i % s->n_heads;
        if (b < 0 || b >= s->batch || h < 0 || h >= s->n_heads) { rc = 1; break; }
        int kv = h / (s->n_heads / s->n_kv_heads);
        int L = seq_lens[b];
        int chunk = (L + n_splits - 1) / n_splits;
        orc_scores(s, q, k, b, h, L, sc);
        for (int sp = 0; sp < n_splits; ++sp) {
            int64_t a = (int64_t)sp * chunk, z = a + chunk;
            int j0 = a < L ? (int)a : L, j1 = z < L ? (int)z : L;
            orc_segment(s, v, b, kv, sc, j0, j1, bc, flags, pm + sp, pl + sp,
                        pO + (int64_t)sp * dv);
        }
        if (parts_m) memcpy(parts_m + (int64_t)i * n_splits, pm, sizeof(double) * n_splits);
        if (parts_l) memcpy(parts_l + (int64_t)i * n_splits, pl, sizeof(double) * n_splits);
        if (parts_O)
            memcpy(parts_O + (int64_t)i * n_splits * dv, pO, sizeof(double) * n_splits * dv);
        rc = orc_merge(n_splits, pm, pl, pO, dv, form, flags, NULL, NULL,
                       out + (int64_t)i * dv);
    }
    free(sc);
    free(pm);
    free(pl);
    free(pO);
    return rc;
}

/* Thread count OpenMP would use (1 when built without OpenMP). */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
