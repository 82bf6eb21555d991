/*
 * attn_oracle.c — plain, slow, obviously correct fp64 CPU oracle for exact
 * scaled-dot-product attention forward (output O and per-row log-sum-exp).
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg may build, load or call this file. It shares no
 * code, header, table or helper with the CUDA path, and the CUDA path never
 * reaches it.
 *
 * What it computes — the plain definition, since the method is exact:
 *   "Flash Attention optimization" skill page (hermes-agent, mlops-flash-attention),
 *     workflow 1 step 2 ("standard attention"): weights = softmax(q kᵀ / √d_k),
 *     out = weights · v; step 4 repeats it with the explicit scale 1/8 at d = 64;
 *     workflow 2 steps 2-3: layout [batch, seq, heads, dim], causal masking,
 *     K/V with fewer heads (MQA/GQA), window_size = (left, right) with -1 = none.
 *   "What is memory-efficient attention for long context on 8x H100?"
 *     (aivaro.ru, answers 650), section 2: the IO-aware tiled method is exact,
 *     i.e. it returns this same softmax(Q Kᵀ) V; it only changes where S lives.
 *
 * For every batch b, query head h < Hq and row i < L, with g = h / (Hq / Hkv):
 *   J_i      = { j : 0 <= j < L, (causal => j <= i), (window_left >= 0 => j >= i - window_left) }
 *   s_ij     = scale * sum_k q[b,i,h,k] * k[b,j,g,k]            (double)
 *   m_i      = max_{j in J_i} s_ij
 *   l_i      = sum_{j in J_i} exp(s_ij - m_i)
 *   O[b,i,h] = sum_{j in J_i} exp(s_ij - m_i) * v[b,j,g,:] / l_i
 *   LSE[b,h,i] = m_i + ln(l_i)                                  (natural log)
 * An empty J_i (impossible for the supported masks) gives O = 0 and LSE = -inf.
 *
 * Readings of points the pages leave open (each is listed in the design notes):
 *   - layout [B, L, H, d] contiguous for Q, K, V and O; LSE is [B, Hq, L];
 *   - query head h reads K/V head h / (Hq / Hkv) (contiguous groups);
 *   - window_left = w admits keys i-w .. i (w + 1 keys), -1 = no window;
 *   - the scale multiplies the raw dot product before the max;
 *   - inputs are the exact fp16 / bf16 bit patterns, widened exactly to double.
 *
 * Build: cc -O2 -fopenmp -fPIC -shared attn_oracle.c -lm (no -ffast-math: the
 * sums run in the written order).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_FP16 = 0, ORACLE_BF16 = 1 };

/* Exact widening of one 16-bit storage value to double.
 * bfloat16: the upper half of an IEEE-754 binary32 value.
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 *           exponent 0 is the subnormal range f * 2^-24, exponent 31 is inf/NaN. */
static double widen16(uint16_t bits, int dtype)
{
    if (dtype == ORACLE_BF16) {
        uint32_t u = (uint32_t)bits << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)frac, -24);
    else if (e == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(frac + 1024), e - 25);
    return sign ? -mag : mag;
}

void oracle_widen(const uint16_t *in, int dtype, double *out, int64_t n)
{
    for (int64_t t = 0; t < n; ++t)
        out[t] = widen16(in[t], dtype);
}

/* One output row (b, h, i). `s` is scratch for up to L scores. */
static void attn_row(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                     int64_t L, int64_t Hq, int64_t Hkv, int64_t d, int causal,
                     int64_t window_left, double scale, int64_t b, int64_t h, int64_t i,
                     double *s, double *qrow, double *o, double *lse)
{
    int64_t g = h / (Hq / Hkv);

    /* the visible key range J_i = [j_lo, j_hi) */
    int64_t j_lo = 0, j_hi = L;
    if (causal)
        j_hi = i + 1;
    if (window_left >= 0 && i - window_left > j_lo)
        j_lo = i - window_left;

    for (int64_t c = 0; c < d; ++c)
        o[c] = 0.0;
    if (j_hi <= j_lo) {
        *lse = -INFINITY;
        return;
    }

    const uint16_t *qi = q + ((b * L + i) * Hq + h) * d;
    for (int64_t c = 0; c < d; ++c)
        qrow[c] = widen16(qi[c], dtype);

    /* scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = j_lo; j < j_hi; ++j) {
        const uint16_t *kj = k + ((b * L + j) * Hkv + g) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += qrow[c] * widen16(kj[c], dtype);
        s[j - j_lo] = scale * dot;
        if (s[j - j_lo] > m)
            m = s[j - j_lo];
    }

    /* normaliser */
    double l = 0.0;
    for (int64_t j = j_lo; j < j_hi; ++j)
        l += exp(s[j - j_lo] - m);

    /* weighted sum of values */
    for (int64_t j = j_lo; j < j_hi; ++j) {
        const uint16_t *vj = v + ((b * L + j) * Hkv + g) * d;
        double p = exp(s[j - j_lo] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            o[c] += p * widen16(vj[c], dtype);
    }
    *lse = m + log(l);
}

/* Rows are flat LSE indices r = (b * Hq + h) * L + i, 0 <= r < B*Hq*L.
 * o_rows: nrows x d doubles; lse_rows: nrows doubles.
 * Returns 0 on success, -1 on a bad argument (nothing written). */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                     int64_t B, int64_t L, int64_t Hq, int64_t Hkv, int64_t d, int causal,
                     int64_t window_left, double scale, const int64_t *rows, int64_t nrows,
                     double *o_rows, double *lse_rows)
{
    if (!q || !k || !v || !rows || !o_rows || !lse_rows)
        return -1;
    if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv != 0 || window_left < -1)
        return -1;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= B * Hq * L)
            return -1;

    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !qrow) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s || !qrow)
                continue;
            int64_t i = rows[r] % L;
            int64_t bh = rows[r] / L;
            int64_t h = bh % Hq;
            int64_t b = bh / Hq;
            attn_row(q, k, v, dtype, L, Hq, Hkv, d, causal, window_left, scale, b, h, i, s,
                     qrow, o_rows + r * d, lse_rows + r);
        }
        free(s);
        free(qrow);
    }
    return bad ? -2 : 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
