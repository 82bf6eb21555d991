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
 *   J_i      = { j : 0 <= j < L, (causal => j <= i), (window_left >= 0 => j >= i - window_left),
 *                   (window_right >= 0 => j <= i + window_right) }
 *   s_ij     = scale * sum_k q[b,i,h,k] * k[b,j,g,k]            (double)
 *   m_i      = max_{j in J_i} s_ij
 *   l_i      = sum_{j in J_i} exp(s_ij - m_i)
 *   O[b,i,h] = sum_{j in J_i} exp(s_ij - m_i) * v[b,j,g,:] / l_i
 *   LSE[b,h,i] = m_i + ln(l_i)                                  (natural log)
 * An empty J_i (impossible for the supported masks) gives O = 0 and LSE = -inf.
 *
 * Decode-shaped problems (oracle_attn_rows_kv): Lq query rows against Lk >= Lq
 * keys, the queries being the LAST Lq positions of the sequence, so row i sits at
 * position p_i = Lk - Lq + i and J_i is the set above with i replaced by p_i and
 * L by Lk (with Lq = Lk this is the square problem). Reading: the pages say a
 * generation step reads the whole KV cache ("What is memory-efficient attention
 * ...", section 1, key limitations), i.e. the new query attends to every cached
 * key before it; bottom-right alignment is that statement for Lq new queries.
 * A key sub-range [key_lo, key_hi) restricts J_i further: the partial result of
 * one split of the keys. A right window window_right = r >= 0 restricts it to
 * j <= p_i + r ("Flash Attention optimization" skill page, workflow 2 step 3:
 * window_size = (left, right), -1 = unbounded; (256, 256) is its symmetric
 * example); causal is the right window 0.
 *
 * Merge of partial results over disjoint key sets (oracle_merge): the softmax
 * over a union of key sets, written from its definition. With LSE_s = m_s + ln l_s
 * of part s, the total normaliser is sum_s exp(LSE_s), so
 *   LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) * O_s.
 * This is how attention computed in parts is combined ("What is memory-efficient
 * attention ...", section 4, ring attention computing attention by parts).
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

enum { ORACLE_FP16 = 0, ORACLE_BF16 = 1, ORACLE_FP8_E4M3 = 2 };

/* Exact widening of one storage value to double.
 * bfloat16: the upper half of an IEEE-754 binary32 value.
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 *           exponent 0 is the subnormal range f * 2^-24, exponent 31 is inf/NaN.
 * float8 e4m3 (in the low byte; the FP8 inputs of the "Flash Attention
 *           optimization" skill page, workflow 3 step 3, torch.float8_e4m3fn):
 *           1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; exponent 0 is
 *           the subnormal range f * 2^-9; exponent 15 with fraction 7 is NaN (there
 *           is no infinity), so the largest value is 448. */
static double widen16(uint16_t bits, int dtype)
{
    if (dtype == ORACLE_FP8_E4M3) {
        int sign8 = (bits >> 7) & 1;
        int e8 = (bits >> 3) & 0xf;
        int f8 = bits & 7;
        double m8;
        if (e8 == 15 && f8 == 7)
            m8 = NAN;
        else if (e8 == 0)
            m8 = ldexp((double)f8, -9);
        else
            m8 = ldexp((double)(f8 + 8), e8 - 10);
        return sign8 ? -m8 : m8;
    }
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

/* One output row (b, h, i) of Lq query rows against Lk keys, restricted to keys
 * [key_lo, key_hi). `s` is scratch for up to Lk scores. */
static void attn_row(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                     int64_t Lq, int64_t Lk, int64_t Hq, int64_t Hkv, int64_t d, int causal,
                     int64_t window_left, int64_t window_right, double scale, int64_t key_lo,
                     int64_t key_hi,
                     int64_t b, int64_t h, int64_t i, double *s, double *qrow, double *o,
                     double *lse)
{
    int64_t g = h / (Hq / Hkv);
    int64_t pos = Lk - Lq + i; /* position of query row i in the sequence */

    /* the visible key range J_i = [j_lo, j_hi) */
    int64_t j_lo = 0, j_hi = Lk;
    if (causal)
        j_hi = pos + 1;
    if (window_right >= 0 && pos + window_right + 1 < j_hi)
        j_hi = pos + window_right + 1;
    if (window_left >= 0 && pos - window_left > j_lo)
        j_lo = pos - window_left;
    if (key_lo > j_lo)
        j_lo = key_lo;
    if (key_hi < j_hi)
        j_hi = key_hi;

    for (int64_t c = 0; c < d; ++c)
        o[c] = 0.0;
    if (j_hi <= j_lo) {
        *lse = -INFINITY;
        return;
    }

    const uint16_t *qi = q + ((b * Lq + i) * Hq + h) * d;
    for (int64_t c = 0; c < d; ++c)
        qrow[c] = widen16(qi[c], dtype);

    /* scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = j_lo; j < j_hi; ++j) {
        const uint16_t *kj = k + ((b * Lk + j) * Hkv + g) * d;
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
        const uint16_t *vj = v + ((b * Lk + j) * Hkv + g) * d;
        double p = exp(s[j - j_lo] - m) / l;
        for (int64_t c = 0; c < d; ++c)
            o[c] += p * widen16(vj[c], dtype);
    }
    *lse = m + log(l);
}

/* Rows are flat LSE indices r = (b * Hq + h) * Lq + i, 0 <= r < B*Hq*Lq.
 * q: [B, Lq, Hq, d]; k, v: [B, Lk, Hkv, d]; keys restricted to [key_lo, key_hi).
 * o_rows: nrows x d doubles; lse_rows: nrows doubles.
 * Returns 0 on success, -1 on a bad argument (nothing written). */
int oracle_attn_rows_kv(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                        int64_t B, int64_t Lq, int64_t Lk, int64_t Hq, int64_t Hkv, int64_t d,
                        int causal, int64_t window_left, int64_t window_right, double scale,
                        int64_t key_lo, int64_t key_hi, const int64_t *rows, int64_t nrows,
                        double *o_rows, double *lse_rows)
{
    if (!q || !k || !v || !rows || !o_rows || !lse_rows)
        return -1;
    if (B < 1 || Lq < 1 || Lk < Lq || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv != 0 ||
        window_left < -1 || window_right < -1 || key_lo < 0 || key_hi > Lk || key_lo > key_hi)
        return -1;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16 && dtype != ORACLE_FP8_E4M3)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= B * Hq * Lq)
            return -1;

    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Lk);
        double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !qrow) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s || !qrow)
                continue;
            int64_t i = rows[r] % Lq;
            int64_t bh = rows[r] / Lq;
            int64_t h = bh % Hq;
            int64_t b = bh / Hq;
            attn_row(q, k, v, dtype, Lq, Lk, Hq, Hkv, d, causal, window_left, window_right, scale,
                     key_lo, key_hi, b, h, i, s, qrow, o_rows + r * d, lse_rows + r);
        }
        free(s);
        free(qrow);
    }
    return bad ? -2 : 0;
}

/* The square problem (Lq = Lk = L, all keys): rows r = (b * Hq + h) * L + i. */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                     int64_t B, int64_t L, int64_t Hq, int64_t Hkv, int64_t d, int causal,
                     int64_t window_left, double scale, const int64_t *rows, int64_t nrows,
                     double *o_rows, double *lse_rows)
{
    return oracle_attn_rows_kv(q, k, v, dtype, B, L, L, Hq, Hkv, d, causal, window_left, -1,
                               scale, 0, L, rows, nrows, o_rows, lse_rows);
}

/* Gradients of the square problem (Lq = Lk = L) for an upstream gradient dO of O:
 * the chain rule applied to the definition above. With P_ij = exp(s_ij - LSE_i) on
 * J_i (0 elsewhere) and O_i = sum_j P_ij v_j:
 *   D_i   = sum_c dO_ic O_ic
 *   dV_j  = sum_{i : j in J_i} P_ij dO_i
 *   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_{i : j in J_i} dS_ij q_i
 * with dK and dV summed over the query heads that share a K/V head. O and LSE are
 * recomputed here in double from the definition. The spec page ("compare Hyena vs
 * FlashAttention at 128k", stage 5) lists the backward pass as not measured; this
 * is its plain definition. dq: [B, L, Hq, d]; dk, dv: [B, L, Hkv, d] (doubles).
 * Returns 0, -1 on a bad argument, -2 when scratch cannot be allocated. */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                    int dtype, int64_t B, int64_t L, int64_t Hq, int64_t Hkv, int64_t d,
                    int causal, int64_t window_left, double scale, double *dq, double *dk,
                    double *dv)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv)
        return -1;
    if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv != 0 || window_left < -1)
        return -1;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16 && dtype != ORACLE_FP8_E4M3)
        return -1;
    int64_t G = Hq / Hkv;
    int bad = 0;
    memset(dq, 0, sizeof(double) * (size_t)(B * L * Hq * d));
    memset(dk, 0, sizeof(double) * (size_t)(B * L * Hkv * d));
    memset(dv, 0, sizeof(double) * (size_t)(B * L * Hkv * d));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bg = 0; bg < B * Hkv; ++bg) {
        int64_t b = bg / Hkv, g = bg % Hkv;
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double *qi = (double *)malloc(sizeof(double) * (size_t)d);
        double *doi = (double *)malloc(sizeof(double) * (size_t)d);
        double *oi = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !qi || !doi || !oi) {
#pragma omp atomic write
            bad = 1;
        } else {
            for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                for (int64_t i = 0; i < L; ++i) {
                    int64_t j_lo = 0, j_hi = L;
                    if (causal)
                        j_hi = i + 1;
                    if (window_left >= 0 && i - window_left > j_lo)
                        j_lo = i - window_left;
                    if (j_hi <= j_lo)
                        continue;
                    const uint16_t *qrow = q + ((b * L + i) * Hq + h) * d;
                    const uint16_t *drow = dout + ((b * L + i) * Hq + h) * d;
                    for (int64_t c = 0; c < d; ++c) {
                        qi[c] = widen16(qrow[c], dtype);
                        doi[c] = widen16(drow[c], dtype);
                        oi[c] = 0.0;
                    }
                    /* scores, their maximum, the normaliser and LSE */
                    double m = -INFINITY;
                    for (int64_t j = j_lo; j < j_hi; ++j) {
                        const uint16_t *krow = k + ((b * L + j) * Hkv + g) * d;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c)
                            dot += qi[c] * widen16(krow[c], dtype);
                        s[j - j_lo] = dot * scale;
                        if (s[j - j_lo] > m)
                            m = s[j - j_lo];
                    }
                    double l = 0.0;
                    for (int64_t j = j_lo; j < j_hi; ++j)
                        l += exp(s[j - j_lo] - m);
                    double lse = m + log(l);
                    /* O_i and D_i */
                    for (int64_t j = j_lo; j < j_hi; ++j) {
                        const uint16_t *vrow = v + ((b * L + j) * Hkv + g) * d;
                        double p = exp(s[j - j_lo] - lse);
                        for (int64_t c = 0; c < d; ++c)
                            oi[c] += p * widen16(vrow[c], dtype);
                    }
                    double D = 0.0;
                    for (int64_t c = 0; c < d; ++c)
                        D += doi[c] * oi[c];
                    /* gradients */
                    double *dqi = dq + ((b * L + i) * Hq + h) * d;
                    for (int64_t j = j_lo; j < j_hi; ++j) {
                        const uint16_t *krow = k + ((b * L + j) * Hkv + g) * d;
                        const uint16_t *vrow = v + ((b * L + j) * Hkv + g) * d;
                        double *dkj = dk + ((b * L + j) * Hkv + g) * d;
                        double *dvj = dv + ((b * L + j) * Hkv + g) * d;
                        double p = exp(s[j - j_lo] - lse);
                        double dp = 0.0;
                        for (int64_t c = 0; c < d; ++c)
                            dp += doi[c] * widen16(vrow[c], dtype);
                        double ds = p * (dp - D);
                        for (int64_t c = 0; c < d; ++c) {
                            dqi[c] += scale * ds * widen16(krow[c], dtype);
                            dkj[c] += scale * ds * qi[c];
                            dvj[c] += p * doi[c];
                        }
                    }
                }
            }
        }
        free(s);
        free(qi);
        free(doi);
        free(oi);
    }
    return bad ? -2 : 0;
}

/* Combine nparts partial results of the same nrows rows, each over a disjoint
 * set of keys: o_parts is nparts x nrows x d, lse_parts nparts x nrows (natural
 * log; -inf for a part that saw no key). Writes o (nrows x d) and lse (nrows). */
void oracle_merge(int64_t nparts, int64_t nrows, int64_t d, const double *o_parts,
                  const double *lse_parts, double *o, double *lse)
{
    for (int64_t r = 0; r < nrows; ++r) {
        double m = -INFINITY;
        for (int64_t p = 0; p < nparts; ++p)
            if (lse_parts[p * nrows + r] > m)
                m = lse_parts[p * nrows + r];
        for (int64_t c = 0; c < d; ++c)
            o[r * d + c] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double total = 0.0;
        for (int64_t p = 0; p < nparts; ++p)
            total += exp(lse_parts[p * nrows + r] - m);
        lse[r] = m + log(total);
        for (int64_t p = 0; p < nparts; ++p) {
            double w = exp(lse_parts[p * nrows + r] - lse[r]);
            for (int64_t c = 0; c < d; ++c)
                o[r * d + c] += w * o_parts[(p * nrows + r) * d + c];
        }
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
