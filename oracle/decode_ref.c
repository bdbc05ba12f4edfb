/*
 * Oracle for paged-KV decode attention: plain, slow, float64.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; tests, the smoke check and the benchmark's CPU baseline do.
 * It shares no code with the CUDA library.
 *
 * What it computes (XQA page "TensorRT-LLM 源码完全拆解(二十九)", section
 * "先把 decode 注意力的约束写清楚"): for request b, KV head h and group member g
 *
 *     s_t   = sigma * sum_d q[b, h*G+g, d] * K(b,h,t,d)          t < L_b
 *     lse   = M + ln sum_t exp(s_t - M),   M = max_t s_t
 *     out_d = sum_t exp(s_t - lse) * V(b,h,t,d)
 *
 * with K and V gathered through the block table from the paged pool
 * (XQA page, section "Hopper:一次 TMA 只搬一个页": pool[page][slot][head][d],
 * page = block_table[b][t / P], slot = t % P).
 *
 * KV element formats:
 *   0  bf16 bits
 *   1  e4m3 bytes times a per-(head, tensor) fp32 scale (XQA page, section
 *      "Hopper 路径上 V 不做显式反量化": the KV scale multiplies the stored value)
 *   2  656-byte MLA token (FlashMLA page, section "数据加载"): 512 e4m3 values,
 *      4 fp32 scales (one per 128 values), 64 bf16 RoPE values. K is the 576
 *      values (dequantised NoPE then RoPE); V is the first D_v of them. The
 *      page's dequantisation goes FP8 -> half -> float32, times the float32
 *      scale, -> bfloat16 ("计算环节一"); the products then run on those
 *      bfloat16 values ("数据加载"). So a NoPE value here is
 *      bf16(float32(e4m3) * scale): the float32 product, rounded to nearest
 *      even, then rounded to bf16 (nearest even).
 *   3  float64 (pins only)
 *
 * Split reference: the same sum restricted to a token range [t0, t1), giving a
 * partial output and its lse (an empty range gives lse = -inf and output 0),
 * and the merge of partials (XQA page, section "归约怎么记":
 * m = max m_i, l = sum l_i e^(m_i - m), O = (1/l) sum O~_i e^(m_i - m)),
 * written here in the lse form lse = M + ln sum_i e^(lse_i - M),
 * out = sum_i e^(lse_i - lse) o_i.
 *
 * Parity pins live in tests/test_oracle.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { REF_BF16 = 0, REF_FP8 = 1, REF_MLA656 = 2, REF_F64 = 3 };

typedef struct {
    int32_t B, H_kv, G, D_qk, D_v, P, max_pages, num_pages, kv_dtype, pad;
    double softmax_scale;
} ref_desc;

/* e4m3 (OCP FP8): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN; no infinities. */
double ref_e4m3_value(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);   /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* bf16 is the top half of an IEEE binary32 */
double ref_bf16_value(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
}

static double f32_at(const uint8_t *p)
{
    float f;
    memcpy(&f, p, 4);
    return (double)f;
}

/* Nearest bf16 (ties to even) of a float32, for finite values. */
static double bf16_round(float f)
{
    uint32_t w;
    memcpy(&w, &f, 4);
    uint32_t keep = w >> 16, rest = w & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1;
    return ref_bf16_value((uint16_t)keep);
}

/* Decode logical token t of (b, h) into k[D_qk] and v[D_v]. Returns 0, or -1
 * if the block table points outside the pool. */
static int gather_token(const ref_desc *d, const void *k_pool, const void *v_pool,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_table, int b, int h, int t,
                        double *k, double *v)
{
    int32_t page = block_table[(int64_t)b * d->max_pages + t / d->P];
    int slot = t % d->P;
    if (page < 0 || page >= d->num_pages)
        return -1;
    int64_t row = ((int64_t)page * d->P + slot) * d->H_kv + h;   /* [page][slot][head] */
    if (d->kv_dtype == REF_BF16) {
        const uint16_t *kr = (const uint16_t *)k_pool + row * d->D_qk;
        const uint16_t *vr = (const uint16_t *)v_pool + row * d->D_v;
        for (int i = 0; i < d->D_qk; i++) k[i] = ref_bf16_value(kr[i]);
        for (int i = 0; i < d->D_v; i++) v[i] = ref_bf16_value(vr[i]);
    } else if (d->kv_dtype == REF_FP8) {
        const uint8_t *kr = (const uint8_t *)k_pool + row * d->D_qk;
        const uint8_t *vr = (const uint8_t *)v_pool + row * d->D_v;
        double ks = (double)k_scale[h], vs = (double)v_scale[h];
        for (int i = 0; i < d->D_qk; i++) k[i] = ref_e4m3_value(kr[i]) * ks;
        for (int i = 0; i < d->D_v; i++) v[i] = ref_e4m3_value(vr[i]) * vs;
    } else if (d->kv_dtype == REF_MLA656) {
        const uint8_t *r = (const uint8_t *)k_pool + row * 656;
        for (int i = 0; i < 512; i++)
            k[i] = bf16_round((float)(ref_e4m3_value(r[i]) * f32_at(r + 512 + 4 * (i / 128))));
        for (int i = 0; i < 64; i++) {
            uint16_t bits = (uint16_t)(r[528 + 2 * i] | (r[528 + 2 * i + 1] << 8));
            k[512 + i] = ref_bf16_value(bits);
        }
        for (int i = 0; i < d->D_v; i++) v[i] = k[i];
    } else {
        const double *kr = (const double *)k_pool + row * d->D_qk;
        const double *vr = (const double *)v_pool + row * d->D_v;
        for (int i = 0; i < d->D_qk; i++) k[i] = kr[i];
        for (int i = 0; i < d->D_v; i++) v[i] = vr[i];
    }
    return 0;
}

/*
 * Attention of heads g in [g0, g1) of (b, h) over n tokens: token i is
 * toks[i] when toks is not NULL (a list, for sparse decode), else t0 + i (the
 * range [t0, t0 + n)).
 * q64: float64 queries [B][H_kv*G][D_qk]. Writes out[(g1-g0)][D_v], lse[g1-g0].
 * Returns 0, or -1 on a bad page id.
 */
static int attend_tokens(const ref_desc *d, const double *q64, const void *k_pool,
                         const void *v_pool, const float *k_scale, const float *v_scale,
                         const int32_t *block_table, int b, int h, int g0, int g1,
                         const int32_t *toks, int t0, int n, double *out, double *lse)
{
    int ng = g1 - g0;
    int Dq = d->D_qk, Dv = d->D_v, Hq = d->H_kv * d->G;
    memset(out, 0, sizeof(double) * (size_t)ng * Dv);
    if (n <= 0) {
        for (int g = 0; g < ng; g++) lse[g] = -INFINITY;
        return 0;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)ng * n);
    double *k = (double *)malloc(sizeof(double) * Dq);
    double *v = (double *)malloc(sizeof(double) * Dv);
    int rc = 0;
    /* scores */
    for (int i = 0; i < n && rc == 0; i++) {
        if (gather_token(d, k_pool, v_pool, k_scale, v_scale, block_table, b, h, toks ? toks[i] : t0 + i, k, v)) {
            rc = -1;
            break;
        }
        for (int g = 0; g < ng; g++) {
            const double *qr = q64 + ((int64_t)b * Hq + (int64_t)h * d->G + g0 + g) * Dq;
            double acc = 0.0;
            for (int j = 0; j < Dq; j++) acc += qr[j] * k[j];
            s[(size_t)g * n + i] = d->softmax_scale * acc;
        }
    }
    if (rc == 0) {
        /* log-sum-exp per head */
        for (int g = 0; g < ng; g++) {
            double M = -INFINITY, Z = 0.0;
            for (int i = 0; i < n; i++) if (s[(size_t)g * n + i] > M) M = s[(size_t)g * n + i];
            for (int i = 0; i < n; i++) Z += exp(s[(size_t)g * n + i] - M);
            lse[g] = M + log(Z);
        }
        /* weighted sum of V */
        for (int i = 0; i < n; i++) {
            gather_token(d, k_pool, v_pool, k_scale, v_scale, block_table, b, h, toks ? toks[i] : t0 + i, k, v);
            for (int g = 0; g < ng; g++) {
                double w = exp(s[(size_t)g * n + i] - lse[g]);
                double *o = out + (size_t)g * Dv;
                for (int j = 0; j < Dv; j++) o[j] += w * v[j];
            }
        }
    }
    free(s);
    free(k);
    free(v);
    return rc;
}

/*
 * units: n_units records {b, h, g0, g1, t0, t1}; t1 < 0 means "to L_b".
 * Output for unit u starts at out + u*out_stride (out_stride >= (g1-g0)*D_v)
 * and lse + u*lse_stride. Runs the units in parallel (OpenMP) when built so.
 * Returns the number of units that hit a bad page id.
 */
int ref_attend_units(const ref_desc *d, const double *q64, const void *k_pool,
                     const void *v_pool, const float *k_scale, const float *v_scale,
                     const int32_t *block_table, const int32_t *seqlens, int n_units,
                     const int32_t *units, double *out, int64_t out_stride, double *lse,
                     int64_t lse_stride)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int u = 0; u < n_units; u++) {
        const int32_t *r = units + 6 * u;
        int t1 = r[5] < 0 ? seqlens[r[0]] : r[5];
        if (attend_tokens(d, q64, k_pool, v_pool, k_scale, v_scale, block_table, r[0], r[1],
                          r[2], r[3], NULL, r[4], t1 - r[4], out + (int64_t)u * out_stride,
                          lse + (int64_t)u * lse_stride))
            bad++;
    }
    return bad;
}

/*
 * Sparse decode (FlashMLA page, the decode call with top-k `indices`): unit u
 * {b, h, g0, g1, off, n} attends over the n token positions tokens[off ..
 * off + n) of request b (the caller keeps only positions inside [0, L_b); a
 * position listed twice is two terms of the sum). Outputs as in
 * ref_attend_units. Returns the number of units that hit a bad page id.
 */
int ref_attend_lists(const ref_desc *d, const double *q64, const void *k_pool,
                     const void *v_pool, const float *k_scale, const float *v_scale,
                     const int32_t *block_table, int n_units, const int32_t *units,
                     const int32_t *tokens, double *out, int64_t out_stride, double *lse,
                     int64_t lse_stride)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int u = 0; u < n_units; u++) {
        const int32_t *r = units + 6 * u;
        if (attend_tokens(d, q64, k_pool, v_pool, k_scale, v_scale, block_table, r[0], r[1],
                          r[2], r[3], tokens + r[4], 0, r[5], out + (int64_t)u * out_stride,
                          lse + (int64_t)u * lse_stride))
            bad++;
    }
    return bad;
}

/* Merge n partials (o_i [n][D], lse_i [n]) of one query head into out[D], *lse. */
void ref_combine(int n, int D, const double *o_parts, const double *lse_parts, double *out,
                 double *lse)
{
    double M = -INFINITY;
    for (int i = 0; i < n; i++) if (lse_parts[i] > M) M = lse_parts[i];
    memset(out, 0, sizeof(double) * D);
    if (M == -INFINITY) {   /* every partial empty: no tokens at all */
        *lse = -INFINITY;
        return;
    }
    double Z = 0.0;
    for (int i = 0; i < n; i++) Z += exp(lse_parts[i] - M);
    *lse = M + log(Z);
    for (int i = 0; i < n; i++) {
        double w = exp(lse_parts[i] - *lse);
        for (int j = 0; j < D; j++) out[j] += w * o_parts[(size_t)i * D + j];
    }
}

int ref_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
