/*
 * gqaq_oracle.c -- plain, slow, fp64 CPU oracle for the decode-attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this file's library.  It shares no code, header,
 * table or helper with the CUDA library: fp16 decoding below is its own
 * IEEE-754 bit-field routine and nothing here includes a CUDA header.
 *
 * Sources (page title + section):
 *  [OPT]   "Core ML Decode Optimization: Removing the 1.9 GiB Per-Token Copy
 *          Caused by GQA repeat_kv" (OptAI engineering blog), sections
 *          2 "Why Does GQA Replicate KV?" and 3 "Fold Q Instead of Expanding KV".
 *  [QUEST] "Quest: Query-Aware Sparsity for Efficient Long-Context LLM
 *          Inference" (reviewer's summary, jaehun.me), sections "page score is
 *          not an attention probability" (the U(p,q) equation and its upper
 *          bound), "separating page count and token budget" (B = K*S) and
 *          "how the bytes read shrink" (the bytes model).
 *
 * Every function works on double arrays.  Layouts are row-major:
 *   q      [Hq][D]              one sequence's query heads
 *   k, v   [Hkv][Lmax][D]       one sequence's key / value cache
 *   meta   [Hkv][Pmax][2][D]    page minimum row, then page maximum row
 *   scores [Hkv][Pmax]
 *   idx    [Hkv][K]             selected page indices, ascending, -1 padded
 * L is the number of valid tokens (rows [0, L) are attended to), S the page
 * size, Pmax = ceil(Lmax / S) and P = ceil(L / S) the number of valid pages.
 *
 * Parity status: every function below is pinned by a CPU test against
 * something other than itself (a library routine, a closed form, the pages'
 * worked example or brute force); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 -> binary64, from the bit fields (exact).               */
/* ------------------------------------------------------------------------ */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24);              /* subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(mant + 1024), expo - 25); /* (1024+mant) * 2^(e-25) */
    }
    return sign ? -v : v;
}

/* Low-bit KV caches. Neither page defines one: the OPT post's section 5
 * ("KV Cache Update Operations Remain") names the cache-write path as the
 * next target, and the Quest review's section on the 7.03x kernel and 2.23x
 * decode figures says its 4-bit condition is weight quantization, not a
 * 4-bit KV store. Both formats below are this library's own plainest choices,
 * written out here so the GPU variants have a definition to be checked
 * against.
 *
 * 8-bit floating point E4M3 (the fp8 KV-cache variant): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; no infinities, and the codes
 * S.1111.111 are NaN. Normal codes are (8 + m) * 2^(e - 10), subnormal ones
 * (e = 0) m * 2^-9; the largest finite magnitude is 448. */
double oracle_e4m3_to_f64(uint8_t code)
{
    const int sgn = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return sgn ? -v : v;
}

/* fp32 value -> E4M3 code: the nearest of the 127 non-negative finite
 * magnitudes (ties to the even code, i.e. the even mantissa), sign kept;
 * magnitudes above 448 saturate to 448 ("satfinite"); NaN -> 0x7F. */
uint8_t oracle_f32_to_e4m3(float y)
{
    if (isnan(y)) return 0x7F;
    const int sgn = signbit(y) ? 1 : 0;
    const double a = fabs((double)y);
    int best = 0x7E;
    if (a <= 448.0) {
        double best_err = INFINITY;
        for (int c = 0; c <= 0x7E; ++c) {
            const double err = fabs(a - oracle_e4m3_to_f64((uint8_t)c));
            if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) != 0)) {
                best_err = err;
                best = c;
            }
        }
    }
    return (uint8_t)((sgn << 7) | best);
}

void oracle_e4m3_array_to_f64(const uint8_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_e4m3_to_f64(src[i]);
}

void oracle_f32_array_to_e4m3(const float *src, uint8_t *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_f32_to_e4m3(src[i]);
}

/* ------------------------------------------------------------------------ */
/* 4-bit KV cache (a format chosen here, see above): symmetric INT4 with   */
/* one fp32 scale per (token, head) row of D channels.                       */
/*   scale = amax / 7            (fp32 division; amax = max |x| of the row)  */
/*   q     = clamp(rne(x / scale), -7, 7)   (fp32 division, ties to even)    */
/*   code  = q + 8 (a nibble; channel 2i in the low nibble of byte i)        */
/* A row of zeros gets scale 0 and codes 8.  Value = (code - 8) * scale.     */
/* float arithmetic throughout, so the two IEEE divisions round the same     */
/* way as the GPU's.                                                         */
/* ------------------------------------------------------------------------ */
void oracle_int4_quantize_rows(const float *x, int64_t rows, int d, uint8_t *codes, float *scales)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * d;
        float amax = 0.0f;
        for (int i = 0; i < d; ++i) {
            float a = fabsf(xr[i]);
            if (a > amax)
                amax = a;
        }
        float scale = amax / 7.0f;
        scales[r] = scale;
        uint8_t *cr = codes + r * (d / 2);
        for (int i = 0; i < d / 2; ++i)
            cr[i] = 0;
        for (int i = 0; i < d; ++i) {
            int q = 0;
            if (scale > 0.0f) {
                float t = rintf(xr[i] / scale);
                q = t > 7.0f ? 7 : (t < -7.0f ? -7 : (int)t);
            }
            uint8_t nib = (uint8_t)(q + 8);
            cr[i / 2] |= (i & 1) ? (uint8_t)(nib << 4) : nib;
        }
    }
}

void oracle_int4_dequantize_rows(const uint8_t *codes, const float *scales, int64_t rows, int d, double *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < d; ++i) {
            uint8_t byte = codes[r * (d / 2) + i / 2];
            int nib = (i & 1) ? (byte >> 4) : (byte & 15);
            out[r * d + i] = (double)(nib - 8) * (double)scales[r];
        }
}

void oracle_f16_array_to_f64(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_f16_to_f64(src[i]);
}

/* ------------------------------------------------------------------------ */
/* Softmax attention of one query row over n key/value rows (fp64).          */
/* s_t = scale * q . k_t ; p = softmax(s) ; out = sum_t p_t v_t              */
/* ------------------------------------------------------------------------ */
static void attend_rows(int d, int64_t n, const double *qrow, const double *krows,
                        const double *vrows, double scale, double *s, double *out)
{
    double smax = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int i = 0; i < d; ++i)
            dot += qrow[i] * krows[t * d + i];
        s[t] = scale * dot;
        if (s[t] > smax)
            smax = s[t];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        s[t] = exp(s[t] - smax);
        sum += s[t];
    }
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int64_t t = 0; t < n; ++t)
            acc += s[t] * vrows[t * d + i];
        out[i] = acc / sum;
    }
}

/* ------------------------------------------------------------------------ */
/* [OPT] section 2: attention with an explicit repeat_kv.  For each query    */
/* head h the KV head h / G is copied into a fresh buffer (the replica the   */
/* "tile" op makes), then ordinary per-head attention runs on the replica.   */
/* The valid-length prefix mask plays the role of the additive context mask. */
/* Returns 0, or -1 on bad arguments / allocation failure.                   */
/* ------------------------------------------------------------------------ */
int oracle_attn_repeat_kv(int hq, int hkv, int d, int64_t lmax, int64_t l,
                          const double *q, const double *k, const double *v,
                          double scale, double *out)
{
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || l <= 0 || l > lmax)
        return -1;
    int group = hq / hkv;
    double *krep = (double *)malloc(sizeof(double) * (size_t)(l * d));
    double *vrep = (double *)malloc(sizeof(double) * (size_t)(l * d));
    double *s = (double *)malloc(sizeof(double) * (size_t)l);
    if (!krep || !vrep || !s) {
        free(krep); free(vrep); free(s);
        return -1;
    }
    for (int h = 0; h < hq; ++h) {
        int kv = h / group;                 /* repeat_kv order: h = G*kv + g */
        memcpy(krep, k + (int64_t)kv * lmax * d, sizeof(double) * (size_t)(l * d));
        memcpy(vrep, v + (int64_t)kv * lmax * d, sizeof(double) * (size_t)(l * d));
        attend_rows(d, l, q + (int64_t)h * d, krep, vrep, scale, s, out + (int64_t)h * d);
    }
    free(krep); free(vrep); free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [OPT] "Prefill Needs Separate Design": with q_len > 1 new tokens the      */
/* group axis is merged into the sequence axis, and each row keeps its own   */
/* causal mask.  Plain definition, explicit repeat_kv: the chunk's tokens    */
/* sit at cache rows start .. start+q_len-1, and token t of query head h     */
/* attends to cache rows 0 .. start+t of KV head h / G.                      */
/*   q, out [Hq][q_len][D];  k, v [Hkv][Lmax][D]                             */
/* ------------------------------------------------------------------------ */
int oracle_prefill_repeat_kv(int hq, int hkv, int d, int64_t lmax, int q_len, int64_t start,
                             const double *q, const double *k, const double *v,
                             double scale, double *out)
{
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || q_len <= 0 || start < 0 || start + q_len > lmax)
        return -1;
    int group = hq / hkv;
    int64_t l = start + q_len;
    double *krep = (double *)malloc(sizeof(double) * (size_t)(l * d));
    double *vrep = (double *)malloc(sizeof(double) * (size_t)(l * d));
    double *s = (double *)malloc(sizeof(double) * (size_t)l);
    if (!krep || !vrep || !s) {
        free(krep); free(vrep); free(s);
        return -1;
    }
    for (int h = 0; h < hq; ++h) {
        int kv = h / group;                 /* repeat_kv order: h = G*kv + g */
        memcpy(krep, k + (int64_t)kv * lmax * d, sizeof(double) * (size_t)(l * d));
        memcpy(vrep, v + (int64_t)kv * lmax * d, sizeof(double) * (size_t)(l * d));
        for (int t = 0; t < q_len; ++t) {
            const int64_t off = ((int64_t)h * q_len + t) * d;
            attend_rows(d, start + t + 1, q + off, krep, vrep, scale, s, out + off);
        }
    }
    free(krep); free(vrep); free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [OPT] section 3: the folded form.  Q [Hq][D] is read as [Hkv][G][D]       */
/* (a reshape, no copy) and each KV head is read in place for its G rows.    */
/* Same arithmetic per row as the repeat_kv form, so the two agree bit for   */
/* bit when the (kv, g) order matches.                                       */
/* ------------------------------------------------------------------------ */
int oracle_attn_folded(int hq, int hkv, int d, int64_t lmax, int64_t l,
                       const double *q, const double *k, const double *v,
                       double scale, double *out)
{
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || l <= 0 || l > lmax)
        return -1;
    int group = hq / hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)l);
    if (!s)
        return -1;
    for (int kv = 0; kv < hkv; ++kv) {
        const double *kh = k + (int64_t)kv * lmax * d;
        const double *vh = v + (int64_t)kv * lmax * d;
        for (int g = 0; g < group; ++g) {
            const double *qrow = q + ((int64_t)kv * group + g) * d;  /* q_fold[kv][g] */
            double *orow = out + ((int64_t)kv * group + g) * d;      /* out_fold[kv][g] */
            attend_rows(d, l, qrow, kh, vh, scale, s, orow);
        }
    }
    free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [QUEST] page metadata: for page p and channel i, m_{p,i} is the minimum   */
/* and M_{p,i} the maximum of the keys stored in the page.  Page p holds     */
/* tokens [p*S, min(p*S+S, L)).  Pages at or beyond ceil(L/S) are untouched. */
/* ------------------------------------------------------------------------ */
int oracle_page_minmax(int hkv, int d, int64_t lmax, int64_t l, int s,
                       const double *k, double *meta)
{
    if (hkv <= 0 || d <= 0 || s <= 0 || l < 0 || l > lmax)
        return -1;
    int64_t pmax = (lmax + s - 1) / s;
    int64_t pvalid = (l + s - 1) / s;
    for (int kv = 0; kv < hkv; ++kv) {
        for (int64_t p = 0; p < pvalid; ++p) {
            int64_t t0 = p * s;
            int64_t t1 = t0 + s < l ? t0 + s : l;
            double *mn = meta + (((int64_t)kv * pmax + p) * 2 + 0) * d;
            double *mx = meta + (((int64_t)kv * pmax + p) * 2 + 1) * d;
            for (int i = 0; i < d; ++i) {
                double lo = k[((int64_t)kv * lmax + t0) * d + i];
                double hi = lo;
                for (int64_t t = t0 + 1; t < t1; ++t) {
                    double x = k[((int64_t)kv * lmax + t) * d + i];
                    if (x < lo) lo = x;
                    if (x > hi) hi = x;
                }
                mn[i] = lo;
                mx[i] = hi;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Page min/max over an E4M3 key cache (the 8-bit variant above): the same  */
/* per-page, per-channel minimum and maximum as oracle_page_minmax, of the  */
/* keys' values, kept as E4M3 codes. With one positive scale per tensor the */
/* dequantized bounds are scale * value(code). Values are compared after    */
/* decoding; a zero bound is stored as the code 0x00 (+0), so each bound    */
/* has exactly one code (E4M3 repeats no other value). Caches hold no NaN   */
/* codes. Pages at or beyond P are left as they are.                        */
/* ------------------------------------------------------------------------ */
static uint8_t canonical_e4m3(uint8_t code)
{
    return (code & 0x7F) == 0 ? 0 : code;
}

int oracle_page_minmax_e4m3(int hkv, int d, int64_t lmax, int64_t l, int s,
                            const uint8_t *k, uint8_t *meta)
{
    if (hkv <= 0 || d <= 0 || s <= 0 || l < 0 || l > lmax)
        return -1;
    int64_t pmax = (lmax + s - 1) / s;
    int64_t pvalid = (l + s - 1) / s;
    for (int kv = 0; kv < hkv; ++kv) {
        for (int64_t p = 0; p < pvalid; ++p) {
            int64_t t0 = p * s;
            int64_t t1 = t0 + s < l ? t0 + s : l;
            uint8_t *mn = meta + (((int64_t)kv * pmax + p) * 2 + 0) * d;
            uint8_t *mx = meta + (((int64_t)kv * pmax + p) * 2 + 1) * d;
            for (int i = 0; i < d; ++i) {
                uint8_t clo = k[((int64_t)kv * lmax + t0) * d + i], chi = clo;
                double lo = oracle_e4m3_to_f64(clo), hi = lo;
                for (int64_t t = t0 + 1; t < t1; ++t) {
                    uint8_t c = k[((int64_t)kv * lmax + t) * d + i];
                    double x = oracle_e4m3_to_f64(c);
                    if (x < lo) { lo = x; clo = c; }
                    if (x > hi) { hi = x; chi = c; }
                }
                mn[i] = canonical_e4m3(clo);
                mx[i] = canonical_e4m3(chi);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [QUEST] page score U(p,q) = sum_i max(q_i m_{p,i}, q_i M_{p,i}).  With    */
/* grouped query heads, one page set serves a KV head's G query heads, so    */
/* the KV head's score is the largest U over its G folded query rows.        */
/* Pages at or beyond P get -inf.                                            */
/* ------------------------------------------------------------------------ */
int oracle_page_scores(int hq, int hkv, int d, int64_t pmax, int64_t pvalid,
                       const double *q, const double *meta, double *scores)
{
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || pvalid < 0 || pvalid > pmax)
        return -1;
    int group = hq / hkv;
    for (int kv = 0; kv < hkv; ++kv) {
        for (int64_t p = 0; p < pmax; ++p) {
            if (p >= pvalid) {
                scores[(int64_t)kv * pmax + p] = -INFINITY;
                continue;
            }
            const double *mn = meta + (((int64_t)kv * pmax + p) * 2 + 0) * d;
            const double *mx = meta + (((int64_t)kv * pmax + p) * 2 + 1) * d;
            double best = -INFINITY;
            for (int g = 0; g < group; ++g) {
                const double *qrow = q + ((int64_t)kv * group + g) * d;
                double u = 0.0;
                for (int i = 0; i < d; ++i) {
                    double a = qrow[i] * mn[i];
                    double b = qrow[i] * mx[i];
                    u += (a > b) ? a : b;
                }
                if (u > best)
                    best = u;
            }
            scores[(int64_t)kv * pmax + p] = best;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [QUEST] top-K page selection: sort the pages by descending score (lower   */
/* page index first on equal scores), keep the first min(K, P), and return   */
/* them in ascending page order, padded with -1 up to K.                     */
/* ------------------------------------------------------------------------ */
typedef struct { double score; int64_t page; } scored_page;

static int by_score_desc_then_page(const void *a, const void *b)
{
    const scored_page *x = (const scored_page *)a, *y = (const scored_page *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->page > y->page) - (x->page < y->page);
}

static int by_int32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int oracle_topk_pages(int hkv, int64_t pmax, int64_t pvalid, int kpages,
                      const double *scores, int32_t *idx)
{
    if (hkv <= 0 || kpages <= 0 || pvalid < 0 || pvalid > pmax)
        return -1;
    scored_page *tmp = (scored_page *)malloc(sizeof(scored_page) * (size_t)(pvalid > 0 ? pvalid : 1));
    if (!tmp)
        return -1;
    for (int kv = 0; kv < hkv; ++kv) {
        for (int64_t p = 0; p < pvalid; ++p) {
            tmp[p].score = scores[(int64_t)kv * pmax + p];
            tmp[p].page = p;
        }
        qsort(tmp, (size_t)pvalid, sizeof(scored_page), by_score_desc_then_page);
        int64_t n = pvalid < kpages ? pvalid : kpages;
        int32_t *row = idx + (int64_t)kv * kpages;
        for (int64_t j = 0; j < n; ++j)
            row[j] = (int32_t)tmp[j].page;
        qsort(row, (size_t)n, sizeof(int32_t), by_int32);
        for (int64_t j = n; j < kpages; ++j)
            row[j] = -1;
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [QUEST] attention over the selected pages only: for each query head h,    */
/* gather the rows of KV head h/G that lie in its listed pages (page p       */
/* contributes tokens [p*S, min(p*S+S, L))) into fresh buffers, then run     */
/* ordinary softmax attention over the gathered rows.  Entries < 0 or >= P   */
/* are skipped.  Returns -1 if a head ends up with no token.                 */
/* ------------------------------------------------------------------------ */
int oracle_sparse_attn(int hq, int hkv, int d, int64_t lmax, int64_t l, int s,
                       int kpages, const double *q, const double *k, const double *v,
                       const int32_t *idx, double scale, double *out)
{
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || s <= 0 || l <= 0 || l > lmax ||
        kpages <= 0)
        return -1;
    int group = hq / hkv;
    int64_t pvalid = (l + s - 1) / s;
    int64_t cap = (int64_t)kpages * s;
    double *kg = (double *)malloc(sizeof(double) * (size_t)(cap * d));
    double *vg = (double *)malloc(sizeof(double) * (size_t)(cap * d));
    double *sc = (double *)malloc(sizeof(double) * (size_t)cap);
    if (!kg || !vg || !sc) {
        free(kg); free(vg); free(sc);
        return -1;
    }
    int rc = 0;
    for (int h = 0; h < hq && rc == 0; ++h) {
        int kv = h / group;
        const int32_t *row = idx + (int64_t)kv * kpages;
        int64_t n = 0;
        for (int j = 0; j < kpages; ++j) {
            int64_t p = row[j];
            if (p < 0 || p >= pvalid)
                continue;
            int64_t t1 = p * s + s < l ? p * s + s : l;
            for (int64_t t = p * s; t < t1; ++t) {
                memcpy(kg + n * d, k + ((int64_t)kv * lmax + t) * d, sizeof(double) * (size_t)d);
                memcpy(vg + n * d, v + ((int64_t)kv * lmax + t) * d, sizeof(double) * (size_t)d);
                ++n;
            }
        }
        if (n == 0) {
            rc = -1;
            break;
        }
        attend_rows(d, n, q + (int64_t)h * d, kg, vg, scale, sc, out + (int64_t)h * d);
    }
    free(kg); free(vg); free(sc);
    return rc;
}
