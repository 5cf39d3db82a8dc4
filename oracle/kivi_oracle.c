/*
 * kivi_oracle.c -- plain, slow CPU oracle (TEST INFRASTRUCTURE ONLY; see
 * kivi_oracle.h for the sources, numerics and layout).  Every loop here is
 * written for reading, not for speed.  Build flags must keep IEEE fp32
 * semantics: -O2 -ffp-contract=off, never -ffast-math.
 */
#include "kivi_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* [P4] section 1: M_KV = 2 L B T H_kv d b.                                  */
double orc_kv_bytes(int64_t L, int64_t B, int64_t T, int64_t H_kv, int64_t d,
                    double bytes_per_elem)
{
    return 2.0 * (double)L * (double)B * (double)T * (double)H_kv *
           (double)d * bytes_per_elem;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                    /* zero / subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)f, e - 25);        /* (1 + f/1024) 2^(e-15) */
    return sign ? -v : v;
}

static float half_to_float(uint16_t h)
{
    return (float)orc_half_to_double(h);              /* exact: fp16 in fp32 */
}

/* ------------------------------------------------------------------------ */
/* [P5] section 2: scale = (max - min) / (2^b - 1), floored at 1e-8;
 * zero = round(-min / scale).  All operations in fp32, round half to even.  */
void orc_quant_params(float mn, float mx, int bits, float *s, float *z)
{
    float qmax = (float)((1 << bits) - 1);
    float range = mx - mn;
    float scale = range / qmax;
    if (scale < 1e-8f)
        scale = 1e-8f;
    float neg_min = -mn;
    float ratio = neg_min / scale;
    float zero = rintf(ratio);
    if (zero == 0.0f)
        zero = 0.0f;      /* store a zero point of zero as +0, never -0 */
    *s = scale;
    *z = zero;
}

/* Smallest IEEE binary16 value >= x, for 0 < x < 65504, returned as a
 * float (every binary16 value is exact in binary32).  The binary16 grid has
 * spacing 2^(e - 10) in [2^e, 2^(e + 1)) for e >= -14 and 2^-24 below 2^-14. */
static float half_ceil(float x)
{
    int e;
    frexp((double)x, &e);                 /* x = m 2^e, 0.5 <= m < 1 */
    int ulp_exp = (e - 1) - 10;           /* x in [2^(e-1), 2^e) */
    if (ulp_exp < -24)
        ulp_exp = -24;
    double ulp = ldexp(1.0, ulp_exp);
    return (float)(ceil((double)x / ulp) * ulp);
}

/* [P2] "KIVI -- the reference paper": scale and zero point stored as fp16.
 * Range-guarded form of the same quantiser: s is rounded up to a binary16
 * value, at least 2^-24 (the smallest positive binary16; the 1e-8 floor lies
 * below it) and at least |min| / 2048, so that z = rint(-min / s) satisfies
 * |z| <= 2048 and is an exact binary16 integer. */
void orc_quant_params_f16(float mn, float mx, int bits, float *s, float *z)
{
    float qmax = (float)((1 << bits) - 1);
    float range = mx - mn;
    float scale = range / qmax;
    float guard = fabsf(mn) / 2048.0f;
    if (scale < guard)
        scale = guard;
    if (scale < 0x1p-24f)
        scale = 0x1p-24f;
    scale = half_ceil(scale);
    float neg_min = -mn;
    float ratio = neg_min / scale;
    float zero = rintf(ratio);
    if (zero == 0.0f)
        zero = 0.0f;
    *s = scale;
    *z = zero;
}

/* [P5] section 2: q = clamp(round(x / S) + Z, 0, 2^b - 1); the rounding is
 * applied to x / S before the zero point is added. */
int orc_encode(float x, float s, float z, int bits)
{
    int64_t qmax = ((int64_t)1 << bits) - 1;
    float ratio = x / s;
    int64_t q = (int64_t)rintf(ratio) + (int64_t)z;
    if (q < 0)
        q = 0;
    if (q > qmax)
        q = qmax;
    return (int)q;
}

static void quant_params_meta(float mn, float mx, int bits, int meta, float *s, float *z)
{
    if (meta == ORC_META_FP16)
        orc_quant_params_f16(mn, mx, bits, s, z);
    else
        orc_quant_params(mn, mx, bits, s, z);
}

/* [P4] section 3.1, "Key per-channel: fix a channel and group consecutive
 * tokens" -- one (s, z) per column of the [G][d] block. */
void orc_quantize_k_group_m(const float *x, int G, int d, int bits, int meta,
                            float *s, float *z, uint8_t *codes)
{
    for (int c = 0; c < d; ++c) {
        float mn = x[c], mx = x[c];
        for (int t = 1; t < G; ++t) {
            float v = x[(int64_t)t * d + c];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        quant_params_meta(mn, mx, bits, meta, &s[c], &z[c]);
        for (int t = 0; t < G; ++t)
            codes[(int64_t)t * d + c] =
                (uint8_t)orc_encode(x[(int64_t)t * d + c], s[c], z[c], bits);
    }
}

void orc_quantize_k_group(const float *x, int G, int d, int bits,
                          float *s, float *z, uint8_t *codes)
{
    orc_quantize_k_group_m(x, G, d, bits, ORC_META_FP32, s, z, codes);
}

/* [P4] section 3.1, "Value per-token: fix a token and group along channels"
 * -- one (s, z) per run of G channels of one token. */
void orc_quantize_v_token_m(const float *x, int G, int d, int bits, int meta,
                            float *s, float *z, uint8_t *codes)
{
    for (int j = 0; j < d / G; ++j) {
        float mn = x[j * G], mx = x[j * G];
        for (int i = 1; i < G; ++i) {
            float v = x[j * G + i];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        quant_params_meta(mn, mx, bits, meta, &s[j], &z[j]);
        for (int i = 0; i < G; ++i)
            codes[j * G + i] = (uint8_t)orc_encode(x[j * G + i], s[j], z[j], bits);
    }
}

void orc_quantize_v_token(const float *x, int G, int d, int bits,
                          float *s, float *z, uint8_t *codes)
{
    orc_quantize_v_token_m(x, G, d, bits, ORC_META_FP32, s, z, codes);
}

/* ------------------------------------------------------------------------ */
/* FP8 KV ("09 -- KV Cache Quantization", "The lazy default: FP8 KV"; "4.4 KV
 * Cache quantization", section 4.2: FP8 still needs a scale).  E4M3: 4
 * exponent bits (bias 7), 3 mantissa bits, largest finite 448, no infinity.
 * E5M2: 5 exponent bits (bias 15), 2 mantissa bits, largest finite 57344.   */

static void fp8_shape(int fmt, int *ebits, int *mbits, double *maxv)
{
    if (fmt == ORC_FP8_E5M2) {
        *ebits = 5; *mbits = 2; *maxv = 57344.0;
    } else {
        *ebits = 4; *mbits = 3; *maxv = 448.0;
    }
}

/* Nearest representable value (ties to the even mantissa), saturated to the
 * largest finite value; x finite. */
double orc_fp8_round(double x, int fmt)
{
    int ebits, mbits;
    double maxv;
    fp8_shape(fmt, &ebits, &mbits, &maxv);
    const int emin = 1 - ((1 << (ebits - 1)) - 1);    /* smallest normal exponent */
    double a = fabs(x);
    if (a == 0.0)
        return x;                                     /* keeps the sign of zero */
    int e;
    frexp(a, &e);                                     /* a in [2^(e-1), 2^e) */
    int ex = e - 1 < emin ? emin : e - 1;
    double q = ldexp(1.0, ex - mbits);                /* spacing of the grid at a */
    double v = nearbyint(a / q) * q;                  /* round half to even */
    if (v > maxv)
        v = maxv;
    return x < 0 ? -v : v;
}

/* The byte of a representable value v (sign, exponent, mantissa). */
uint8_t orc_fp8_bits(double v, int fmt)
{
    int ebits, mbits;
    double maxv;
    fp8_shape(fmt, &ebits, &mbits, &maxv);
    const int bias = (1 << (ebits - 1)) - 1;
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int ex = e - 1;
    if (ex < 1 - bias)                                 /* subnormal: a = m 2^(1-bias-mbits) */
        return (uint8_t)(sign | (uint8_t)ldexp(a, mbits - (1 - bias)));
    uint8_t m = (uint8_t)(ldexp(a, mbits - ex) - (double)(1 << mbits));
    return (uint8_t)(sign | ((ex + bias) << mbits) | m);
}

double orc_fp8_value(uint8_t b, int fmt)
{
    int ebits, mbits;
    double maxv;
    fp8_shape(fmt, &ebits, &mbits, &maxv);
    const int bias = (1 << (ebits - 1)) - 1;
    int sign = b >> 7, ex = (b >> mbits) & ((1 << ebits) - 1), m = b & ((1 << mbits) - 1);
    double v = ex == 0 ? ldexp((double)m, 1 - bias - mbits)
                       : ldexp((double)(m + (1 << mbits)), ex - bias - mbits);
    return sign ? -v : v;
}

/* Channel c goes to byte c*bits/8 at bit offset (c mod (8/bits))*bits. */
void orc_pack_row(const uint8_t *codes, int d, int bits, uint8_t *packed)
{
    int per_byte = 8 / bits;
    memset(packed, 0, (size_t)(d * bits / 8));
    for (int c = 0; c < d; ++c)
        packed[c / per_byte] |= (uint8_t)(codes[c] << ((c % per_byte) * bits));
}

void orc_unpack_row(const uint8_t *packed, int d, int bits, uint8_t *codes)
{
    int per_byte = 8 / bits;
    int mask = (1 << bits) - 1;
    for (int c = 0; c < d; ++c)
        codes[c] = (uint8_t)((packed[c / per_byte] >> ((c % per_byte) * bits)) & mask);
}

/* ------------------------------------------------------------------------ */
/* Cache bookkeeping.                                                        */

static int64_t row_bytes(const orc_cache *c) { return (int64_t)c->d * c->bits / 8; }

typedef struct {
    orc_cache *c;
    const uint16_t *k, *v;
    int64_t T, skip, n, nq_new, r_new;
    int64_t p0, p1;
} prefill_job;

/* fp16 rows of pair p: the Ns sink rows, then the R residual slots. */
static int64_t fp16_rows(const orc_cache *c) { return c->Ns + c->R; }

static uint16_t *resid_slot(const orc_cache *c, uint16_t *buf, int64_t p, int64_t slot)
{
    return buf + (p * fp16_rows(c) + c->Ns + slot) * c->d;
}

/* Concatenation row u of pair p: residual slot u for u < n_resid, else new
 * token u - n_resid (new tokens start at `skip` in the caller's input: the
 * ones before it went to the sink).  Returns fp16 bits. */
static const uint16_t *concat_row(const orc_cache *c, uint16_t *resid,
                                  const uint16_t *fresh, int64_t T, int64_t skip,
                                  int64_t p, int64_t u)
{
    if (u < c->n_resid)
        return resid_slot(c, resid, p, u);
    return fresh + (p * T + skip + (u - c->n_resid)) * c->d;
}

static void prefill_pairs(prefill_job *job)
{
    orc_cache *c = job->c;
    const int d = c->d, G = c->G, R = c->R, bits = c->bits;
    const int64_t rb = row_bytes(c);
    float *xk = malloc(sizeof(float) * (size_t)G * d);
    float *xv = malloc(sizeof(float) * (size_t)d);
    uint8_t *codes = malloc((size_t)G * d);
    uint16_t *keep_k = malloc(sizeof(uint16_t) * (size_t)R * d);
    uint16_t *keep_v = malloc(sizeof(uint16_t) * (size_t)R * d);

    for (int64_t p = job->p0; p < job->p1; ++p) {
        if (c->fp8) {
            /* FP8: every flushed token row on its own, x / scale rounded to
             * the format, one byte per element (no groups, no zero point). */
            for (int64_t u = 0; u < job->nq_new; ++u) {
                const uint16_t *krow = concat_row(c, c->kr, job->k, job->T, job->skip, p, u);
                const uint16_t *vrow = concat_row(c, c->vr, job->v, job->T, job->skip, p, u);
                uint8_t *kd = c->kc + (p * c->cap + c->n_quant + u) * rb;
                uint8_t *vd = c->vc + (p * c->cap + c->n_quant + u) * rb;
                for (int ch = 0; ch < d; ++ch) {
                    float xk = half_to_float(krow[ch]) / c->fp8_k_scale;
                    float xv = half_to_float(vrow[ch]) / c->fp8_v_scale;
                    kd[ch] = orc_fp8_bits(orc_fp8_round(xk, (int)c->fp8), (int)c->fp8);
                    vd[ch] = orc_fp8_bits(orc_fp8_round(xv, (int)c->fp8), (int)c->fp8);
                }
            }
        }
        /* Keys: groups of G consecutive tokens, one (s, z) per channel. */
        for (int64_t j = 0; !c->fp8 && j < job->nq_new / G; ++j) {
            for (int t = 0; t < G; ++t) {
                const uint16_t *row = concat_row(c, c->kr, job->k, job->T, job->skip, p, j * G + t);
                for (int ch = 0; ch < d; ++ch)
                    xk[(int64_t)t * d + ch] = half_to_float(row[ch]);
            }
            int64_t grp = (c->n_quant / G) + j;
            float *s = c->ks + (p * (c->cap / G) + grp) * d;
            float *z = c->kz + (p * (c->cap / G) + grp) * d;
            orc_quantize_k_group_m(xk, G, d, bits, c->meta, s, z, codes);
            for (int t = 0; t < G; ++t) {
                int64_t tok = c->n_quant + j * G + t;
                orc_pack_row(codes + (int64_t)t * d, d, bits,
                             c->kc + (p * c->cap + tok) * rb);
            }
        }
        /* Values: every token on its own, one (s, z) per G channels. */
        for (int64_t u = 0; !c->fp8 && u < job->nq_new; ++u) {
            const uint16_t *row = concat_row(c, c->vr, job->v, job->T, job->skip, p, u);
            for (int ch = 0; ch < d; ++ch)
                xv[ch] = half_to_float(row[ch]);
            int64_t tok = c->n_quant + u;
            float *s = c->vs + (p * c->cap + tok) * (d / G);
            float *z = c->vz + (p * c->cap + tok) * (d / G);
            orc_quantize_v_token_m(xv, G, d, bits, c->meta, s, z, codes);
            orc_pack_row(codes, d, bits, c->vc + (p * c->cap + tok) * rb);
        }
        /* The last r_new tokens of the concatenation become the residual. */
        for (int64_t i = 0; i < job->r_new; ++i) {
            int64_t u = job->nq_new + i;
            memcpy(keep_k + i * d, concat_row(c, c->kr, job->k, job->T, job->skip, p, u),
                   sizeof(uint16_t) * (size_t)d);
            memcpy(keep_v + i * d, concat_row(c, c->vr, job->v, job->T, job->skip, p, u),
                   sizeof(uint16_t) * (size_t)d);
        }
        memcpy(resid_slot(c, c->kr, p, 0), keep_k, sizeof(uint16_t) * (size_t)(job->r_new * d));
        memcpy(resid_slot(c, c->vr, p, 0), keep_v, sizeof(uint16_t) * (size_t)(job->r_new * d));
    }
    free(xk); free(xv); free(codes); free(keep_k); free(keep_v);
}

static void *prefill_thread(void *arg)
{
    prefill_pairs((prefill_job *)arg);
    return NULL;
}

int orc_prefill(orc_cache *c, const uint16_t *k, const uint16_t *v, int64_t T,
                int nthreads)
{
    if (T < 0 || c->R <= 0 || c->G <= 0 || c->Ns < 0)
        return ORC_ERR_ARG;
    if (T == 0)
        return ORC_OK;
    /* "09 -- KV Cache Quantization", "Anti-patterns": the first Ns tokens of
     * the sequence are never quantised.  They fill the sink rows first; only
     * the tokens after them enter the residual / quantised stream. */
    int64_t take = c->Ns - c->n_sink;
    if (take > T)
        take = T;
    int64_t Tq = T - take;
    int64_t n = c->n_resid + Tq;
    int64_t r_new, nq_new;
    if (c->flush == ORC_FLUSH_GROUP) {
        /* [P3] "The streaming complication": a completed key group leaves the
         * window as soon as the window is over-full -- when a token arrives at
         * a full window the oldest G tokens are quantised, so the window holds
         * R - G + 1 .. R tokens once it has filled. */
        int64_t f = n > c->R ? (n - c->R + c->G - 1) / c->G : 0;
        nq_new = f * c->G;
        r_new = n - nq_new;
    } else {
        /* [P4] section 3.2: the whole window is quantised in one batch when a
         * token arrives at a full window. */
        r_new = Tq > 0 ? ((n - 1) % c->R) + 1 : c->n_resid;
        nq_new = Tq > 0 ? n - r_new : 0;
    }
    if (c->n_quant + nq_new > c->cap)
        return ORC_ERR_CAPACITY;
    for (int64_t p = 0; p < c->P; ++p)
        for (int64_t i = 0; i < take; ++i) {
            memcpy(c->kr + (p * fp16_rows(c) + c->n_sink + i) * c->d, k + (p * T + i) * c->d,
                   sizeof(uint16_t) * (size_t)c->d);
            memcpy(c->vr + (p * fp16_rows(c) + c->n_sink + i) * c->d, v + (p * T + i) * c->d,
                   sizeof(uint16_t) * (size_t)c->d);
        }
    c->n_sink += take;
    if (Tq == 0)
        return ORC_OK;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > c->P)
        nthreads = (int)c->P;

    prefill_job *jobs = calloc((size_t)nthreads, sizeof(prefill_job));
    pthread_t *th = calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (prefill_job){c, k, v, T, take, n, nq_new, r_new,
                                c->P * i / nthreads, c->P * (i + 1) / nthreads};
        if (nthreads > 1)
            pthread_create(&th[i], NULL, prefill_thread, &jobs[i]);
        else
            prefill_pairs(&jobs[i]);
    }
    if (nthreads > 1)
        for (int i = 0; i < nthreads; ++i)
            pthread_join(th[i], NULL);
    free(jobs);
    free(th);
    c->n_quant += nq_new;
    c->n_resid = r_new;
    return ORC_OK;
}

int orc_append(orc_cache *c, const uint16_t *k, const uint16_t *v)
{
    return orc_prefill(c, k, v, 1, 1);
}

/* ------------------------------------------------------------------------ */
/* Dequantisation (fp64): x_hat = (q - z) * s; residual tokens are exact.    */

/* Token u of pair p in sequence order: the sink rows, the quantised
 * history, then the residual window.  Sets *row to the fp16 row of a sink
 * or residual token (NULL for a quantised one) and returns the history
 * index of a quantised token. */
static int64_t locate(const orc_cache *c, uint16_t *buf, int64_t p, int64_t u,
                      const uint16_t **row)
{
    if (u < c->n_sink) {
        *row = buf + (p * fp16_rows(c) + u) * c->d;
        return -1;
    }
    u -= c->n_sink;
    if (u < c->n_quant) {
        *row = NULL;
        return u;
    }
    *row = resid_slot(c, buf, p, u - c->n_quant);
    return -1;
}

static void dequant_k_token(const orc_cache *c, int64_t p, int64_t u0, double *out,
                            uint8_t *codes)
{
    const int d = c->d;
    const uint16_t *r;
    const int64_t u = locate(c, c->kr, p, u0, &r);
    if (!r && c->fp8) {
        const uint8_t *b = c->kc + (p * c->cap + u) * row_bytes(c);
        for (int ch = 0; ch < d; ++ch)
            out[ch] = orc_fp8_value(b[ch], (int)c->fp8) * (double)c->fp8_k_scale;
    } else if (!r) {
        orc_unpack_row(c->kc + (p * c->cap + u) * row_bytes(c), d, c->bits, codes);
        const float *s = c->ks + (p * (c->cap / c->G) + u / c->G) * d;
        const float *z = c->kz + (p * (c->cap / c->G) + u / c->G) * d;
        for (int ch = 0; ch < d; ++ch)
            out[ch] = ((double)codes[ch] - (double)z[ch]) * (double)s[ch];
    } else {
        for (int ch = 0; ch < d; ++ch)
            out[ch] = orc_half_to_double(r[ch]);
    }
}

static void dequant_v_token(const orc_cache *c, int64_t p, int64_t u0, double *out,
                            uint8_t *codes)
{
    const int d = c->d, G = c->G;
    const uint16_t *r;
    const int64_t u = locate(c, c->vr, p, u0, &r);
    if (!r && c->fp8) {
        const uint8_t *b = c->vc + (p * c->cap + u) * row_bytes(c);
        for (int ch = 0; ch < d; ++ch)
            out[ch] = orc_fp8_value(b[ch], (int)c->fp8) * (double)c->fp8_v_scale;
    } else if (!r) {
        orc_unpack_row(c->vc + (p * c->cap + u) * row_bytes(c), d, c->bits, codes);
        const float *s = c->vs + (p * c->cap + u) * (d / G);
        const float *z = c->vz + (p * c->cap + u) * (d / G);
        for (int ch = 0; ch < d; ++ch)
            out[ch] = ((double)codes[ch] - (double)z[ch / G]) * (double)s[ch / G];
    } else {
        for (int ch = 0; ch < d; ++ch)
            out[ch] = orc_half_to_double(r[ch]);
    }
}

int64_t orc_tokens(const orc_cache *c) { return c->n_sink + c->n_quant + c->n_resid; }

void orc_dequant_k(const orc_cache *c, int64_t p, double *out)
{
    uint8_t *codes = malloc((size_t)c->d);
    for (int64_t u = 0; u < orc_tokens(c); ++u)
        dequant_k_token(c, p, u, out + u * c->d, codes);
    free(codes);
}

void orc_dequant_v(const orc_cache *c, int64_t p, double *out)
{
    uint8_t *codes = malloc((size_t)c->d);
    for (int64_t u = 0; u < orc_tokens(c); ++u)
        dequant_v_token(c, p, u, out + u * c->d, codes);
    free(codes);
}

/* ------------------------------------------------------------------------ */
/* [P4] section 2: P = softmax(q K^T * tau), o = P V, in fp64.  Two passes
 * over the tokens: scores first, then the max-shifted exponentials.         */

void orc_attention_partial(const orc_cache *c, int g, const uint16_t *q,
                           double tau, int64_t row, int64_t t0, int64_t t1,
                           double *m, double *l, double *o_un)
{
    const int d = c->d;
    const int64_t p = row / g;
    double *qd = malloc(sizeof(double) * (size_t)d);
    double *kv = malloc(sizeof(double) * (size_t)d);
    uint8_t *codes = malloc((size_t)d);
    int64_t n = t1 > t0 ? t1 - t0 : 0;
    double *score = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));

    for (int ch = 0; ch < d; ++ch) {
        qd[ch] = orc_half_to_double(q[row * d + ch]);
        o_un[ch] = 0.0;
    }
    *m = -INFINITY;
    *l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        dequant_k_token(c, p, t0 + i, kv, codes);
        double acc = 0.0;
        for (int ch = 0; ch < d; ++ch)
            acc += qd[ch] * kv[ch];
        score[i] = tau * acc;
        if (score[i] > *m)
            *m = score[i];
    }
    for (int64_t i = 0; i < n; ++i) {
        double w = exp(score[i] - *m);
        *l += w;
        dequant_v_token(c, p, t0 + i, kv, codes);
        for (int ch = 0; ch < d; ++ch)
            o_un[ch] += w * kv[ch];
    }
    free(qd); free(kv); free(codes); free(score);
}

typedef struct {
    const orc_cache *c;
    int g;
    const uint16_t *q;
    double tau;
    const int64_t *rows;
    int64_t i0, i1;
    double *out;
} attn_job;

static void attention_rows(attn_job *job)
{
    const orc_cache *c = job->c;
    const int d = c->d;
    const int64_t ntok = orc_tokens(c);
    for (int64_t i = job->i0; i < job->i1; ++i) {
        int64_t row = job->rows ? job->rows[i] : i;
        double m, l;
        double *o = job->out + i * d;
        orc_attention_partial(c, job->g, job->q, job->tau, row, 0, ntok, &m, &l, o);
        for (int ch = 0; ch < d; ++ch)
            o[ch] /= l;
    }
}

static void *attention_thread(void *arg)
{
    attention_rows((attn_job *)arg);
    return NULL;
}

int orc_attention(const orc_cache *c, int g, const uint16_t *q, double tau,
                  const int64_t *rows, int64_t nrows, double *out, int nthreads)
{
    if (g <= 0)
        return ORC_ERR_ARG;
    if (orc_tokens(c) == 0)
        return ORC_ERR_EMPTY;
    if (!rows)
        nrows = c->P * g;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = nrows > 0 ? (int)nrows : 1;
    attn_job *jobs = calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t *th = calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (attn_job){c, g, q, tau, rows, nrows * i / nthreads,
                             nrows * (i + 1) / nthreads, out};
        if (nthreads > 1)
            pthread_create(&th[i], NULL, attention_thread, &jobs[i]);
        else
            attention_rows(&jobs[i]);
    }
    if (nthreads > 1)
        for (int i = 0; i < nthreads; ++i)
            pthread_join(th[i], NULL);
    free(jobs);
    free(th);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The packed history layout the CUDA library stores (a format, not a step of
 * the method: the pages fix only the grouping axes and "four / two codes per
 * byte").  Written here from the oracle's own arrays so that the two can be
 * compared byte for byte.                                                   */

int orc_value_position(int c, int d, int G, int bits)
{
    int field = (G / 8) * bits;           /* bits of one lane-row's run of a group */
    if (G % 8 != 0 || field < 8)
        return c;                         /* natural order */
    int j = c / G, u = c % G;
    int r = u / (G / 8), e = u % (G / 8);
    return (d / 8) * r + (G / 8) * j + e;
}

int64_t orc_record_bytes(int d, int G, int bits, int meta)
{
    if (bits == 8)
        return 64LL * d;                      /* FP8: 32 tokens of key and value bytes */
    int64_t rb = (int64_t)d * bits / 8, w = meta == ORC_META_FP16 ? 2 : 4;
    return 2 * w * d + (int64_t)G * (2 * rb + 2 * w * (d / G));
}

/* binary16 bit pattern of a float that is exactly a binary16 value (every
 * stored fp16 scale and zero point is: the quantiser makes them so). */
static uint16_t half_bits_exact(float v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs((double)v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                          /* a in [2^(e-1), 2^e) */
    if (e - 1 < -14)                       /* subnormal: a = f 2^-24 */
        return (uint16_t)(sign | (uint16_t)ldexp(a, 24));
    uint16_t f = (uint16_t)(ldexp(a, 10 - (e - 1)) - 1024.0);
    return (uint16_t)(sign | ((e - 1 + 15) << 10) | f);
}

/* Store n metadata values as fp32 or as binary16 bits. */
static void put_meta(uint8_t *dst, const float *src, int n, int meta)
{
    if (meta == ORC_META_FP16) {
        for (int i = 0; i < n; ++i) {
            uint16_t h = half_bits_exact(src[i]);
            memcpy(dst + 2 * i, &h, 2);
        }
    } else {
        memcpy(dst, src, 4 * (size_t)n);
    }
}

void orc_export_history(const orc_cache *c, int64_t p, uint8_t *out)
{
    if (c->fp8) {
        /* records of 32 tokens: key bytes [32][d], then value bytes [32][d] */
        const int d = c->d;
        for (int64_t u = 0; u < c->n_quant; ++u) {
            uint8_t *rec = out + (u / 32) * 64 * d;
            memcpy(rec + (u % 32) * d, c->kc + (p * c->cap + u) * d, (size_t)d);
            memcpy(rec + 32 * d + (u % 32) * d, c->vc + (p * c->cap + u) * d, (size_t)d);
        }
        return;
    }
    const int d = c->d, G = c->G, bits = c->bits, VG = d / G;
    const int64_t rb = row_bytes(c), rec = orc_record_bytes(d, G, bits, c->meta);
    const int w = c->meta == ORC_META_FP16 ? 2 : 4;   /* bytes per scale / zero */
    const int SL = G < 32 ? G : 32;                   /* tokens per sub-slice */
    const int64_t sub = (int64_t)SL * (2 * rb + 2 * w * VG);
    uint8_t *codes = malloc((size_t)d);
    uint8_t *perm = malloc((size_t)d);
    for (int64_t j = 0; j < c->n_quant / G; ++j) {
        uint8_t *r = out + j * rec;
        put_meta(r, c->ks + (p * (c->cap / G) + j) * d, d, c->meta);
        put_meta(r + w * d, c->kz + (p * (c->cap / G) + j) * d, d, c->meta);
        for (int t = 0; t < G; ++t) {
            const int64_t u = j * G + t;                /* history token */
            uint8_t *sl = r + 2 * w * d + (t / SL) * sub;   /* its sub-slice */
            const int i = t % SL;                       /* row in the sub-slice */
            memcpy(sl + i * rb, c->kc + (p * c->cap + u) * rb, (size_t)rb);
            orc_unpack_row(c->vc + (p * c->cap + u) * rb, d, bits, codes);
            for (int ch = 0; ch < d; ++ch)
                perm[orc_value_position(ch, d, G, bits)] = codes[ch];
            orc_pack_row(perm, d, bits, sl + SL * rb + i * rb);
            put_meta(sl + 2 * SL * rb + i * w * VG, c->vs + (p * c->cap + u) * VG, VG, c->meta);
            put_meta(sl + 2 * SL * rb + w * SL * VG + i * w * VG, c->vz + (p * c->cap + u) * VG,
                     VG, c->meta);
        }
    }
    free(codes);
    free(perm);
}
