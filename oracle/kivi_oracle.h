/*
 * kivi_oracle.h -- plain, slow CPU oracle for KIVI-style asymmetric low-bit
 * KV-cache quantisation and decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library (bit_kv_cache_06_gb300/csrc).
 *
 * Sources (web pages; cited by title and section):
 *   [P2]  "09 -- KV Cache Quantization", sections "The structural fact that
 *         makes KV quant work" and "KIVI -- the reference paper".
 *   [P3]  "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
 *         sections "Quantize along the axis that hides the outliers" and
 *         "The streaming complication".
 *   [P4]  "4.4 KV Cache quantization", section 1 (the M_KV byte formula),
 *         section 2 (P = softmax(QK^T / sqrt d)), section 3.1 (two groupings),
 *         section 3.2 (residual cache).
 *   [P5]  "KV Cache INT4 Quantization for 1M+ Token Context Windows",
 *         section 2 (q = clamp(round(x/S) + Z, 0, 2^b - 1), scale floor 1e-8,
 *         zero = round(-min/scale), two 4-bit codes per byte).
 *   [P1]  "KV Cache Quantization (KIVI & FP4) ...", section 4 (four 2-bit codes
 *         per byte).
 *
 * Numerics: the quantiser works in IEEE fp32 (no FMA contraction; build with
 * -ffp-contract=off), rounding half to even; dequantisation and attention
 * work in fp64.
 *
 * Layout of one cache of P (batch, kv-head) pairs -- identical byte for byte
 * to the CUDA library's so that buffers can be compared with memcmp:
 *   kc, vc : uint8 [P][cap][d*bits/8]  codes packed LSB-first along channels
 *   ks, kz : fp32  [P][cap/G][d]       per-channel key scale / zero
 *   vs, vz : fp32  [P][cap][d/G]       per-token value scale / zero
 *   kr, vr : fp16  [P][Ns+R][d]        sink rows, then the residual window
 *                                       (raw bit patterns)
 */
#ifndef KIVI_ORACLE_H
#define KIVI_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* [P4] section 1: M_KV = 2 * L * B * T * H_kv * d * b (b = bytes/element). */
double orc_kv_bytes(int64_t L, int64_t B, int64_t T, int64_t H_kv, int64_t d,
                    double bytes_per_elem);

/* IEEE binary16 bit pattern -> double (exact). */
double orc_half_to_double(uint16_t h);

/* [P5] section 2: asymmetric min/max parameters of one group, fp32.
 * s = max(fl((mx - mn) / (2^b - 1)), 1e-8);  z = rint(fl(-mn / s)), with a
 * zero result stored as +0 (the pages do not fix the sign of a zero zero
 * point; fixing it makes stored zero points comparable bit for bit). */
void orc_quant_params(float mn, float mx, int bits, float *s, float *z);

enum { ORC_META_FP32 = 0, ORC_META_FP16 = 1 };

/* [P2] "KIVI -- the reference paper" (scale and zero point in fp16): the
 * same quantiser with s rounded UP to a binary16 value that is at least
 * 2^-24 and at least |mn| / 2048 (so |z| <= 2048, an exact binary16
 * integer); z = rint(fl(-mn / s)), +0 for a zero. */
void orc_quant_params_f16(float mn, float mx, int bits, float *s, float *z);

/* [P5] section 2: q = clamp(rint(fl(x / s)) + z, 0, 2^b - 1). */
int orc_encode(float x, float s, float z, int bits);

/* [P4] section 3.1: Key per channel.  x is a [G][d] row-major block (row =
 * token, column = channel); each column gets its own (s, z).  codes [G][d]
 * unpacked, one code per byte. */
void orc_quantize_k_group(const float *x, int G, int d, int bits,
                          float *s, float *z, uint8_t *codes);

/* [P4] section 3.1: Value per token.  x is one token row [d]; each run of G
 * channels gets its own (s, z).  s, z are [d/G]; codes [d] unpacked. */
void orc_quantize_v_token(const float *x, int G, int d, int bits,
                          float *s, float *z, uint8_t *codes);

/* [P1] section 4 / [P5] section 2: 8/bits codes per byte, LSB first along
 * channels.  codes [d] -> packed [d*bits/8]. */
void orc_pack_row(const uint8_t *codes, int d, int bits, uint8_t *packed);
void orc_unpack_row(const uint8_t *packed, int d, int bits, uint8_t *codes);

typedef struct orc_cache {
    int32_t bits, G, R, d;
    int64_t P;          /* number of (batch, kv-head) pairs */
    int64_t cap;        /* capacity in quantised tokens per pair */
    int64_t n_quant;    /* quantised tokens (multiple of R) */
    int64_t n_resid;    /* fp16 residual tokens, 0..R */
    uint8_t *kc, *vc;
    float *ks, *kz, *vs, *vz;
    uint16_t *kr, *vr;  /* [P][Ns + R][d]: Ns sink rows, then R residual slots */
    int64_t Ns;         /* sink tokens kept fp16 (0 = plain KIVI) */
    int64_t n_sink;     /* sink rows filled, 0..Ns */
    int64_t meta;       /* ORC_META_FP32 or ORC_META_FP16 (values kept in the fp32 arrays) */
    int64_t flush;      /* ORC_FLUSH_WINDOW or ORC_FLUSH_GROUP */
    int64_t fp8;        /* 0: b-bit KIVI codes; ORC_FP8_E4M3 / ORC_FP8_E5M2: FP8 KV (bits 8) */
    float fp8_k_scale;  /* per-tensor scales of the FP8 format */
    float fp8_v_scale;
} orc_cache;

/* FP8 KV ([P2] "The lazy default: FP8 KV"; [P4] section 4.2): each flushed
 * element is stored as fp8(x / scale) -- x / scale in fp32, rounded to the
 * nearest fp8 value (ties to the even mantissa) and saturated to the largest
 * finite one -- one byte per element, with one scale per tensor for K and
 * one for V (1.0 uncalibrated).  Dequantised: fp8 value * scale. */
enum { ORC_FP8_E4M3 = 1, ORC_FP8_E5M2 = 2 };
double orc_fp8_round(double x, int fmt);
uint8_t orc_fp8_bits(double v, int fmt);
double orc_fp8_value(uint8_t b, int fmt);

/* Residual flush policies.  WINDOW ([P4] section 3.2): when a token arrives
 * at a full window of R tokens, all R are quantised in one batch.  GROUP
 * ([P3] "The streaming complication": a completed group is frozen as the
 * window slides): only the oldest G tokens -- one key group -- are quantised,
 * so the window slides in steps of G and holds R - G + 1 .. R tokens once it
 * has filled.  Values follow the same counter.  The residual rows of the
 * oracle are kept oldest first. */
enum { ORC_FLUSH_WINDOW = 0, ORC_FLUSH_GROUP = 1 };

/* Tokens the cache holds: n_sink + n_quant + n_resid. */
int64_t orc_tokens(const orc_cache *c);

enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_CAPACITY = -3, ORC_ERR_EMPTY = -6 };

/* [P4] section 3.2 / [P3] "The streaming complication": append T new tokens
 * (k, v fp16 [P][T][d]) to the cache.  [P2] "Anti-patterns": while fewer than
 * Ns tokens have arrived, new tokens fill the fp16 sink rows and are never
 * quantised.  The tokens after them are logically placed after the current
 * residual; of that concatenation (n = n_resid + T' tokens) the last
 * ((n - 1) mod R) + 1 stay in the fp16 residual and the rest are quantised
 * (keys in G-token groups per channel, values per token; key groups count
 * from the first token after the sink).
 * nthreads > 1 splits the pairs over threads; results do not depend on it. */
int orc_prefill(orc_cache *c, const uint16_t *k, const uint16_t *v, int64_t T,
                int nthreads);

/* One decode-step append: exactly orc_prefill with T = 1 (k, v [P][d]). */
int orc_append(orc_cache *c, const uint16_t *k, const uint16_t *v);

/* Dequantised fp64 keys / values of pair p, all orc_tokens() tokens in
 * sequence order (sink rows exact, quantised history, residual exact):
 * out [n][d]. */
void orc_dequant_k(const orc_cache *c, int64_t p, double *out);
void orc_dequant_v(const orc_cache *c, int64_t p, double *out);

/* [P4] section 2: o = softmax(tau * q K^T) V in fp64 over the quantised
 * history followed by the residual.  q is fp16 [P*g][d] (query head i of
 * pair p is row p*g + i, i.e. query head h_q reads kv head h_q / g).
 * rows: indices into [0, P*g) to evaluate (NULL = all, nrows ignored);
 * out [nrows][d] (or [P*g][d]).  Returns ORC_ERR_EMPTY on an empty cache. */
int orc_attention(const orc_cache *c, int g, const uint16_t *q, double tau,
                  const int64_t *rows, int64_t nrows, double *out, int nthreads);

/* One split of the same attention, over concatenated token positions
 * [t0, t1) of row `row`: m = max score, l = sum exp(score - m),
 * o_un[d] = sum exp(score - m) v (unnormalised).  Empty range: m = -inf,
 * l = 0, o_un = 0. */
void orc_attention_partial(const orc_cache *c, int g, const uint16_t *q,
                           double tau, int64_t row, int64_t t0, int64_t t1,
                           double *m, double *l, double *o_un);

/* ---- the CUDA library's packed history layout (a storage format) ----
 * The quantised history of a pair is a sequence of key-group records, one
 * per G tokens (cap / G records per pair, record j at byte j * rec):
 *   Ks[d] fp32 | Kz[d] fp32 | G/SL sub-slices of SL = min(G, 32) tokens, each
 *     Kc[SL][d*b/8] (codes LSB-first along channels) |
 *     Vc[SL][d*b/8] (codes LSB-first along orc_value_position order) |
 *     Vs[SL][d/G] fp32 | Vz[SL][d/G] fp32
 * rec = orc_record_bytes(d, G, bits, meta) = 8 d + G (2 d b / 8 + 8 d / G);
 * with ORC_META_FP16 every scale and zero point is a binary16 (4 d + G (2 d
 * b / 8 + 4 d / G) bytes). */

/* Stored position of value channel c in its token row: channel c of group
 * j = c / G at u = c mod G goes to (d/8) r + (G/8) j + e with r = u / (G/8),
 * e = u mod (G/8), so that the (G/8)-channel runs with the same r of every
 * group sit next to each other; natural order when a run is shorter than a
 * byte ((G/8) b < 8) or G is not a multiple of 8. */
int orc_value_position(int c, int d, int G, int bits);
int64_t orc_record_bytes(int d, int G, int bits, int meta);

/* The n_quant / G filled records of pair p, from the oracle's arrays. */
void orc_export_history(const orc_cache *c, int64_t p, uint8_t *out);

#ifdef __cplusplus
}
#endif
#endif
