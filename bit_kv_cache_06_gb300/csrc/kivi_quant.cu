// kivi_quant.cu -- streaming KIVI quantiser and residual-window kernels.
//
// Keys are quantised per channel over groups of G consecutive tokens, values
// per token over groups of G channels ("4.4 KV Cache quantization", section
// 3.1), with the asymmetric min/max quantiser of "KV Cache INT4 Quantization
// for 1M+ Token Context Windows", section 2, in IEEE fp32:
//   s = max(fl((max - min) / (2^b - 1)), 1e-8),  z = rint(fl(-min / s)),
//   q = clamp(rint(fl(x / s)) + z, 0, 2^b - 1)   (round half to even).
// Codes are packed LSB-first along channels, 8/b per byte ("KV Cache
// Quantization (KIVI & FP4)", section 4).
//
// One CTA of G/16 warps quantises one G-token block of one (batch, kv-head)
// pair, keys and values together, and writes it as one key-group record of
// the history buffer (layout in include/kivi.h).  A lane owns 16 channels
// (32 bytes, one 256-bit load) of 4 token rows of K and of V; eight lanes
// cover a row, so every warp load reads 1 KB of consecutive rows.  Key
// min/max: over the lane's 4 rows, then across the G/4 row sets through
// shared memory, where the first 64 threads finish one channel pair each
// and publish the encode parameters.  Value min/max: over the lane's 16
// channels, then across the G/16 lanes of the group with shuffles.  Values
// are encoded between the two block barriers.  Traffic per token: 512 B
// read and 64-128 B written.
#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kThreads = 256;                        // FP8 and residual-copy CTAs
constexpr int kRowThreads = kHeadDim / 8;           // 16 threads per token row
constexpr int kRowsPerPass = kThreads / kRowThreads;  // 16 token rows per pass
constexpr int kQTok = 4;                             // token rows per lane and tensor

__device__ __forceinline__ uint4 load_stream(const __half *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16 fp16 channels (32 bytes) of one row: one 256-bit load when the address
// is 32-byte aligned (V8), else two 128-bit loads.
template <bool V8>
__device__ __forceinline__ void load_row16(const __half *p, uint32_t (&r)[8])
{
    if constexpr (V8) {
        asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
              "=r"(r[6]), "=r"(r[7])
            : "l"(p));
    } else {
        asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
            : "l"(p));
        asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
            : "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
            : "l"(p + 8));
    }
}

// Correctly rounded fl(x / s) from r = rn(1 / s): q0 = rn(x r), the residual
// e = x - q0 s is exact with one FMA, and rn(q0 + e r) is the correctly rounded
// quotient (Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  Checked against IEEE
// division on 3e9 random operand pairs (fp16 dividends, arbitrary fp32 pairs,
// divisors 3 and 15): identical except for the sign of a zero quotient, which
// no code or zero point depends on.  Three instructions instead of a full
// division per element.
__device__ __forceinline__ float div_rn(float x, float s, float r)
{
    const float q0 = __fmul_rn(x, r);
    const float e = __fmaf_rn(-q0, s, x);
    return __fmaf_rn(e, r, q0);
}

// rn(1 / (2^b - 1)) for the scale division.
template <int BITS> struct QmaxInv;
template <> struct QmaxInv<2> { static constexpr float value = 0x1.555556p-2f; };
template <> struct QmaxInv<4> { static constexpr float value = 0x1.111112p-4f; };

// s = max(fl((mx - mn) / (2^b - 1)), 1e-8), z = rint(fl(-mn / s)) (+0 for a
// zero), r = rn(1 / s) for the element divisions.
//
// With fp16 storage (MF = 1, "09 -- KV Cache Quantization", "KIVI -- the
// reference paper": scale and zero in fp16) the scale is instead raised to at
// least |mn| / 2048 and 2^-24 and rounded up to a binary16 value, which keeps
// |z| <= 2048, an exact binary16 integer.
template <int BITS, int MF = 0>
__device__ __forceinline__ void quant_params(float mn, float mx, float &s, float &z, float &r)
{
    constexpr float kQmax = float((1 << BITS) - 1);
    float scale = div_rn(__fsub_rn(mx, mn), kQmax, QmaxInv<BITS>::value);
    if constexpr (MF) {
        scale = fmaxf(fmaxf(scale, fabsf(mn) * 0x1p-11f), 0x1p-24f);   // |mn| / 2048: exact
        scale = __half2float(__float2half_ru(scale));
    } else if (scale < 1e-8f) {
        scale = 1e-8f;
    }
    const float inv = __frcp_rn(scale);
    float zero = rintf(div_rn(-mn, scale, inv));
    if (zero == 0.0f)
        zero = 0.0f;    // a zero zero-point is stored as +0
    s = scale;
    z = zero;
    r = inv;
}

// Encode parameters of one group: the stored scale s and zero point z, and
// for the element loop -s, z and r = rn(1 / s).  Every element of a flat
// group (min == max) has code rint(fl(mn / s)) + rint(fl(-mn / s)) = 0,
// division and rounding half to even being odd functions; such a group
// encodes with r = z = 0, which gives that 0 for any element without the
// large quotients that its 1e-8 scale floor would produce.
struct GroupParams {
    float s, z;          // stored
    float ns, ze, re;    // element loop
};

template <int BITS, int MF>
__device__ __forceinline__ GroupParams group_params(float mn, float mx)
{
    GroupParams g;
    float r;
    quant_params<BITS, MF>(mn, mx, g.s, g.z, r);
    const bool flat = mn == mx;
    g.ns = -g.s;
    g.ze = flat ? 0.0f : g.z;
    g.re = flat ? 0.0f : r;
    return g;
}

constexpr float kMagic = 12582912.0f;      // M = 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;

// Codes of a pair of elements as the fp32 values M + clamp(rint(fl(x / s)) +
// z, 0, qmax): the code is the low mantissa bits of the result.  fl(x / s)
// is the correctly rounded quotient (div_rn in fp32x2 lanes).  Adding M
// rounds it half to even to an integer because |fl(x / s)| < 2^22: two
// distinct fp16 values differ by at least 2^-12 of the larger magnitude (or
// by 2^-24 among subnormals), which bounds |x| / s by qmax * 2^12 in a group
// with min < max, and a flat group has r = 0 and quotient 0.  M + rint + z
// is then an exact integer in [2^23, 2^24).  Only the upper clamp can bind:
// z = rint(fl(-mn / s)) = -rint(fl(mn / s)), so the code of mn is exactly 0,
// and x >= mn with monotone steps gives codes >= 0.
template <int BITS>
__device__ __forceinline__ float2 encode2(__half2 xh, float2 ns, float2 z, float2 r)
{
    constexpr float kTop = kMagic + float((1 << BITS) - 1);
    const float2 x = __half22float2(xh);
    const float2 q0 = __fmul2_rn(x, r);
    const float2 e = __ffma2_rn(q0, ns, x);
    const float2 t = __ffma2_rn(e, r, q0);
    const float2 v = __fadd2_rn(__fadd2_rn(t, make_float2(kMagic, kMagic)), z);
    return make_float2(fminf(v.x, kTop), fminf(v.y, kTop));
}

// Sum of kMagicBits << (BITS m) over the 32 / BITS code fields of a word,
// modulo 2^32.  Accumulating the fp32 bit patterns of M + c_m with weights
// 2^(BITS m) onto minus this bias leaves the packed codes (sum c_m 2^(BITS m)
// is below 2^32).
template <int BITS>
__host__ __device__ constexpr uint32_t pack_bias()
{
    uint32_t c = 0;
    for (int m = 0; m < 32 / BITS; ++m)
        c += kMagicBits << (BITS * m);
    return c;
}

// Add the codes of channels m, m + 1 (of a lane's 16, packed LSB first in
// BITS / 2 words) to acc.
template <int BITS>
__device__ __forceinline__ void pack_pair(uint32_t *acc, int m, float2 v)
{
    constexpr int CPW = 32 / BITS;
    acc[m / CPW] += __float_as_uint(v.x) << (BITS * (m % CPW));
    acc[(m + 1) / CPW] += __float_as_uint(v.y) << (BITS * ((m + 1) % CPW));
}

__device__ __forceinline__ __half2 as_h2(uint32_t u)
{
    __half2 h;
    *reinterpret_cast<uint32_t *>(&h) = u;
    return h;
}

__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Row of token u of the concatenation [old residual, new input tokens].
__device__ __forceinline__ const __half *concat_row(const QuantArgs &a, const __half *res,
                                                    const __half *in, int p, int b, int h,
                                                    int64_t u)
{
    if (u < a.n_old) {
        const int slot = (int)((a.head + u) % a.R);          // the residual is a ring
        return res + ((int64_t)p * a.rows + a.Ns + slot) * kHeadDim;
    }
    return in + b * a.in_sb + h * a.in_sh + (u - a.n_old + a.skip) * a.in_st;
}

// Scale and zero point pair j (channels 2j, 2j + 1) of a metadata array.
template <int MF>
__device__ __forceinline__ void meta_store_pair(void *base, int j, float v0, float v1)
{
    if constexpr (MF)
        reinterpret_cast<__half2 *>(base)[j] = __floats2half2_rn(v0, v1);   // exact: binary16 values
    else
        reinterpret_cast<float2 *>(base)[j] = make_float2(v0, v1);
}

// Store a lane's 16 value codes (channels 16 c16 .. 16 c16 + 15, packed LSB
// first in acc) into its token row in the stored channel order: runs of G/8
// channels with the same index inside their group go to bit BITS (16 r +
// (G/8) j) of the row, r being the run's index inside group j.  Natural
// order when a run is shorter than a byte or G = d.
template <int BITS, int G>
__device__ __forceinline__ void store_value_codes(unsigned char *row, const uint32_t *acc, int c16)
{
    constexpr int RL = G / 8, RBITS = RL * BITS;
    if constexpr (RBITS < 8 || G == kHeadDim) {
        if constexpr (BITS == 2)
            reinterpret_cast<uint32_t *>(row)[c16] = acc[0];
        else
            reinterpret_cast<uint2 *>(row)[c16] = make_uint2(acc[0], acc[1]);
    } else {
        static_assert(RBITS == 8 || RBITS == 16 || RBITS == 32, "run width");
        const int j = 16 * c16 / G;              // value group of the lane
        const int r0 = (16 * c16 % G) / RL;      // its first run
#pragma unroll
        for (int k = 0; k < 16 / RL; ++k) {
            const int bit = k * RBITS;
            const uint32_t wv = acc[bit / 32] >> (bit % 32);
            unsigned char *dst = row + BITS * (16 * (r0 + k) + RL * j) / 8;
            if constexpr (RBITS == 8)
                *dst = (unsigned char)wv;
            else if constexpr (RBITS == 16)
                *reinterpret_cast<uint16_t *>(dst) = (uint16_t)wv;
            else
                *reinterpret_cast<uint32_t *>(dst) = wv;
        }
    }
}

template <int BITS, int G, int MF>
__global__ void __launch_bounds__(2 * G) quantize_kv_kernel(QuantArgs a)
{
    constexpr int D = kHeadDim;
    constexpr int W = G / 16;          // warps
    constexpr int NT = 32 * W;         // threads
    constexpr int RS = 4 * W;          // row sets (warp, lane quad) of the key reduction
    constexpr int SET = 132;           // words per row set: 128 + 4 against bank conflicts
    constexpr int LPG = G / 16;        // lanes per value group
    constexpr int NW = BITS / 2;       // packed words per 16 codes
    constexpr int VG = D / G;
    using RC = Rec<BITS, G, MF>;
    static_assert(G % 16 == 0 && G <= D, "group size");
    // per row set and lane: (min, max) of its 8 channel pairs, four 16-byte
    // chunks rotated by c16 / 2
    __shared__ __align__(16) uint32_t red[RS * SET];
    // per lane column c16: 12 float4 chunks (-s, z, r of channel quads 0..3)
    // at slot (chunk + c16) mod 16
    __shared__ __align__(16) float4 prm[8 * 16];

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int q = lane >> 3, c16 = lane & 7;
    const int64_t grp = blockIdx.x;
    const int p = blockIdx.y;
    const int b = p / a.Hkv;
    const int h = p % a.Hkv;
    const int t0 = 16 * w + q;                      // the lane's rows: t0 + 4 i
    const int64_t u0 = grp * G + t0;

    uint32_t kx[kQTok][8], vx[kQTok][8];
    if (a.v8 && grp * G >= a.n_old) {               // new input rows, 32-byte aligned
        const int64_t off = b * a.in_sb + h * a.in_sh + (u0 - a.n_old + a.skip) * a.in_st + 16 * c16;
#pragma unroll
        for (int i = 0; i < kQTok; ++i) {
            load_row16<true>(a.k_in + off + 4 * i * a.in_st, kx[i]);
            load_row16<true>(a.v_in + off + 4 * i * a.in_st, vx[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < kQTok; ++i) {
            load_row16<false>(concat_row(a, a.k_res, a.k_in, p, b, h, u0 + 4 * i) + 16 * c16, kx[i]);
            load_row16<false>(concat_row(a, a.v_res, a.v_in, p, b, h, u0 + 4 * i) + 16 * c16, vx[i]);
        }
    }
    unsigned char *rec = a.hist + ((int64_t)p * (a.cap / G) + a.n_quant / G + grp) * RC::BYTES;

    // ---- keys: per-channel min/max over the G tokens (fp16, exact) --------
    {
        uint32_t mm[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            __half2 lo = as_h2(kx[0][k]), hi = lo;
#pragma unroll
            for (int i = 1; i < kQTok; ++i) {
                lo = __hmin2(lo, as_h2(kx[i][k]));
                hi = __hmax2(hi, as_h2(kx[i][k]));
            }
            mm[2 * k] = as_u32(lo);
            mm[2 * k + 1] = as_u32(hi);
        }
        uint32_t *set = red + (4 * w + q) * SET + 16 * c16;
#pragma unroll
        for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4 *>(set + 4 * ((v + (c16 >> 1)) & 3)) =
                make_uint4(mm[4 * v], mm[4 * v + 1], mm[4 * v + 2], mm[4 * v + 3]);
    }
    __syncthreads();
    for (int j = tid; j < D / 2; j += NT) {         // channels 2j, 2j + 1
        const int jc = j >> 3, k = j & 7;
        const uint32_t *src = red + 16 * jc + 4 * (((k >> 1) + (jc >> 1)) & 3) + 2 * (k & 1);
        uint2 o = *reinterpret_cast<const uint2 *>(src);
        __half2 lo = as_h2(o.x), hi = as_h2(o.y);
#pragma unroll
        for (int rs = 1; rs < RS; ++rs) {
            o = *reinterpret_cast<const uint2 *>(src + rs * SET);
            lo = __hmin2(lo, as_h2(o.x));
            hi = __hmax2(hi, as_h2(o.y));
        }
        const float2 fl = __half22float2(lo), fh = __half22float2(hi);
        const GroupParams g0 = group_params<BITS, MF>(fl.x, fh.x);
        const GroupParams g1 = group_params<BITS, MF>(fl.y, fh.y);
        float *col = reinterpret_cast<float *>(prm + 16 * jc) + 2 * (k & 1);
        const int v0 = k >> 1;                      // channel quad of the pair
        *reinterpret_cast<float2 *>(col + 4 * ((0 + v0 + jc) & 15)) = make_float2(g0.ns, g1.ns);
        *reinterpret_cast<float2 *>(col + 4 * ((4 + v0 + jc) & 15)) = make_float2(g0.ze, g1.ze);
        *reinterpret_cast<float2 *>(col + 4 * ((8 + v0 + jc) & 15)) = make_float2(g0.re, g1.re);
        meta_store_pair<MF>(rec, j, g0.s, g1.s);
        meta_store_pair<MF>(rec + RC::MW * D, j, g0.z, g1.z);
    }

    // ---- values: per-token groups of G channels, G / 16 lanes per group ----
    // (no key parameter needed: they run before the barrier that publishes those)
#pragma unroll
    for (int i = 0; i < kQTok; ++i) {
        const int t = t0 + 4 * i;
        __half2 lo = as_h2(vx[i][0]), hi = lo;
#pragma unroll
        for (int k = 1; k < 8; ++k) {
            lo = __hmin2(lo, as_h2(vx[i][k]));
            hi = __hmax2(hi, as_h2(vx[i][k]));
        }
        // (min, -max) in one register: the group's lanes reduce it with hmin2
        __half2 mm = __halves2half2(__hmin(__low2half(lo), __high2half(lo)),
                                    __hneg(__hmax(__low2half(hi), __high2half(hi))));
#pragma unroll
        for (int o = 1; o < LPG; o <<= 1)
            mm = __hmin2(mm, as_h2(__shfl_xor_sync(0xffffffffu, as_u32(mm), o)));
        const float2 f = __half22float2(mm);
        const GroupParams g = group_params<BITS, MF>(f.x, -f.y);
        uint32_t acc[NW];
#pragma unroll
        for (int e = 0; e < NW; ++e)
            acc[e] = 0u - pack_bias<BITS>();
        const float2 ns = make_float2(g.ns, g.ns), ze = make_float2(g.ze, g.ze), re = make_float2(g.re, g.re);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            pack_pair<BITS>(acc, 2 * k, encode2<BITS>(as_h2(vx[i][k]), ns, ze, re));
        store_value_codes<BITS, G>(rec + RC::row(t, RC::VC, RC::RB), acc, c16);
        if (c16 % LPG == 0) {
            const int j = 16 * c16 / G;
            meta_store<MF>(rec + RC::row(t, RC::VS, RC::MW * VG), j, g.s);
            meta_store<MF>(rec + RC::row(t, RC::VZ, RC::MW * VG), j, g.z);
        }
    }
    __syncthreads();

    // ---- keys: encode with the published parameters -----------------------
    uint32_t kacc[kQTok][NW];
#pragma unroll
    for (int i = 0; i < kQTok; ++i)
#pragma unroll
        for (int e = 0; e < NW; ++e)
            kacc[i][e] = 0u - pack_bias<BITS>();
    const float4 *P4 = prm + 16 * c16;
#pragma unroll
    for (int v = 0; v < 4; ++v) {                   // channels 4v .. 4v + 3 of the lane
        const float4 ns = P4[(v + c16) & 15], zz = P4[(4 + v + c16) & 15], rr = P4[(8 + v + c16) & 15];
#pragma unroll
        for (int i = 0; i < kQTok; ++i) {
            pack_pair<BITS>(kacc[i], 4 * v,
                            encode2<BITS>(as_h2(kx[i][2 * v]), make_float2(ns.x, ns.y),
                                          make_float2(zz.x, zz.y), make_float2(rr.x, rr.y)));
            pack_pair<BITS>(kacc[i], 4 * v + 2,
                            encode2<BITS>(as_h2(kx[i][2 * v + 1]), make_float2(ns.z, ns.w),
                                          make_float2(zz.z, zz.w), make_float2(rr.z, rr.w)));
        }
    }
#pragma unroll
    for (int i = 0; i < kQTok; ++i) {
        unsigned char *row = rec + RC::row(t0 + 4 * i, RC::KC, RC::RB);
        if constexpr (BITS == 2)
            reinterpret_cast<uint32_t *>(row)[c16] = kacc[i][0];
        else
            reinterpret_cast<uint2 *>(row)[c16] = make_uint2(kacc[i][0], kacc[i][1]);
    }
}

// ----------------------------------------------------------------- FP8 KV ---
// "09 -- KV Cache Quantization", "The lazy default: FP8 KV"; "4.4 KV Cache
// quantization", section 4.2: every element becomes fp8(x / scale) -- x / scale
// correctly rounded in fp32, then rounded to the nearest value of the format
// (ties to even) and saturated to its largest finite value -- one byte per
// element, one scale per tensor.  One CTA writes one 32-token record
// (Kc[32][d] | Vc[32][d]); 16 threads per token row, 8 channels each.

// {x0 -> low byte, x1 -> high byte}
template <int FMT>
__device__ __forceinline__ uint32_t to_fp8x2(float x0, float x1)
{
    uint16_t d;
    if constexpr (FMT == KIVI_FP8_E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(x1), "f"(x0));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(x1), "f"(x0));
    return d;
}

template <int FMT>
__device__ __forceinline__ uint2 fp8_row8(uint4 raw, float s, float r)
{
    const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 x = __half22float2(h[k]);
        w[k] = to_fp8x2<FMT>(div_rn(x.x, s, r), div_rn(x.y, s, r));
    }
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) quantize_fp8_kernel(QuantArgs a)
{
    constexpr int D = kHeadDim, REC = 64 * D;
    const int tid = threadIdx.x, c8 = tid % kRowThreads, r = tid / kRowThreads;
    const int64_t grp = blockIdx.x;
    const int p = blockIdx.y, b = p / a.Hkv, h = p % a.Hkv;
    const float sk = a.fp8_k_scale, sv = a.fp8_v_scale;
    const float rk = __frcp_rn(sk), rv = __frcp_rn(sv);
    unsigned char *rec = a.hist + ((int64_t)p * (a.cap / 32) + a.n_quant / 32 + grp) * REC;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int t = pass * kRowsPerPass + r;                    // token of the record
        const int64_t u = grp * 32 + t;
        const uint4 kx = load_stream(concat_row(a, a.k_res, a.k_in, p, b, h, u) + c8 * 8);
        const uint4 vx = load_stream(concat_row(a, a.v_res, a.v_in, p, b, h, u) + c8 * 8);
        *reinterpret_cast<uint2 *>(rec + t * D + c8 * 8) = fp8_row8<FMT>(kx, sk, rk);
        *reinterpret_cast<uint2 *>(rec + 32 * D + t * D + c8 * 8) = fp8_row8<FMT>(vx, sv, rv);
    }
}

// 16 tokens x 16 chunks of 16 bytes per CTA: input tokens to fp16 rows (the
// sink rows or the residual slots).
__global__ void __launch_bounds__(kThreads) residual_copy_kernel(ResidArgs a)
{
    constexpr int D = kHeadDim;
    const int tid = threadIdx.x;
    const int c8 = tid % kRowThreads;
    const int i = blockIdx.x * kRowsPerPass + tid / kRowThreads;
    if (i >= a.ntok)
        return;
    const int p = blockIdx.y;
    const int b = p / a.Hkv;
    const int h = p % a.Hkv;
    const int64_t src = b * a.in_sb + h * a.in_sh + (a.src_tok0 + i) * a.in_st + c8 * 8;
    const int row = a.ring ? a.dst_row0 + (a.slot0 + i) % a.ring : a.dst_row0 + i;
    const int64_t dst = ((int64_t)p * a.rows + row) * D + c8 * 8;
    *reinterpret_cast<uint4 *>(a.k_res + dst) = load_stream(a.k_in + src);
    *reinterpret_cast<uint4 *>(a.v_res + dst) = load_stream(a.v_in + src);
}

template <int BITS, int MF>
cudaError_t launch_quantize_bits(int G, const QuantArgs &a, int pairs, cudaStream_t s)
{
    dim3 grid((unsigned)(a.nq_new / G), (unsigned)pairs);
    switch (G) {
    case 16: quantize_kv_kernel<BITS, 16, MF><<<grid, 32, 0, s>>>(a); break;
    case 32: quantize_kv_kernel<BITS, 32, MF><<<grid, 64, 0, s>>>(a); break;
    case 64: quantize_kv_kernel<BITS, 64, MF><<<grid, 128, 0, s>>>(a); break;
    case 128: quantize_kv_kernel<BITS, 128, MF><<<grid, 256, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(int bits, int G, int meta, const QuantArgs &a, int pairs, cudaStream_t s)
{
    if (bits == 2)
        return meta ? launch_quantize_bits<2, 1>(G, a, pairs, s) : launch_quantize_bits<2, 0>(G, a, pairs, s);
    if (bits == 4)
        return meta ? launch_quantize_bits<4, 1>(G, a, pairs, s) : launch_quantize_bits<4, 0>(G, a, pairs, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_fp8(int fmt, const QuantArgs &a, int pairs, cudaStream_t s)
{
    dim3 grid((unsigned)(a.nq_new / 32), (unsigned)pairs);
    if (fmt == KIVI_FP8_E4M3)
        quantize_fp8_kernel<KIVI_FP8_E4M3><<<grid, kThreads, 0, s>>>(a);
    else if (fmt == KIVI_FP8_E5M2)
        quantize_fp8_kernel<KIVI_FP8_E5M2><<<grid, kThreads, 0, s>>>(a);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_residual_copy(const ResidArgs &a, int pairs, cudaStream_t s)
{
    dim3 grid((unsigned)((a.ntok + kRowsPerPass - 1) / kRowsPerPass), (unsigned)pairs);
    residual_copy_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kivi
