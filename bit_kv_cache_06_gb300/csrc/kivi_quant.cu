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
// One CTA of 256 threads quantises one G-token block of one (batch, kv-head)
// pair, keys and values together, and writes it as one key-group record of
// the history buffer (layout in include/kivi.h).  Each token row (128 fp16 = 256 B) is read
// by 16 threads with 16-byte loads, so a warp reads two full rows per
// instruction.  The per-channel key reduction runs across the token axis:
// lanes xor 16 first, then the eight warps through shared memory.  Values
// are read in a mapping of their own, two adjacent lanes per (token, channel
// group), so the per-token reduction is local plus one shuffle, and are
// quantised between the two block barriers while the key parameters are
// computed.  Traffic per token: 512 B read and 64-128 B written.
#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kThreads = 256;
constexpr int kRowThreads = kHeadDim / 8;           // 16 threads per token row
constexpr int kRowsPerPass = kThreads / kRowThreads;  // 16 token rows per pass

__device__ __forceinline__ uint4 load_stream(const __half *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
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

// clamp(rint(x / s) + z, 0, qmax) for a pair of elements of a group whose
// minimum is mn, as integer-valued floats, in fp32x2 arithmetic (each lane is
// an IEEE round-to-nearest operation); ns = -s, negated once by the caller.
// rint(x/s) and z are integer-valued; their fp32 sum is exact whenever it
// lies inside the code range and rounds monotonically otherwise, so clamping
// it equals clamping the exact integer sum.  Only the upper clamp is needed:
// z = rint(fl(-mn / s)) = -rint(fl(mn / s)) (division and round-half-even are
// odd functions), so the code of mn is exactly 0, and x >= mn gives
// fl(x / s) >= fl(mn / s) and a code >= 0 (both steps are monotone).
template <int BITS>
__device__ __forceinline__ float2 encode2(float2 x, float2 ns, float2 z, float2 r)
{
    constexpr float kQmax = float((1 << BITS) - 1);
    const float2 q0 = __fmul2_rn(x, r);
    const float2 e = __ffma2_rn(q0, ns, x);
    const float2 t = __ffma2_rn(e, r, q0);
    const float2 q = __fadd2_rn(make_float2(rintf(t.x), rintf(t.y)), z);
    return make_float2(fminf(q.x, kQmax), fminf(q.y, kQmax));
}

// Pack 8 codes (channels 8c..8c+7 of one token, as four (even, odd) pairs)
// LSB first.  The partial sums are integers below 2^16, so every fp32x2 step
// is exact; adding 2^23 puts the integer in the low mantissa bits.
template <int BITS>
__device__ __forceinline__ uint32_t pack8x2(const float2 (&c)[4])
{
    if (BITS == 2) {
        float2 acc = __fmul2_rn(c[0], make_float2(1.0f, 4.0f));
        acc = __ffma2_rn(c[1], make_float2(16.0f, 64.0f), acc);
        acc = __ffma2_rn(c[2], make_float2(256.0f, 1024.0f), acc);
        acc = __ffma2_rn(c[3], make_float2(4096.0f, 16384.0f), acc);
        return __float_as_uint(__fadd_rn(__fadd_rn(acc.x, acc.y), 8388608.0f)) & 0xffffu;
    } else {
        const float2 lo = __ffma2_rn(c[1], make_float2(256.0f, 4096.0f), __fmul2_rn(c[0], make_float2(1.0f, 16.0f)));
        const float2 hi = __ffma2_rn(c[3], make_float2(256.0f, 4096.0f), __fmul2_rn(c[2], make_float2(1.0f, 16.0f)));
        return (__float_as_uint(__fadd_rn(__fadd_rn(lo.x, lo.y), 8388608.0f)) & 0xffffu) |
               (__float_as_uint(__fadd_rn(__fadd_rn(hi.x, hi.y), 8388608.0f)) << 16);
    }
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

// Store this thread's VH value codes (channels vhalf*VH .. of group vg,
// packed eight per word in `packed`) into a token row in the stored channel
// order: runs of G/8 channels go to bit BITS * (16 r + (G/8) vg) of the row,
// r being the run's index inside its group.  Natural order (one contiguous
// store) when a run is shorter than a byte.
template <int BITS, int G, int NW>
__device__ __forceinline__ void store_value_row(unsigned char *row, const uint32_t (&packed)[NW],
                                                int vg, int vhalf)
{
    constexpr int VH = G / 2;
    constexpr int RL = G / 8, RBITS = RL * BITS;     // channels / bits per run
    constexpr int WB = 8 * BITS;                     // bits per packed word
    if constexpr (RBITS < 8 || G == kHeadDim) {
        unsigned char *dst = row + vg * (G * BITS / 8) + vhalf * (VH * BITS / 8);
        if constexpr (BITS == 2) {
            if constexpr (NW == 1) {
                *reinterpret_cast<uint16_t *>(dst) = (uint16_t)packed[0];
            } else {
#pragma unroll
                for (int e = 0; e < NW; e += 2)
                    reinterpret_cast<uint32_t *>(dst)[e / 2] = packed[e] | (packed[e + 1] << 16);
            }
        } else {
#pragma unroll
            for (int e = 0; e < NW; ++e)
                reinterpret_cast<uint32_t *>(dst)[e] = packed[e];
        }
    } else {
        static_assert(RBITS == 8 || RBITS == 16 || RBITS == 32, "run width");
#pragma unroll
        for (int k = 0; k < VH / RL; ++k) {                 // four runs per thread
            const int bit = k * RBITS;
            const uint32_t w = packed[bit / WB] >> (bit % WB);
            const int r = vhalf * (VH / RL) + k;
            unsigned char *dst = row + BITS * (16 * r + RL * vg) / 8;
            if constexpr (RBITS == 8)
                *dst = (unsigned char)w;
            else if constexpr (RBITS == 16)
                *reinterpret_cast<uint16_t *>(dst) = (uint16_t)w;
            else
                *reinterpret_cast<uint32_t *>(dst) = w;
        }
    }
}

template <int BITS, int G, int MF>
__global__ void __launch_bounds__(kThreads) quantize_kv_kernel(QuantArgs a)
{
    constexpr int D = kHeadDim;
    using RC = Rec<BITS, G, MF>;
    constexpr int PASSES = G / kRowsPerPass;
    static_assert(G % kRowsPerPass == 0, "G must be a multiple of 16");

    // per-warp (min, max) of each channel pair, fp16 (exact for fp16 inputs)
    __shared__ uint32_t red_mn[kThreads / 32][D / 2];
    __shared__ uint32_t red_mx[kThreads / 32][D / 2];
    __shared__ __align__(16) float sh_s[D];
    __shared__ __align__(16) float sh_z[D];
    __shared__ __align__(16) float sh_r[D];

    const int tid = threadIdx.x;
    const int c8 = tid % kRowThreads;
    const int r = tid / kRowThreads;
    const int warp = tid / 32;
    const int64_t grp = blockIdx.x;
    const int p = blockIdx.y;
    const int b = p / a.Hkv;
    const int h = p % a.Hkv;

    uint4 kraw[PASSES];
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        const int64_t u = grp * G + i * kRowsPerPass + r;
        kraw[i] = load_stream(concat_row(a, a.k_res, a.k_in, p, b, h, u) + c8 * 8);
    }
    // values: two threads per (token, channel group) -- G tokens x D/G
    // groups x 2 = 2D = 256 items -- each holding half of the group's G
    // channels; the pair sits in adjacent lanes
    constexpr int VG = D / G, VH = G / 2;
    static_assert(2 * D == kThreads, "two threads per value group");
    const int vhalf = tid & 1, vt = (tid >> 1) / VG, vg = (tid >> 1) % VG;
    uint4 vraw[VH / 8];
    {
        const int64_t u = grp * G + vt;
        const __half *vp = concat_row(a, a.v_res, a.v_in, p, b, h, u);
#pragma unroll
        for (int e = 0; e < VH / 8; ++e)
            vraw[e] = load_stream(vp + vg * G + vhalf * VH + e * 8);
    }

    // this group's record
    unsigned char *rec = a.hist + ((int64_t)p * (a.cap / G) + a.n_quant / G + grp) * RC::BYTES;

    // ---- keys: per-channel min/max over the G tokens (fp16, exact) --------
    __half2 mn[4], mx[4];
    {
        const uint32_t *w0 = reinterpret_cast<const uint32_t *>(&kraw[0]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mn[k] = mx[k] = as_h2(w0[k]);
#pragma unroll
        for (int i = 1; i < PASSES; ++i) {
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&kraw[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mn[k] = __hmin2(mn[k], as_h2(w[k]));
                mx[k] = __hmax2(mx[k], as_h2(w[k]));
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        mn[k] = __hmin2(mn[k], as_h2(__shfl_xor_sync(0xffffffffu, as_u32(mn[k]), 16)));
        mx[k] = __hmax2(mx[k], as_h2(__shfl_xor_sync(0xffffffffu, as_u32(mx[k]), 16)));
    }
    if ((tid & 16) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            red_mn[warp][c8 * 4 + k] = as_u32(mn[k]);
            red_mx[warp][c8 * 4 + k] = as_u32(mx[k]);
        }
    }
    __syncthreads();
    if (tid < D / 2) {
        __half2 m0 = as_h2(red_mn[0][tid]), m1 = as_h2(red_mx[0][tid]);
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) {
            m0 = __hmin2(m0, as_h2(red_mn[w][tid]));
            m1 = __hmax2(m1, as_h2(red_mx[w][tid]));
        }
        const float2 f0 = __half22float2(m0), f1 = __half22float2(m1);
        float s0, z0, r0, s1, z1, r1;
        quant_params<BITS, MF>(f0.x, f1.x, s0, z0, r0);
        quant_params<BITS, MF>(f0.y, f1.y, s1, z1, r1);
        sh_s[2 * tid] = s0;
        sh_s[2 * tid + 1] = s1;
        sh_z[2 * tid] = z0;
        sh_z[2 * tid + 1] = z1;
        sh_r[2 * tid] = r0;
        sh_r[2 * tid + 1] = r1;
        meta_store<MF>(rec, 2 * tid, s0);
        meta_store<MF>(rec, 2 * tid + 1, s1);
        meta_store<MF>(rec + RC::MW * D, 2 * tid, z0);
        meta_store<MF>(rec + RC::MW * D, 2 * tid + 1, z1);
    }
    // the values need no key parameter: they run while the first D/2
    // threads finish those, before the barrier that publishes them
    // ---- values: per-token groups of G channels, two threads per group -----
    {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(vraw);
        __half2 lo = as_h2(w[0]), hi = lo;
#pragma unroll
        for (int e = 1; e < VH / 2; ++e) {
            lo = __hmin2(lo, as_h2(w[e]));
            hi = __hmax2(hi, as_h2(w[e]));
        }
        // (min, -max) in one register: the pair reduces with a single hmin2
        __half2 mm = __halves2half2(__hmin(__low2half(lo), __high2half(lo)),
                                    __hneg(__hmax(__low2half(hi), __high2half(hi))));
        mm = __hmin2(mm, as_h2(__shfl_xor_sync(0xffffffffu, as_u32(mm), 1)));
        const float2 f = __half22float2(mm);
        float s, z, rr;
        quant_params<BITS, MF>(f.x, -f.y, s, z, rr);
        const __half2 *hx = reinterpret_cast<const __half2 *>(vraw);
        uint32_t packed[VH / 8];
#pragma unroll
        for (int e = 0; e < VH / 8; ++e) {
            float2 code[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                code[k] = encode2<BITS>(__half22float2(hx[4 * e + k]), make_float2(-s, -s),
                                        make_float2(z, z), make_float2(rr, rr));
            packed[e] = pack8x2<BITS>(code);
        }
        store_value_row<BITS, G>(rec + RC::row(vt, RC::VC, RC::RB), packed, vg, vhalf);
        if (vhalf == 0) {
            meta_store<MF>(rec + RC::row(vt, RC::VS, RC::MW * VG), vg, s);
            meta_store<MF>(rec + RC::row(vt, RC::VZ, RC::MW * VG), vg, z);
        }
    }

    __syncthreads();

    float ks8[8], kz8[8], kr8[8];   // ks8 holds -s: the encode takes the negated scale
    {
        const float4 *S4 = reinterpret_cast<const float4 *>(sh_s + c8 * 8);
        const float4 *Z4 = reinterpret_cast<const float4 *>(sh_z + c8 * 8);
        const float4 *R4 = reinterpret_cast<const float4 *>(sh_r + c8 * 8);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const float4 s4 = S4[v], z4 = Z4[v], r4 = R4[v];
            ks8[4 * v + 0] = -s4.x; ks8[4 * v + 1] = -s4.y; ks8[4 * v + 2] = -s4.z; ks8[4 * v + 3] = -s4.w;
            kz8[4 * v + 0] = z4.x; kz8[4 * v + 1] = z4.y; kz8[4 * v + 2] = z4.z; kz8[4 * v + 3] = z4.w;
            kr8[4 * v + 0] = r4.x; kr8[4 * v + 1] = r4.y; kr8[4 * v + 2] = r4.z; kr8[4 * v + 3] = r4.w;
        }
    }
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        const __half2 *hx = reinterpret_cast<const __half2 *>(&kraw[i]);
        float2 code[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            code[k] = encode2<BITS>(__half22float2(hx[k]), make_float2(ks8[2 * k], ks8[2 * k + 1]),
                                    make_float2(kz8[2 * k], kz8[2 * k + 1]),
                                    make_float2(kr8[2 * k], kr8[2 * k + 1]));
        const uint32_t packed = pack8x2<BITS>(code);
        unsigned char *krow = rec + RC::row(i * kRowsPerPass + r, RC::KC, RC::RB);
        if (BITS == 2)
            reinterpret_cast<uint16_t *>(krow)[c8] = (uint16_t)packed;
        else
            reinterpret_cast<uint32_t *>(krow)[c8] = packed;
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
    case 16: quantize_kv_kernel<BITS, 16, MF><<<grid, kThreads, 0, s>>>(a); break;
    case 32: quantize_kv_kernel<BITS, 32, MF><<<grid, kThreads, 0, s>>>(a); break;
    case 64: quantize_kv_kernel<BITS, 64, MF><<<grid, kThreads, 0, s>>>(a); break;
    case 128: quantize_kv_kernel<BITS, 128, MF><<<grid, kThreads, 0, s>>>(a); break;
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
