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
// pair, keys and values together.  Each token row (128 fp16 = 256 B) is read
// by 16 threads with 16-byte loads, so a warp reads two full rows per
// instruction.  The per-channel key reduction runs across the token axis:
// lanes xor 16 first, then the eight warps through shared memory.  The
// per-token value reduction runs across the G/8 lanes that hold one channel
// group.  All work is HBM-bound: 512 B read and 64-128 B written per token.
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

__device__ __forceinline__ void unpack8(const uint4 &raw, float (&x)[8])
{
    const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

template <int BITS>
__device__ __forceinline__ void quant_params(float mn, float mx, float &s, float &z)
{
    constexpr float kQmax = float((1 << BITS) - 1);
    float scale = __fdiv_rn(__fsub_rn(mx, mn), kQmax);
    if (scale < 1e-8f)
        scale = 1e-8f;
    float zero = rintf(__fdiv_rn(-mn, scale));
    if (zero == 0.0f)
        zero = 0.0f;    // a zero zero-point is stored as +0
    s = scale;
    z = zero;
}

// clamp(rint(x / s) + z, 0, qmax).  rint(x/s) and z are integer-valued
// floats; their fp32 sum is exact whenever it lies inside the code range and
// rounds monotonically otherwise, so clamping it equals clamping the exact
// integer sum.
template <int BITS>
__device__ __forceinline__ uint32_t encode(float x, float s, float z)
{
    constexpr float kQmax = float((1 << BITS) - 1);
    float q = __fadd_rn(rintf(__fdiv_rn(x, s)), z);
    q = fminf(fmaxf(q, 0.0f), kQmax);
    return static_cast<uint32_t>(q);
}

template <int BITS, int G>
__global__ void __launch_bounds__(kThreads) quantize_kv_kernel(QuantArgs a)
{
    constexpr int D = kHeadDim;
    constexpr int PASSES = G / kRowsPerPass;
    constexpr int VLANES = G / 8;                     // lanes holding one value group
    static_assert(G % kRowsPerPass == 0, "G must be a multiple of 16");

    __shared__ float red_mn[kThreads / 32][D];
    __shared__ float red_mx[kThreads / 32][D];
    __shared__ float sh_s[D];
    __shared__ float sh_z[D];

    const int tid = threadIdx.x;
    const int c8 = tid % kRowThreads;
    const int r = tid / kRowThreads;
    const int warp = tid / 32;
    const int64_t grp = blockIdx.x;
    const int p = blockIdx.y;
    const int b = p / a.Hkv;
    const int h = p % a.Hkv;

    uint4 kraw[PASSES], vraw[PASSES];
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        const int64_t u = grp * G + i * kRowsPerPass + r;
        const __half *kp, *vp;
        if (u < a.n_old) {
            const int64_t off = ((int64_t)p * a.R + u) * D;
            kp = a.k_res + off;
            vp = a.v_res + off;
        } else {
            const int64_t off = b * a.in_sb + h * a.in_sh + (u - a.n_old) * a.in_st;
            kp = a.k_in + off;
            vp = a.v_in + off;
        }
        kraw[i] = load_stream(kp + c8 * 8);
        vraw[i] = load_stream(vp + c8 * 8);
    }

    const int64_t row0 = (int64_t)p * a.cap + a.n_quant + grp * G;  // first code row

    // ---- keys: per-channel min/max over the G tokens ----------------------
    float mn[8], mx[8];
    {
        float x[8];
        unpack8(kraw[0], x);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            mn[k] = mx[k] = x[k];
#pragma unroll
        for (int i = 1; i < PASSES; ++i) {
            unpack8(kraw[i], x);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                mn[k] = fminf(mn[k], x[k]);
                mx[k] = fmaxf(mx[k], x[k]);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        mn[k] = fminf(mn[k], __shfl_xor_sync(0xffffffffu, mn[k], 16));
        mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 16));
    }
    if ((tid & 16) == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            red_mn[warp][c8 * 8 + k] = mn[k];
            red_mx[warp][c8 * 8 + k] = mx[k];
        }
    }
    __syncthreads();
    if (tid < D) {
        float m0 = red_mn[0][tid], m1 = red_mx[0][tid];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) {
            m0 = fminf(m0, red_mn[w][tid]);
            m1 = fmaxf(m1, red_mx[w][tid]);
        }
        float s, z;
        quant_params<BITS>(m0, m1, s, z);
        sh_s[tid] = s;
        sh_z[tid] = z;
        const int64_t mrow = ((int64_t)p * (a.cap / G) + a.n_quant / G + grp) * D;
        a.ks[mrow + tid] = s;
        a.kz[mrow + tid] = z;
    }
    __syncthreads();

    float ks8[8], kz8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        ks8[k] = sh_s[c8 * 8 + k];
        kz8[k] = sh_z[c8 * 8 + k];
    }
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        float x[8];
        unpack8(kraw[i], x);
        uint32_t packed = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            packed |= encode<BITS>(x[k], ks8[k], kz8[k]) << (k * BITS);
        const int64_t row = row0 + i * kRowsPerPass + r;
        if (BITS == 2)
            reinterpret_cast<uint16_t *>(a.kc + row * (D / 4))[c8] = (uint16_t)packed;
        else
            reinterpret_cast<uint32_t *>(a.kc + row * (D / 2))[c8] = packed;
    }

    // ---- values: per-token groups of G channels ---------------------------
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
        float x[8];
        unpack8(vraw[i], x);
        float m0 = x[0], m1 = x[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) {
            m0 = fminf(m0, x[k]);
            m1 = fmaxf(m1, x[k]);
        }
#pragma unroll
        for (int off = 1; off < VLANES; off <<= 1) {
            m0 = fminf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
        }
        float s, z;
        quant_params<BITS>(m0, m1, s, z);
        uint32_t packed = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            packed |= encode<BITS>(x[k], s, z) << (k * BITS);
        const int64_t row = row0 + i * kRowsPerPass + r;
        if (BITS == 2)
            reinterpret_cast<uint16_t *>(a.vc + row * (D / 4))[c8] = (uint16_t)packed;
        else
            reinterpret_cast<uint32_t *>(a.vc + row * (D / 2))[c8] = packed;
        if (c8 % VLANES == 0) {
            const int64_t m = row * (D / G) + c8 / VLANES;
            a.vs[m] = s;
            a.vz[m] = z;
        }
    }
}

// 16 tokens x 16 chunks of 16 bytes per CTA.
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
    const int64_t dst = ((int64_t)p * a.R + a.dst_slot0 + i) * D + c8 * 8;
    *reinterpret_cast<uint4 *>(a.k_res + dst) = load_stream(a.k_in + src);
    *reinterpret_cast<uint4 *>(a.v_res + dst) = load_stream(a.v_in + src);
}

template <int BITS>
cudaError_t launch_quantize_bits(int G, const QuantArgs &a, int pairs, cudaStream_t s)
{
    dim3 grid((unsigned)(a.nq_new / G), (unsigned)pairs);
    switch (G) {
    case 16: quantize_kv_kernel<BITS, 16><<<grid, kThreads, 0, s>>>(a); break;
    case 32: quantize_kv_kernel<BITS, 32><<<grid, kThreads, 0, s>>>(a); break;
    case 64: quantize_kv_kernel<BITS, 64><<<grid, kThreads, 0, s>>>(a); break;
    case 128: quantize_kv_kernel<BITS, 128><<<grid, kThreads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(int bits, int G, const QuantArgs &a, int pairs, cudaStream_t s)
{
    if (bits == 2)
        return launch_quantize_bits<2>(G, a, pairs, s);
    if (bits == 4)
        return launch_quantize_bits<4>(G, a, pairs, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_residual_copy(const ResidArgs &a, int pairs, cudaStream_t s)
{
    dim3 grid((unsigned)((a.ntok + kRowsPerPass - 1) / kRowsPerPass), (unsigned)pairs);
    residual_copy_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kivi
