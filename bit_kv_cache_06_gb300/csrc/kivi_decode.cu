// kivi_decode.cu -- split-K decode attention over the packed KIVI cache.
//
// o = softmax(tau * q K^T) V ("4.4 KV Cache quantization", section 2) for one
// new query per head, over the quantised history followed by the fp16
// residual window, which "takes part in Attention together with the
// already-quantized history" (same page, section 3.2).  Keys are dequantised
// per channel and values per token inside the tile loop, never into a full
// fp16 buffer ("09 -- KV Cache Quantization", "Per-channel vs per-token in the
// actual attention kernel").  Grouped-query attention: the g = Hq / Hkv query
// heads of one kv head are processed together, so each code byte is read
// once per kv head.
//
// Split-K (flash-decoding): blockIdx.x = split, blockIdx.y = (batch, kv-head)
// pair.  Split s covers a contiguous range of 128-token chunks of the
// quantised history; the last split also covers the residual.  Each split
// keeps a running max and sum per query head (scores in the log2 domain,
// q pre-scaled by tau * log2 e) and writes (m, l, unnormalised o) to the
// workspace; decode_combine_kernel merges the splits:
//   M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  o = sum_i 2^(m_i - M) o_i / L.
#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kThreads = 128;      // = kChunk tokens in the key phase, = d channels in the value phase

template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int c)
{
    constexpr int PER_WORD = 32 / BITS;
    return (w[c / PER_WORD] >> ((c % PER_WORD) * BITS)) & ((1u << BITS) - 1u);
}

template <int MAXG>
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Online-softmax update for one tile: sc[i] is this thread's token score for
// query head i (-inf for no token).  Writes p_s[tid][i], updates the running
// (m, l) and returns the rescale factor of the previous accumulators.
template <int MAXG>
__device__ __forceinline__ void softmax_tile(const float (&sc)[MAXG], float (&m_run)[MAXG],
                                             float (&l_run)[MAXG], float (&alpha)[MAXG],
                                             float (*p_s)[MAXG], float (*red)[MAXG])
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        float v = warp_max<MAXG>(sc[i]);
        if (lane == 0)
            red[warp][i] = v;
    }
    __syncthreads();
    float pv[MAXG];
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        float tmax = fmaxf(fmaxf(red[0][i], red[1][i]), fmaxf(red[2][i], red[3][i]));
        float m_new = fmaxf(m_run[i], tmax);
        alpha[i] = exp2f(m_run[i] - m_new);
        pv[i] = exp2f(sc[i] - m_new);
        p_s[tid][i] = pv[i];
        m_run[i] = m_new;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        float v = warp_sum(pv[i]);
        if (lane == 0)
            red[warp][i] = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MAXG; ++i)
        l_run[i] = l_run[i] * alpha[i] + ((red[0][i] + red[1][i]) + (red[2][i] + red[3][i]));
}

// CUDA-core variant: one thread per token for q.k, one thread per channel for p.v.
template <int BITS, int G, int MAXG>
__global__ void __launch_bounds__(kThreads) decode_split_simt(DecodeArgs a)
{
    constexpr int D = kHeadDim;
    constexpr int T = kChunk;
    constexpr int NG = T / G;          // key groups per chunk
    constexpr int RB = D * BITS / 8;   // code bytes per token
    constexpr int VG = D / G;          // value groups per token
    constexpr int WORDS = RB / 4;

    __shared__ float q_s[D][MAXG];
    __shared__ float ks_s[NG][D];
    __shared__ float kz_s[NG][D];
    __shared__ float p_s[T][MAXG];
    __shared__ float vs_s[T][VG];
    __shared__ float vz_s[T][VG];
    __shared__ __align__(16) uint8_t vc_s[T * RB];
    __shared__ float red[kThreads / 32][MAXG];

    const int tid = threadIdx.x;
    const int split = blockIdx.x;
    const int p = blockIdx.y;
    const int b = p / a.Hkv;
    const int h = p % a.Hkv;
    const int Hq = a.Hkv * a.g;
    const int64_t qrow0 = (int64_t)b * Hq + (int64_t)h * a.g;

    for (int idx = tid; idx < MAXG * D; idx += kThreads) {
        const int i = idx / D, c = idx % D;
        q_s[c][i] = (i < a.g) ? __half2float(a.q[(qrow0 + i) * D + c]) * a.scale_log2 : 0.0f;
    }

    const int64_t nchunks = (a.n_quant + T - 1) / T;
    const int64_t t_lo = (int64_t)split * nchunks / a.S * T;
    const int64_t t_hi = min((int64_t)(split + 1) * nchunks / a.S * T, a.n_quant);

    float m_run[MAXG], l_run[MAXG], o[MAXG], alpha[MAXG], sc[MAXG];
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.0f;
        o[i] = 0.0f;
    }

    // ---- quantised history ---------------------------------------------
    for (int64_t t0 = t_lo; t0 < t_hi; t0 += T) {
        const int n = (int)min((int64_t)T, t_hi - t0);   // a multiple of G
        __syncthreads();
        for (int idx = tid; idx < (n / G) * D; idx += kThreads) {
            const int gi = idx / D, c = idx % D;
            const int64_t gm = ((int64_t)p * (a.cap / G) + t0 / G + gi) * D + c;
            ks_s[gi][c] = a.ks[gm];
            kz_s[gi][c] = a.kz[gm];
        }
        for (int idx = tid; idx < n * VG; idx += kThreads) {
            const int64_t gm = ((int64_t)p * a.cap + t0) * VG + idx;
            vs_s[idx / VG][idx % VG] = a.vs[gm];
            vz_s[idx / VG][idx % VG] = a.vz[gm];
        }
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.vc + ((int64_t)p * a.cap + t0) * RB);
            uint4 *dst = reinterpret_cast<uint4 *>(vc_s);
            for (int idx = tid; idx < n * RB / 16; idx += kThreads)
                dst[idx] = src[idx];
        }
        __syncthreads();

        // key phase: thread = token
        if (tid < n) {
            uint32_t w[WORDS];
            const uint4 *src = reinterpret_cast<const uint4 *>(a.kc + ((int64_t)p * a.cap + t0 + tid) * RB);
#pragma unroll
            for (int v4 = 0; v4 < WORDS / 4; ++v4) {
                uint4 x = src[v4];
                w[4 * v4 + 0] = x.x;
                w[4 * v4 + 1] = x.y;
                w[4 * v4 + 2] = x.z;
                w[4 * v4 + 3] = x.w;
            }
            const int gi = tid / G;
            float acc[MAXG];
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                acc[i] = 0.0f;
#pragma unroll 16
            for (int c = 0; c < D; ++c) {
                const float kh = ((float)code_at<BITS>(w, c) - kz_s[gi][c]) * ks_s[gi][c];
#pragma unroll
                for (int i = 0; i < MAXG; ++i)
                    acc[i] = fmaf(q_s[c][i], kh, acc[i]);
            }
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                sc[i] = acc[i];
        } else {
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                sc[i] = -INFINITY;
        }
        softmax_tile<MAXG>(sc, m_run, l_run, alpha, p_s, red);

        // value phase: thread = channel
        const int c = tid;
        const int j = c / G;
        const int byte = c * BITS / 8;
        const int shift = (c % (8 / BITS)) * BITS;
#pragma unroll
        for (int i = 0; i < MAXG; ++i)
            o[i] *= alpha[i];
        for (int t = 0; t < n; ++t) {
            const uint32_t code = (vc_s[t * RB + byte] >> shift) & ((1u << BITS) - 1u);
            const float vh = ((float)code - vz_s[t][j]) * vs_s[t][j];
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                o[i] = fmaf(p_s[t][i], vh, o[i]);
        }
    }

    // ---- fp16 residual window (last split) -----------------------------
    if (split == a.S - 1) {
        for (int t0 = 0; t0 < a.n_resid; t0 += T) {
            const int n = min(T, a.n_resid - t0);
            __syncthreads();
            if (tid < n) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.kr + ((int64_t)p * a.R + t0 + tid) * D);
                float acc[MAXG];
#pragma unroll
                for (int i = 0; i < MAXG; ++i)
                    acc[i] = 0.0f;
#pragma unroll 4
                for (int v4 = 0; v4 < D / 8; ++v4) {
                    uint4 x = src[v4];
                    const __half2 *hh = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(hh[e]);
                        const int c = v4 * 8 + 2 * e;
#pragma unroll
                        for (int i = 0; i < MAXG; ++i) {
                            acc[i] = fmaf(q_s[c][i], f.x, acc[i]);
                            acc[i] = fmaf(q_s[c + 1][i], f.y, acc[i]);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < MAXG; ++i)
                    sc[i] = acc[i];
            } else {
#pragma unroll
                for (int i = 0; i < MAXG; ++i)
                    sc[i] = -INFINITY;
            }
            softmax_tile<MAXG>(sc, m_run, l_run, alpha, p_s, red);
            const int c = tid;
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                o[i] *= alpha[i];
            for (int t = 0; t < n; ++t) {
                const float vh = __half2float(a.vr[((int64_t)p * a.R + t0 + t) * D + c]);
#pragma unroll
                for (int i = 0; i < MAXG; ++i)
                    o[i] = fmaf(p_s[t][i], vh, o[i]);
            }
        }
    }

    // ---- partials ----------------------------------------------------------
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        if (i < a.g) {
            const int64_t row = qrow0 + i;
            a.ws_o[(row * a.S + split) * D + tid] = o[i];
            if (tid == 0) {
                a.ws_m[row * a.S + split] = m_run[i];
                a.ws_l[row * a.S + split] = l_run[i];
            }
        }
    }
}

__global__ void __launch_bounds__(kHeadDim) decode_combine_kernel(CombineArgs a)
{
    constexpr int D = kHeadDim;
    const int64_t row = blockIdx.x;
    const int c = threadIdx.x;
    const float *m = a.ws_m + row * a.S;
    const float *l = a.ws_l + row * a.S;
    float M = -INFINITY;
    for (int s = 0; s < a.S; ++s)
        M = fmaxf(M, m[s]);
    float L = 0.0f, O = 0.0f;
    for (int s = 0; s < a.S; ++s) {
        if (l[s] > 0.0f) {
            const float w = exp2f(m[s] - M);
            L = fmaf(l[s], w, L);
            O = fmaf(w, a.ws_o[(row * a.S + s) * D + c], O);
        }
    }
    a.out[row * D + c] = __float2half_rn(O / L);
}

template <int BITS, int G>
cudaError_t launch_split_bg(const DecodeArgs &a, int pairs, cudaStream_t s)
{
    dim3 grid((unsigned)a.S, (unsigned)pairs);
    if (a.g <= 1)
        decode_split_simt<BITS, G, 1><<<grid, kThreads, 0, s>>>(a);
    else if (a.g <= 2)
        decode_split_simt<BITS, G, 2><<<grid, kThreads, 0, s>>>(a);
    else if (a.g <= 4)
        decode_split_simt<BITS, G, 4><<<grid, kThreads, 0, s>>>(a);
    else
        decode_split_simt<BITS, G, 8><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_split_b(int G, const DecodeArgs &a, int pairs, cudaStream_t s)
{
    switch (G) {
    case 16: return launch_split_bg<BITS, 16>(a, pairs, s);
    case 32: return launch_split_bg<BITS, 32>(a, pairs, s);
    case 64: return launch_split_bg<BITS, 64>(a, pairs, s);
    case 128: return launch_split_bg<BITS, 128>(a, pairs, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_partial(int bits, int G, const DecodeArgs &a, int pairs, cudaStream_t s)
{
    if (bits == 2)
        return launch_split_b<2>(G, a, pairs, s);
    if (bits == 4)
        return launch_split_b<4>(G, a, pairs, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const CombineArgs &a, int rows, cudaStream_t s)
{
    decode_combine_kernel<<<(unsigned)rows, kHeadDim, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kivi
