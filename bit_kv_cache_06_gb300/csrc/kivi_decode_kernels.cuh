// kivi_decode_kernels.cuh -- split-K decode attention over the packed KIVI
// cache: the kernels and their launchers, templated on the code width, the
// group size, the query group and the metadata width.  Included by
// kivi_decode.cu (fp32 scales and zero points) and kivi_decode_f16.cu (fp16),
// so that the two sets of instantiations compile in parallel.
//
// o = softmax(tau * q K^T) V ("4.4 KV Cache quantization", section 2) for one
// new query per head, over the quantised history followed by the fp16
// residual window, which "takes part in Attention together with the
// already-quantized history" (same page, section 3.2).  Keys are dequantised
// per channel and values per token inside the tile loop, never into a full
// fp16 buffer ("09 -- KV Cache Quantization", "Per-channel vs per-token in the
// actual attention kernel").  The g = Hq / Hkv query heads of one kv head are
// processed together, so each code byte is read once per kv head.
//
// Work split (flash-decoding): grid = (S, pairs), one wave.  Block s of a pair
// covers a contiguous range of 128-token chunks of the quantised history and
// writes partial s; block S-1 also covers the fp16 residual (folded into its
// own partial by the tensor-core kernel, which leaves partial S empty; written
// as partial S by the CUDA-core kernel).  A
// partial is (m, l, unnormalised o) per query head -- scores in the log2
// domain, q pre-scaled by tau * log2 e.  The S + 1 partials merge as
//   M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  o = sum_i 2^(m_i - M) o_i / L,
// either in the last block of the pair to finish (combine_if_last) or in
// decode_combine_kernel.
//
// Two history kernels:
//  * decode_split_mma (G = 32, 64, 128): tensor cores (mma.sync m16n8k16 f16,
//    fp32 accumulate).  q.k puts tokens on the mma rows and channels on k;
//    p.v puts channels on the rows and tokens on k.  The per-channel key
//    scale and the per-token value scale are folded into the non-code operand
//    (q*s for keys, p*s for values), so the code operand is exact: each pair
//    of codes is masked out of the packed bytes into the mantissa of an
//    fp16x2 pair of subnormals code * 2^(o - 24) (one AND per pair on the key
//    side; a shift and an AND on the value side, which puts every code at the
//    top of the mantissa because the products of a subnormal are aligned as
//    if it were 2^-14, and o = sum p s code - sum p s z cancels heavily).  The
//    folded key operand is carried as an fp16 hi + lo pair (22 significant
//    bits) scaled by a power of two per key group; with a query group of 4
//    the hi and lo columns fill the n = 8 mma tile, with a group of 8 they are
//    two mma into one accumulator.  Each warp streams its own run of 32-token
//    slices through a private cp.async.bulk pipeline (mbarrier completion,
//    bounded waits), so the main loop has no block-wide barrier.
//  * decode_split_simt: CUDA cores, fp32 throughout (G = 16 and reference).
#pragma once

#include "kivi_internal.cuh"

#include <atomic>
#include <type_traits>

namespace kivi {
namespace {

constexpr int kThreads = 128;
constexpr long long kWaitLimitCycles = 1ll << 32;   // about 2 s at 2 GHz
constexpr unsigned kStatusWaitTimeout = 1u;

// ------------------------------------------------------------ reductions ---

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

// Write one partial (m, l, o) for query row `row`; partials are [row][S+1].
__device__ __forceinline__ void store_partial(const DecodeArgs &a, int64_t row, int part, float m,
                                              float l, float o, int c)
{
    const int64_t idx = row * (a.S + 1) + part;
    a.ws_o[idx * kHeadDim + c] = o;
    if (c == 0) {
        a.ws_m[idx] = m;
        a.ws_l[idx] = l;
    }
}

// Merge the S1 partials of query row `row` into out for NC consecutive
// channels from c0:  M = max m_i, L = sum l_i 2^(m_i - M),
// o = sum 2^(m_i - M) o_i / L over the partials with l_i > 0.  The partials
// are read in batches of eight with no load depending on another (one L2
// round trip per batch); a running maximum rescales what earlier batches
// summed.  Every channel sees the same arithmetic whatever NC is, so the
// fused and the two-launch merges agree bit for bit.
template <int NC>
__device__ __forceinline__ void merge_row(const float *ws_m, const float *ws_l, const float *ws_o,
                                          __half *out, int64_t row, int S1, int c0)
{
    constexpr int D = kHeadDim, NB = 8;
    static_assert(NC == 1 || NC == 4 || NC == 8, "one channel, or one or two float4 of them");
    using Vec = typename std::conditional<NC == 1, float, float4>::type;
    constexpr int VW = NC == 1 ? 1 : 4;          // floats per vector
    constexpr int NV = NC / VW;                  // vectors per partial
    const float *mr = ws_m + row * S1, *lr = ws_l + row * S1;
    const Vec *orow = reinterpret_cast<const Vec *>(ws_o + row * S1 * D + c0);
    float M = -INFINITY, L = 0.0f;
    float O[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k)
        O[k] = 0.0f;
    struct Batch {
        float mm[NB], ll[NB], oo[NB][NC];
    };
    auto load = [&](Batch &b, int s0) {
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const bool in = s0 + u < S1;
            b.mm[u] = in ? __ldcg(mr + s0 + u) : -INFINITY;
            b.ll[u] = in ? __ldcg(lr + s0 + u) : 0.0f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                Vec x;
                if (in)
                    x = __ldcg(orow + (int64_t)(s0 + u) * (D / VW) + v);
                else
                    x = Vec{};
                const float *xf = reinterpret_cast<const float *>(&x);
#pragma unroll
                for (int k = 0; k < VW; ++k)
                    b.oo[u][v * VW + k] = xf[k];
            }
        }
    };
    auto fold = [&](const Batch &b) {
        float bm = M;
#pragma unroll
        for (int u = 0; u < NB; ++u)
            if (b.ll[u] > 0.0f)
                bm = fmaxf(bm, b.mm[u]);
        if (bm == -INFINITY)
            return;                             // nothing summed so far
        const float r = exp2f(M - bm);          // 0 until something was summed
        L *= r;
#pragma unroll
        for (int k = 0; k < NC; ++k)
            O[k] *= r;
        M = bm;
#pragma unroll
        for (int u = 0; u < NB; ++u)
            if (b.ll[u] > 0.0f) {
                const float w = exp2f(b.mm[u] - M);
                L = fmaf(b.ll[u], w, L);
#pragma unroll
                for (int k = 0; k < NC; ++k)
                    O[k] = fmaf(w, b.oo[u][k], O[k]);
            }
    };
    for (int s0 = 0; s0 < S1; s0 += NB) {
        Batch b;
        load(b, s0);
        fold(b);
    }
#pragma unroll
    for (int k = 0; k < NC; ++k)
        out[row * D + c0 + k] = __float2half_rn(O[k] / L);
}

// Pull the fp16 rows (sink and residual) of pair p into L2 at the start of
// the block that owns them; the block reads them only after its share of the
// history.
__device__ __forceinline__ void prefetch_rows(const DecodeArgs &a, int p, int row0, int n)
{
    if (n <= 0)
        return;
    const uint32_t bytes = (uint32_t)n * kHeadDim * 2;
    const int64_t off = ((int64_t)p * a.rows + row0) * kHeadDim;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.kr + off), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.vr + off), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_residual(const DecodeArgs &a, int p)
{
    const int nr = a.n_fp16 - a.n_sink;                 // residual tokens in the ring
    const int run = min(nr, a.R - a.head);              // up to the end of the ring
    if (a.head == 0 && a.n_sink == a.Ns) {
        prefetch_rows(a, p, 0, a.n_fp16);               // one contiguous run of rows
        return;
    }
    prefetch_rows(a, p, 0, a.n_sink);
    prefetch_rows(a, p, a.Ns + a.head, run);
    prefetch_rows(a, p, a.Ns, nr - run);
}

// Fused combine: when a.out is set, every block of pair p takes a ticket
// after writing its partials; the block that takes the last one merges the
// pair's S + 1 partials into out and re-arms the counter for the next call.
// No block ever waits for another (the classic threadfence reduction).
// FAST (the tensor-core kernel of query group 8) merges the heads of a
// group larger than four in half-warps at once; otherwise one warp per head
// (fewer registers).  Both give the same bits.
template <bool FAST>
__device__ void combine_if_last(const DecodeArgs &a, int p, int *s_last)
{
    if (a.out == nullptr)
        return;
    __syncthreads();                       // all partial stores of this block issued
    if (threadIdx.x == 0) {
        __threadfence();
        *s_last = atomicAdd(a.counters + p, 1u) == (unsigned)a.S - 1u;
    }
    __syncthreads();
    if (!*s_last)
        return;
    __threadfence();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = p / a.Hkv, h = p % a.Hkv;
    const int64_t qrow0 = (int64_t)b * a.Hkv * a.g + (int64_t)h * a.g;
    static_assert(kThreads == 128, "four warps merge up to eight query heads");
    if (!FAST || a.g <= kThreads / 32) {
        // one warp per query head, four channels per lane
        for (int hh = warp; hh < a.g; hh += kThreads / 32)
            merge_row<4>(a.ws_m, a.ws_l, a.ws_o, a.out, qrow0 + hh, a.S + 1, 4 * lane);
    } else {
        // more heads than warps: one half-warp per query head, eight
        // channels per lane, so every head is merged at once instead of
        // two after one another
        const int hh = 2 * warp + (lane >> 4);
        if (hh < a.g)
            merge_row<8>(a.ws_m, a.ws_l, a.ws_o, a.out, qrow0 + hh, a.S + 1, 8 * (lane & 15));
    }
    if (threadIdx.x == 0)
        a.counters[p] = 0u;
}

// ================================================================ SIMT =====
// One thread per token for q.k, one thread per channel for p.v, block-wide
// online softmax.  Shared state lives in a caller-provided buffer.

template <int MAXG>
struct SimtSmem {
    float q[kHeadDim][MAXG];
    float p[kChunk][MAXG];
    float red[kThreads / 32][MAXG];
};

// Online-softmax update for one tile: sc[i] is this thread's token score for
// query head i (-inf for no token).  Writes p[tid][i], updates the running
// (m, l) and returns the rescale factor of the previous accumulators.
template <int MAXG>
__device__ __forceinline__ void softmax_tile(const float (&sc)[MAXG], float (&m_run)[MAXG],
                                             float (&l_run)[MAXG], float (&alpha)[MAXG],
                                             SimtSmem<MAXG> &sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        float v = warp_max(sc[i]);
        if (lane == 0)
            sm.red[warp][i] = v;
    }
    __syncthreads();
    float pv[MAXG];
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        float tmax = fmaxf(fmaxf(sm.red[0][i], sm.red[1][i]), fmaxf(sm.red[2][i], sm.red[3][i]));
        float m_new = fmaxf(m_run[i], tmax);
        alpha[i] = exp2f(m_run[i] - m_new);
        pv[i] = exp2f(sc[i] - m_new);
        sm.p[tid][i] = pv[i];
        m_run[i] = m_new;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        float v = warp_sum(pv[i]);
        if (lane == 0)
            sm.red[warp][i] = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < MAXG; ++i)
        l_run[i] = l_run[i] * alpha[i] + ((sm.red[0][i] + sm.red[1][i]) + (sm.red[2][i] + sm.red[3][i]));
}

template <int MAXG>
__device__ __forceinline__ void simt_load_q(const DecodeArgs &a, int64_t qrow0, SimtSmem<MAXG> &sm)
{
    for (int idx = threadIdx.x; idx < MAXG * kHeadDim; idx += kThreads) {
        const int i = idx / kHeadDim, c = idx % kHeadDim;
        sm.q[c][i] = (i < a.g) ? __half2float(a.q[(qrow0 + i) * kHeadDim + c]) * a.scale_log2 : 0.0f;
    }
}

// The fp16 rows (sink and residual window) of pair p as partial number a.S.
template <int MAXG>
__device__ void residual_partial(const DecodeArgs &a, int p, SimtSmem<MAXG> &sm)
{
    constexpr int D = kHeadDim;
    constexpr int T = kChunk;
    const int tid = threadIdx.x;
    const int b = p / a.Hkv, h = p % a.Hkv;
    const int64_t qrow0 = (int64_t)b * a.Hkv * a.g + (int64_t)h * a.g;
    simt_load_q<MAXG>(a, qrow0, sm);
    float m_run[MAXG], l_run[MAXG], o[MAXG], alpha[MAXG], sc[MAXG];
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.0f;
        o[i] = 0.0f;
    }
    for (int t0 = 0; t0 < a.n_fp16; t0 += T) {
        const int n = min(T, a.n_fp16 - t0);
        __syncthreads();
        if (tid < n) {
            const int row = fp16_row(t0 + tid, a.n_sink, a.Ns, a.R, a.head);
            const uint4 *src = reinterpret_cast<const uint4 *>(a.kr + ((int64_t)p * a.rows + row) * D);
            float acc[MAXG];
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                acc[i] = 0.0f;
            uint4 xs[D / 8];                    // the whole row in flight at once
#pragma unroll
            for (int v4 = 0; v4 < D / 8; ++v4)
                xs[v4] = src[v4];
#pragma unroll
            for (int v4 = 0; v4 < D / 8; ++v4) {
                const uint4 x = xs[v4];
                const __half2 *hh = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(hh[e]);
                    const int c = v4 * 8 + 2 * e;
#pragma unroll
                    for (int i = 0; i < MAXG; ++i) {
                        acc[i] = fmaf(sm.q[c][i], f.x, acc[i]);
                        acc[i] = fmaf(sm.q[c + 1][i], f.y, acc[i]);
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
        softmax_tile<MAXG>(sc, m_run, l_run, alpha, sm);
        const int c = tid;
#pragma unroll
        for (int i = 0; i < MAXG; ++i)
            o[i] *= alpha[i];
        // value rows in batches of 16 independent loads
        const __half *vcol = a.vr + (int64_t)p * a.rows * D + c;
        for (int tb = 0; tb < n; tb += 16) {
            float vh[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                vh[u] = tb + u < n
                            ? __half2float(vcol[(int64_t)fp16_row(t0 + tb + u, a.n_sink, a.Ns, a.R, a.head) * D])
                            : 0.0f;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (tb + u < n) {
#pragma unroll
                    for (int i = 0; i < MAXG; ++i)
                        o[i] = fmaf(sm.p[tb + u][i], vh[u], o[i]);
                }
        }
    }
#pragma unroll
    for (int i = 0; i < MAXG; ++i)
        if (i < a.g)
            store_partial(a, qrow0 + i, a.S, m_run[i], l_run[i], o[i], tid);
}

template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int c)
{
    constexpr int PER_WORD = 32 / BITS;
    return (w[c / PER_WORD] >> ((c % PER_WORD) * BITS)) & ((1u << BITS) - 1u);
}

template <int BITS, int G, int MAXG>
struct SimtHistSmem {
    static constexpr int NG = kChunk / G, RB = kHeadDim * BITS / 8, VG = kHeadDim / G;
    SimtSmem<MAXG> base;
    float ks[NG][kHeadDim];
    float kz[NG][kHeadDim];
    float vs[kChunk][VG];
    float vz[kChunk][VG];
    __align__(16) uint8_t vc[kChunk * RB];
};

template <int BITS, int G, int MAXG, int MF>
__global__ void __launch_bounds__(kThreads) decode_split_simt(DecodeArgs a)
{
    constexpr int D = kHeadDim;
    constexpr int T = kChunk;
    using SM = SimtHistSmem<BITS, G, MAXG>;
    using RC = Rec<BITS, G, MF>;
    constexpr int RB = SM::RB, VG = SM::VG, WORDS = RB / 4;
    __shared__ SM sm;

    const int tid = threadIdx.x;
    const int split = blockIdx.x;
    const int p = blockIdx.y;
    __shared__ int s_last;
    const int b = p / a.Hkv;
    const int h = p % a.Hkv;
    const int64_t qrow0 = (int64_t)b * a.Hkv * a.g + (int64_t)h * a.g;
    if (split == a.S - 1 && tid == 0)
        prefetch_residual(a, p);
    simt_load_q<MAXG>(a, qrow0, sm.base);

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

    for (int64_t t0 = t_lo; t0 < t_hi; t0 += T) {
        const int n = (int)min((int64_t)T, t_hi - t0);   // a multiple of G
        __syncthreads();
        // this chunk's key-group records
        const uint8_t *recs = a.hist + ((int64_t)p * (a.cap / G) + t0 / G) * RC::BYTES;
        for (int idx = tid; idx < (n / G) * D; idx += kThreads) {
            const int gi = idx / D, c = idx % D;
            sm.ks[gi][c] = meta_load<MF>(recs + gi * RC::BYTES, c);
            sm.kz[gi][c] = meta_load<MF>(recs + gi * RC::BYTES + RC::MW * D, c);
        }
        for (int idx = tid; idx < n * VG; idx += kThreads) {
            const int tt = idx / VG, j = idx % VG;
            const uint8_t *rec = recs + (tt / G) * RC::BYTES;
            sm.vs[tt][j] = meta_load<MF>(rec + RC::row(tt % G, RC::VS, RC::MW * VG), j);
            sm.vz[tt][j] = meta_load<MF>(rec + RC::row(tt % G, RC::VZ, RC::MW * VG), j);
        }
        for (int idx = tid; idx < n * RB / 16; idx += kThreads) {
            const int tt = idx / (RB / 16), v4 = idx % (RB / 16);
            const uint8_t *rec = recs + (tt / G) * RC::BYTES;
            reinterpret_cast<uint4 *>(sm.vc)[idx] =
                reinterpret_cast<const uint4 *>(rec + RC::row(tt % G, RC::VC, RB))[v4];
        }
        __syncthreads();

        // key phase: thread = token
        if (tid < n) {
            uint32_t w[WORDS];
            const uint4 *src = reinterpret_cast<const uint4 *>(
                recs + (tid / G) * RC::BYTES + RC::row(tid % G, RC::KC, RB));
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
#pragma unroll
            for (int c = 0; c < D; ++c) {
                const float kh = ((float)code_at<BITS>(w, c) - sm.kz[gi][c]) * sm.ks[gi][c];
#pragma unroll
                for (int i = 0; i < MAXG; ++i)
                    acc[i] = fmaf(sm.base.q[c][i], kh, acc[i]);
            }
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                sc[i] = acc[i];
        } else {
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                sc[i] = -INFINITY;
        }
        softmax_tile<MAXG>(sc, m_run, l_run, alpha, sm.base);

        // value phase: thread = channel (at its stored position in the row)
        const int c = tid;
        const int j = c / G;
        const int pos = value_pos<BITS, G>(c);
        const int byte = pos * BITS / 8;
        const int shift = (pos % (8 / BITS)) * BITS;
#pragma unroll
        for (int i = 0; i < MAXG; ++i)
            o[i] *= alpha[i];
        for (int t = 0; t < n; ++t) {
            const uint32_t code = (sm.vc[t * RB + byte] >> shift) & ((1u << BITS) - 1u);
            const float vh = ((float)code - sm.vz[t][j]) * sm.vs[t][j];
#pragma unroll
            for (int i = 0; i < MAXG; ++i)
                o[i] = fmaf(sm.base.p[t][i], vh, o[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < MAXG; ++i)
        if (i < a.g)
            store_partial(a, qrow0 + i, split, m_run[i], l_run[i], o[i], tid);
    if (split == a.S - 1) {                // the last split also owns the residual window
        __syncthreads();
        residual_partial<MAXG>(a, p, sm.base);
    }
    combine_if_last<false>(a, p, &s_last);
}

// ================================================================ MMA ======

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(phase)
                 : "memory");
    return ok != 0;
}

// Bounded wait: false if the phase did not complete within kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase)
{
    if (mbar_try_wait(bar, phase))
        return true;
    const long long start = clock64();
    while (!mbar_try_wait(bar, phase))
        if (clock64() - start > kWaitLimitCycles)
            return false;
    return true;
}

// Barrier arm and 1-D bulk copy global -> shared (completing on an mbarrier,
// with an L2 cache policy for the source lines), predicated: every lane
// executes them, only lanes with pred set act, so the issuing code needs no
// branch.
__device__ __forceinline__ void mbar_expect_tx_if(bool pred, uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t"
                 "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}"
                 ::"r"(bar), "r"(bytes), "r"((uint32_t)pred) : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint_if(bool pred, uint32_t dst, const void *src, uint32_t bytes,
                                                 uint32_t bar, uint64_t policy)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %5, 0;\n\t"
                 "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;\n\t}"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy), "r"((uint32_t)pred)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_if(bool pred)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t@p fence.proxy.async.shared::cta;\n\t}"
                 ::"r"((uint32_t)pred) : "memory");
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Offset o at which a code taken from bit `pos` of a 16-bit half lands in the
// fp16 mantissa: the field must stay below bit 10, so fields that start
// higher are first moved down by 8 bits.
__host__ __device__ constexpr int code_o(int pos, int bits) { return pos + bits <= 10 ? pos : pos - 8; }

// Key-side code pair: (code_lo, code_hi) from bits [pos, pos + BITS) of each
// 16-bit half of x, as an fp16x2 pair of exact subnormals code * 2^(o - 24)
// with o = code_o(pos, BITS): with the exponent field zero the masked mantissa
// bits are the value, and the other operand carries 2^-o.  Fields above bit 9
// come from xs (x with the two bytes of each half swapped, one prmt per word)
// instead of a shift of x.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair_k(uint32_t x, uint32_t xs, int pos)
{
    if (pos + BITS <= 10)
        return x & ((((1u << BITS) - 1u) << pos) * 0x00010001u);
    return xs & ((((1u << BITS) - 1u) << (pos - 8)) * 0x00010001u);
}

// 2^x rounded by the hardware approximation (subnormal results flush to 0).
__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Mantissa offset of the value-side code operand: the top of the subnormal
// mantissa (bits 8-9 for 2-bit codes, 6-9 for 4-bit codes).
template <int BITS>
constexpr int kCodeTop = 10 - BITS;

// Value-side code pair: as code_pair_k, but always at offset kCodeTop,
// code * 2^(kCodeTop - 24), undone by the output scale.
// The tensor core aligns the products of an mma on the operands' exponent
// fields, and a subnormal counts as 2^-14 whatever its leading zeros; a code
// low in the mantissa therefore loses up to 10 bits of its product with the
// other operand.  At the top it loses at most BITS - 1 of them.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair_top(uint32_t x, int pos)
{
    constexpr int OT = kCodeTop<BITS>;
    const uint32_t x2 = pos <= OT ? x << (OT - pos) : x >> (pos - OT);
    return x2 & ((((1u << BITS) - 1u) << OT) * 0x00010001u);
}

// fp16x2 {lo half: x0, hi half: x1}, rounded to nearest.
__device__ __forceinline__ uint32_t pack_f16(float x0, float x1)
{
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(x1), "f"(x0));
    return d;
}

// x = hi + lo with hi = x truncated to 11 significant bits (exact in fp16 in
// its normal range) and lo the remainder rounded to fp16: 22 bits together.
__device__ __forceinline__ float trunc11(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// Token order inside a 16-token k-tile: mma row/k index m holds token tau(m).
// Chosen so that the shared-memory code loads of both operands are free of
// bank conflicts (key rows r, r + 8 at 8-byte offsets; value rows 2t, 2t + 1,
// 2t + 8, 2t + 9 at 4-byte offsets).
__device__ __forceinline__ int tau(int m) { return m ^ ((m >> 2) & 1); }

// x >> 8 on the multiply pipe: moves the fields above bit 9 of each 16-bit
// half down by eight bits (the high half's low byte enters the low half's
// bits 8-15, where no mask below bit 8 reaches).
__device__ __forceinline__ uint32_t down8(uint32_t x) { return __umulhi(x, 1u << 24); }

// Two fp8 values (low byte first) widened to an fp16x2 pair (exact: every
// E4M3 and E5M2 value is an fp16 value).
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint16_t x)
{
    uint32_t d;
    if constexpr (FMT == KIVI_FP8_E5M2)
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(d) : "h"(x));
    else
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(x));
    return d;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t x, __half2 f)
{
    __half2 h = __hmul2(*reinterpret_cast<const __half2 *>(&x), f);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int BITS, int G, int GQ, int MF, int F8 = 0>
struct MmaCfg {
    using RC = Rec<BITS, G, MF>;
    static constexpr int D = kHeadDim;
    static constexpr int W = 32;                     // tokens per warp slice
    static constexpr int RB = RC::RB;                // code bytes per token
    static constexpr int VG = RC::VG;                // value groups per token
    static constexpr int MT = G / 16;                // value m-tiles per group
    static constexpr int UG = G / W;                 // slices per key group
    static constexpr int CH = 2 * BITS;              // value-code bytes per lane per token
    // A stage holds one 32-token sub-slice of a record; the first one of a
    // group also carries the group's key scales and zero points (META bytes
    // in front).  Copies of the other sub-slices land behind META.
    static constexpr int STAGE = RC::META + RC::SUB;
    static constexpr int BSTEP = 2 * 128 + 16;       // one k-step of B: two 8x8 fp16 tiles + pad
    static constexpr int NSET = GQ == 4 ? 1 : 2;     // hi/lo interleaved in one set, or two sets
    static constexpr int BWARP = NSET * 8 * BSTEP;
    // FP8 mode: the stages hold raw fp8 tiles in flight (16 key rows, then 16
    // value rows), so the widened fp16 tile has a region of its own behind
    // the barriers, followed by a second query operand in the channel order
    // of the FP8 key fragments
    static constexpr int TST_TILE = 16 * (2 * D + 16);   // one staged 16-row fp16 tile
    static constexpr int per_warp_base(int stages) { return (stages * STAGE + BWARP + stages * 8 + 127) / 128 * 128; }
    // Packed history: the fp16 tiles run before the history when a staging
    // region of their own still leaves three blocks per SM (their loads then
    // overlap the first history copy instead of ending the block's work);
    // otherwise after it, staged in the idle stage buffer.
    static constexpr bool TILES_FIRST =
        !F8 && GQ == 4 && 3 * ((kThreads / 32) * (per_warp_base(2) + TST_TILE) + 1024) <= 233472;
    static constexpr int TST = F8 ? TST_TILE + BWARP : (TILES_FIRST ? TST_TILE : 0);
    static constexpr int per_warp(int stages) { return per_warp_base(stages) + TST; }
    static constexpr int STAGES = 2;
    static constexpr int PER_WARP = per_warp(STAGES);
    static constexpr int NWARP = kThreads / 32;
    static constexpr int SMEM = NWARP * PER_WARP;
    static constexpr int TSTOFF = PER_WARP - TST;    // the FP8 mode's fp16 tile
    static constexpr int NH = GQ / 4;                // query heads owned per thread
    static_assert(G >= W && RC::SL == W, "tensor-core kernel: key groups of 32+ tokens");
    static_assert(STAGE % 16 == 0 && RC::SUB % 16 == 0 && RC::META % 16 == 0 &&
                      BWARP % 16 == 0 && PER_WARP % 128 == 0,
                  "stage layout must keep 16-byte alignment");
};

// History split: the block's token range is cut into key groups and each
// warp runs its own contiguous run of groups, one 32-token sub-slice at a
// time, through a private STAGES-deep cp.async.bulk pipeline (one copy per
// sub-slice: the records keep a sub-slice's codes and metadata together), so
// the main loop has no block-wide barrier.
// F8 = KIVI_FP8_E4M3 / KIVI_FP8_E5M2: the FP8 KV history instead of packed
// codes -- each warp takes 16-token tiles of the block's range, converts the
// fp8 rows to fp16 while staging them and runs them through the same tile
// path as the fp16 rows (BITS, G only size the per-warp buffers then).
template <int BITS, int G, int GQ, int MF, int F8 = 0>
__global__ void __launch_bounds__(kThreads, 3) decode_split_mma(DecodeArgs a)
{
    using C = MmaCfg<BITS, G, GQ, MF, F8>;
    using RC = typename C::RC;
    constexpr int D = C::D, RB = C::RB, VG = C::VG, MT = C::MT, NH = C::NH;
    constexpr int UG = C::UG, CH = C::CH;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, t = lane & 3;
    const int split = blockIdx.x;
    const int p = blockIdx.y;
    __shared__ int s_last;
    __shared__ int s_failed;          // a warp's bounded wait gave up
    const int b = p / a.Hkv, h = p % a.Hkv;
    const int64_t qrow0 = (int64_t)b * a.Hkv * a.g + (int64_t)h * a.g;
    if (tid == 0)
        s_failed = 0;
    if (split == a.S - 1 && tid == 0)
        prefetch_residual(a, p);
    __syncthreads();                  // s_failed is cleared before any wait can set it

    // this block's 128-token chunks, as key groups; then this warp's run
    const int64_t nchunks = (a.n_quant + kChunk - 1) / kChunk;
    const int64_t c0 = (int64_t)split * nchunks / a.S, c1 = (int64_t)(split + 1) * nchunks / a.S;
    const int64_t g0 = c0 * (kChunk / G);
    const int64_t g1 = min(c1 * (kChunk / G), a.n_quant / G);
    const int64_t ng = g1 > g0 ? g1 - g0 : 0;
    const int64_t wg0 = g0 + ng * warp / C::NWARP;
    const int nw = F8 ? 0 : (int)((g0 + ng * (warp + 1) / C::NWARP - wg0) * UG);   // sub-slices
    const uint8_t *wrec = a.hist + ((int64_t)p * (a.cap / G) + wg0) * RC::BYTES;

    unsigned char *wbase = smem + warp * C::PER_WARP;
    unsigned char *bbuf = wbase + C::STAGES * C::STAGE;
    const uint32_t wbase_s = smem_u32(wbase);
    const uint32_t bbuf_s = smem_u32(bbuf);
    const uint32_t bar0 = wbase_s + C::STAGES * C::STAGE + C::BWARP;
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s)
            mbar_init(bar0 + 8 * s, 1);
        fence_proxy_async();
    }
    __syncwarp();

    // The history is read once: its copies may leave L2 first.
    uint64_t stream_policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream_policy));

    // Fill stage i % STAGES with sub-slice i of this warp's run: one copy and
    // one barrier, issued by lane 0 when go is set (every lane computes the
    // operands).  Sub-slice 0 of a group brings the group's Ks, Kz along.
    // `extra` bytes are expected on top of the copy (the failure-path test
    // hook; 0 otherwise).
    auto issue = [&](int i, bool go, uint32_t extra) {
        const int stage = i % C::STAGES;
        const int sub = UG == 1 ? 0 : i % UG;
        const uint32_t bytes = sub == 0 ? RC::META + RC::SUB : RC::SUB;
        const uint32_t bar = bar0 + 8 * stage;
        const uint32_t dst = wbase_s + stage * C::STAGE + (sub == 0 ? 0 : RC::META);
        const uint8_t *src = wrec + (int64_t)(i / UG) * RC::BYTES + (sub == 0 ? 0 : RC::META + sub * RC::SUB);
        mbar_expect_tx_if(go, bar, bytes + extra);
        bulk_g2s_hint_if(go, dst, src, bytes, bar, stream_policy);
    };
    const bool poison = a.poison_first_copy && warp == 0 && split == 0 && p == 0;
    // Key B operand: this lane builds the entries of k-step bs, k positions
    // 2bq, 2bq+1, 2bq+8, 2bq+9 (channels ch[0..3]) for every column.
    const int bq = lane >> 3, bs = lane & 7;
    int ch[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        ch[i] = (BITS == 2) ? 32 * bq + 8 * i + bs : 32 * bq + 16 * (bs >> 2) + (bs & 3) + 4 * i;
    // The query loads go out before the first history copies: issued after
    // them, they queued behind the whole grid's first burst of copies
    // (measured: the query arrived 3.6 us after the start on the 8B layer).
    __half qh[GQ][4];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            qh[hh][i] = (hh < a.g) ? a.q[(qrow0 + hh) * D + ch[i]] : __float2half(0.0f);
    // Only the first sub-slice at the start: the later stages are filled once
    // it has landed, which halves the grid's first burst of copies and with
    // it the wait for the first data.
    if (nw > 0)
        issue(0, lane == 0, poison ? 16u : 0u);

    const int o_k = code_o((BITS == 2) ? 2 * bs : 4 * (bs & 3), BITS);
    // q * tau * log2(e) * 2^-o_k: the code operand of this k-step carries 2^o_k
    float qreg[GQ][4];
    float qmax = 0.0f;
    const float f_o = exp2i(-o_k);
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float qv = __half2float(qh[hh][i]) * a.scale_log2;
            qmax = fmaxf(qmax, fabsf(qv));
            qreg[hh][i] = qv * f_o;
        }
    qmax = warp_max(qmax);

    // value accumulators, fp32 pairs: query group 4 keeps (row r, row r + 8)
    // of head t; query group 8 keeps (heads 2t, 2t + 1) of row r and of row
    // r + 8
    constexpr int NO = GQ == 4 ? 1 : 2;
    float2 o_acc[8][NO];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < NO; ++k)
            o_acc[i][k] = make_float2(0.0f, 0.0f);
    float m_run[NH], l_part[NH], zacc[VG][NH], zq[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        m_run[j] = -INFINITY;
        l_part[j] = 0.0f;
        zq[j] = 0.0f;
#pragma unroll
        for (int v = 0; v < VG; ++v)
            zacc[v][j] = 0.0f;
    }
    // Online softmax over one slice's scores (log2 domain, [k-tile][row r /
    // r + 8][head slot]): running max, p = 2^(score - max), running sum, and
    // the history accumulators rescaled by alpha = 2^(old max - new max).  The
    // rescale is unconditional (alpha = 1 when no maximum moved): a few packed
    // multiplies on the lightly used FMA pipe cost less than the vote and the
    // branch that would skip them.
    auto softmax_step = [&](const float (&sc)[2][2][NH], float (&pr)[2][2][NH], float (&alpha)[NH]) {
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            float mx = fmaxf(fmaxf(sc[0][0][j], sc[0][1][j]), fmaxf(sc[1][0][j], sc[1][1][j]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[j], mx);
            alpha[j] = ex2_ftz(m_run[j] - m_new);
            m_run[j] = m_new;
            float sum = 0.0f;
#pragma unroll
            for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    pr[kt][rr][j] = ex2_ftz(sc[kt][rr][j] - m_new);
                    sum += pr[kt][rr][j];
                }
            l_part[j] = fmaf(l_part[j], alpha[j], sum);
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const float2 al = make_float2(alpha[0], alpha[NH - 1]);
#pragma unroll
            for (int k = 0; k < NO; ++k)
                o_acc[mt][k] = __fmul2_rn(o_acc[mt][k], al);
        }
#pragma unroll
        for (int v = 0; v < VG; ++v)
#pragma unroll
            for (int j = 0; j < NH; ++j)
                zacc[v][j] *= alpha[j];
    };

    bool failed = false;

    // ---- the fp16 rows (sink and residual window; last split): 16-token
    // tiles dealt to the warps, through the same online softmax.  Each tile's key rows, then its
    // value rows, are staged in this warp's (now idle) stage buffer; the key
    // tile enters the mma as it is (ldmatrix), the value tile transposed
    // (ldmatrix.trans), against the query alone (no scale, no zero point).
    // Outputs go to ores, in natural channel order.
    constexpr int RT = 16;                              // tokens per residual tile
    constexpr int RS = D * 2 + 16;                      // padded staged row, bytes
    static_assert(F8 ? C::STAGE >= 2 * RT * D && C::TST == RT * RS + C::BWARP
                     : (C::TILES_FIRST ? C::TST == RT * RS : C::STAGES * C::STAGE >= RT * RS),
                  "tile staging");
    float2 ores[8][NO];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < NO; ++k)
            ores[i][k] = make_float2(0.0f, 0.0f);
    int ntile = 0;       // this block's tiles (FP8 history, then fp16 rows)
    auto run_tiles = [&]() {
        // FP8 history tiles of this block (none for packed codes), then the fp16
        // tiles (last split)
        const int64_t h_lo = F8 ? min(c0 * kChunk, a.n_quant) : 0;
        const int nht = F8 ? (int)((min(c1 * kChunk, a.n_quant) - h_lo) / RT) : 0;
        // the pair's fp16 tiles are dealt round-robin to its S blocks (tile
        // split, split + S, ...), so no block carries them all on the critical path
        const int nft = (a.n_fp16 + RT - 1) / RT;
        const int nmine = failed || split >= nft ? 0 : (nft - split + a.S - 1) / a.S;
        ntile = nht + nmine;
        // FP8 mode: this warp's history tiles (warp, warp + NWARP, ... below nht)
        // stream through its STAGES-deep pipeline, tile j into stage j % STAGES
        // (its 16 key rows, then its 16 value rows: two copies, one barrier)
        const int nhw = F8 && warp < nht ? (nht - warp + C::NWARP - 1) / C::NWARP : 0;
        auto issue_tile = [&](int j, bool go) {
            const int64_t t0 = h_lo + (int64_t)(warp + C::NWARP * j) * RT;
            const uint8_t *src = a.hist + ((int64_t)p * (a.cap / 32) + t0 / 32) * (64 * D) + (t0 % 32) * D;
            const uint32_t dst = wbase_s + (j % C::STAGES) * C::STAGE;
            const uint32_t bar = bar0 + 8 * (j % C::STAGES);
            mbar_expect_tx_if(go, bar, 2 * RT * D);
            bulk_g2s_hint_if(go, dst, src, RT * D, bar, stream_policy);
            bulk_g2s_hint_if(go, dst + RT * D, src + 32 * D, RT * D, bar, stream_policy);
        };
        // bounded wait for tile j; on failure the copies in flight (j .. j +
        // STAGES - 1) get one more bounded wait, as for the packed history
        auto wait_tile = [&](int j) -> bool {
            if (mbar_wait(bar0 + 8 * (j % C::STAGES), (uint32_t)(j / C::STAGES) & 1u))
                return true;
            if (lane == 0) {
                atomicOr(a.status, kStatusWaitTimeout);
                s_failed = 1;
                for (int k2 = j; k2 < nhw && k2 < j + C::STAGES; ++k2)
                    mbar_wait(bar0 + 8 * (k2 % C::STAGES), (uint32_t)(k2 / C::STAGES) & 1u);
            }
            return false;
        };
        if constexpr (F8) {
            for (int j = 0; j < nhw && j < C::STAGES; ++j)
                issue_tile(j, lane == 0);
        }
        if (warp < ntile) {
            // B operand of tau * log2(e) * q * 2^Er: this lane fills k-step bs,
            // k positions 2bq, 2bq+1, 2bq+8, 2bq+9 of channels cn[0..3] -- in
            // natural order (16 bs + k) for the staged fp16 tiles, and for the
            // FP8 key fragments (built from the raw rows, see below) in the order
            // that gives each lane 32 consecutive channels of its rows:
            // k-step s, k = 2t + e -> 32 t + 4 s + e, k = 2t + 8 + e -> 32 t + 4 s + 2 + e
            int Er = 14 - (((__float_as_int(qmax) >> 23) & 0xff) - 127);
            Er = min(max(Er, -100), 100);
            const float kscale_r = exp2i(-Er), fEr = exp2i(Er);
            unsigned char *bbuf8 = wbase + C::TSTOFF + RT * RS;
            const uint32_t bbuf8_s = wbase_s + C::TSTOFF + RT * RS;
    #pragma unroll
            for (int order = 0; order < (F8 ? 2 : 1); ++order) {
                const int cn[4] = {order ? 32 * bq + 4 * bs : 16 * bs + 2 * bq,
                                   order ? 32 * bq + 4 * bs + 1 : 16 * bs + 2 * bq + 1,
                                   order ? 32 * bq + 4 * bs + 2 : 16 * bs + 2 * bq + 8,
                                   order ? 32 * bq + 4 * bs + 3 : 16 * bs + 2 * bq + 9};
    #pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    float v[4], hi[4], lo[4];
    #pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) {
                        v[i2] = (hh < a.g) ? __half2float(a.q[(qrow0 + hh) * D + cn[i2]]) * a.scale_log2 * fEr : 0.0f;
                        hi[i2] = trunc11(v[i2]);
                        lo[i2] = v[i2] - hi[i2];
                    }
                    unsigned char *base = (order ? bbuf8 : bbuf) + bs * C::BSTEP + bq * 4;
                    if constexpr (GQ == 4) {
                        *reinterpret_cast<uint32_t *>(base + (2 * hh) * 16) = pack_f16(hi[0], hi[1]);
                        *reinterpret_cast<uint32_t *>(base + (2 * hh + 1) * 16) = pack_f16(lo[0], lo[1]);
                        *reinterpret_cast<uint32_t *>(base + 128 + (2 * hh) * 16) = pack_f16(hi[2], hi[3]);
                        *reinterpret_cast<uint32_t *>(base + 128 + (2 * hh + 1) * 16) = pack_f16(lo[2], lo[3]);
                    } else {
                        *reinterpret_cast<uint32_t *>(base + hh * 16) = pack_f16(hi[0], hi[1]);
                        *reinterpret_cast<uint32_t *>(base + 128 + hh * 16) = pack_f16(hi[2], hi[3]);
                        *reinterpret_cast<uint32_t *>(base + 8 * C::BSTEP + hh * 16) = pack_f16(lo[0], lo[1]);
                        *reinterpret_cast<uint32_t *>(base + 8 * C::BSTEP + 128 + hh * 16) = pack_f16(lo[2], lo[3]);
                    }
                }
            }
            unsigned char *tst = wbase + ((F8 || C::TILES_FIRST) ? C::TSTOFF : 0);   // one staged 16-row tile
            const uint32_t tst_s = wbase_s + ((F8 || C::TILES_FIRST) ? C::TSTOFF : 0);
            // 16 rows x 16 chunks of 16 bytes of fp16 tokens t0r ..; rows past
            // the window are zero (their p is 0 and 0 * 0 stays 0)
            auto stage_rows = [&](const __half *buf, int t0r, int n) {
    #pragma unroll
                for (int c = lane; c < RT * 16; c += 32) {
                    const int row = c >> 4, col = c & 15;
                    uint4 x = make_uint4(0u, 0u, 0u, 0u);
                    if (row < n) {
                        const int fr = fp16_row(t0r + row, a.n_sink, a.Ns, a.R, a.head);
                        x = __ldcg(reinterpret_cast<const uint4 *>(buf + ((int64_t)p * a.rows + fr) * D) + col);
                    }
                    *reinterpret_cast<uint4 *>(tst + row * RS + col * 16) = x;
                }
            };
            // a raw FP8 tile in stage `stage` (key rows at 0, value rows at RT d),
            // widened to fp16 (exact) into the staged tile
            auto stage_fp8 = [&](int stage, int part) {
                const unsigned char *src = wbase + stage * C::STAGE + part;
                // A quarter-warp takes four 16-byte chunks of each of two
                // rows, the odd row from the other half of the row: its loads
                // cover 128 distinct bytes of banks, and its 32-byte stores
                // land four banks apart on the two rows (RS = 16 mod 128), so
                // neither the loads nor the stores conflict.
                static_assert(RS % 128 == 16, "staged row stride");
                const int odd = (lane >> 2) & 1;
    #pragma unroll
                for (int k = 0; k < RT * 8 / 32; ++k) {
                    const int row = 2 * ((lane >> 3) + 4 * (k & 1)) + odd;
                    const int chunk = (lane & 3) + 4 * ((k >> 1) ^ odd);   // 16 fp8 per chunk
                    const uint4 x = *reinterpret_cast<const uint4 *>(src + row * D + chunk * 16);
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
                    uint32_t hv[8];
    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        hv[2 * k] = fp8x2_to_f16x2<F8>((uint16_t)(w[k] & 0xffffu));
                        hv[2 * k + 1] = fp8x2_to_f16x2<F8>((uint16_t)(w[k] >> 16));
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(tst + row * RS + chunk * 32);
                    dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
                }
            };
            for (int tile = warp; tile < ntile; tile += C::NWARP) {
                const bool hist = F8 && tile < nht;            // an FP8 history tile
                const int t0r = (split + (tile - nht) * a.S) * RT;
                const int n = hist ? RT : min(RT, a.n_fp16 - t0r);
                const int jh = hist ? (tile - warp) / C::NWARP : 0;   // index among the warp's FP8 tiles
                __syncwarp();                               // previous tile fully read
                if (hist) {
                    if (!wait_tile(jh)) {
                        failed = true;
                        break;
                    }
                } else {
                    stage_rows(a.kr, t0r, n);
                }
                __syncwarp();
                // scores: K[16 tokens][128] . B.  FP8 keys go straight from the
                // raw rows into the A fragments: this lane's rows r, r + 8 hold
                // channels 32 t .. 32 t + 31 of k-steps 0..7 (4 bytes each, in the
                // channel order of the second query operand), widened in
                // registers; staged fp16 rows come through ldmatrix.
                float cacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                auto score_steps = [&](auto fp8_keys) {
                    constexpr bool K8 = decltype(fp8_keys)::value;
                    uint32_t kw[16];
                    if constexpr (K8) {
                        const unsigned char *raw = wbase + (jh % C::STAGES) * C::STAGE + 32 * t;
    #pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const uint4 x0 = *reinterpret_cast<const uint4 *>(raw + (r + 8 * h2) * D);
                            const uint4 x1 = *reinterpret_cast<const uint4 *>(raw + (r + 8 * h2) * D + 16);
                            kw[8 * h2 + 0] = x0.x; kw[8 * h2 + 1] = x0.y; kw[8 * h2 + 2] = x0.z; kw[8 * h2 + 3] = x0.w;
                            kw[8 * h2 + 4] = x1.x; kw[8 * h2 + 5] = x1.y; kw[8 * h2 + 6] = x1.z; kw[8 * h2 + 7] = x1.w;
                        }
                    }
    #pragma unroll
                    for (int s = 0; s < 8; s += 2) {
                        uint32_t bh[4];
                        [[maybe_unused]] uint32_t bl[4];
                        const uint32_t baddr = (K8 ? bbuf8_s : bbuf_s) + (s + ((lane >> 3) >> 1)) * C::BSTEP +
                                               ((lane >> 3) & 1) * 128 + (lane & 7) * 16;
                        ldmatrix_x4(baddr, bh);
                        if constexpr (GQ == 8)
                            ldmatrix_x4(baddr + 8 * C::BSTEP, bl);
    #pragma unroll
                        for (int ss = 0; ss < 2; ++ss) {
                            uint32_t ak[4];
                            if constexpr (K8) {
                                const uint32_t w0 = kw[s + ss], w1 = kw[8 + s + ss];
                                ak[0] = fp8x2_to_f16x2<F8 ? F8 : KIVI_FP8_E4M3>((uint16_t)(w0 & 0xffffu));
                                ak[1] = fp8x2_to_f16x2<F8 ? F8 : KIVI_FP8_E4M3>((uint16_t)(w1 & 0xffffu));
                                ak[2] = fp8x2_to_f16x2<F8 ? F8 : KIVI_FP8_E4M3>((uint16_t)(w0 >> 16));
                                ak[3] = fp8x2_to_f16x2<F8 ? F8 : KIVI_FP8_E4M3>((uint16_t)(w1 >> 16));
                            } else {
                                ldmatrix_x4(tst_s + ((lane & 7) + ((lane >> 3) & 1) * 8) * RS +
                                                (16 * (s + ss) + ((lane >> 4) & 1) * 8) * 2, ak);
                            }
                            mma_f16(cacc, ak[0], ak[1], ak[2], ak[3], bh[2 * ss], bh[2 * ss + 1]);
                            if constexpr (GQ == 8)
                                mma_f16(cacc, ak[0], ak[1], ak[2], ak[3], bl[2 * ss], bl[2 * ss + 1]);
                        }
                    }
                };
                if (F8 && hist)
                    score_steps(std::integral_constant<bool, F8 != 0>{});
                else
                    score_steps(std::false_type{});
                float sc[2][2][NH];
    #pragma unroll
                for (int j = 0; j < NH; ++j)
                    sc[1][0][j] = sc[1][1][j] = -INFINITY;  // one k-tile per residual tile
                // FP8 history keys carry the key scale: k = fp8 * k_scale
                const float ks = hist ? kscale_r * a.fp8_k_scale : kscale_r;
                if constexpr (GQ == 4) {
                    sc[0][0][0] = (cacc[0] + cacc[1]) * ks;
                    sc[0][1][0] = (cacc[2] + cacc[3]) * ks;
                } else {
                    sc[0][0][0] = cacc[0] * ks;
                    sc[0][0][NH - 1] = cacc[1] * ks;
                    sc[0][1][0] = cacc[2] * ks;
                    sc[0][1][NH - 1] = cacc[3] * ks;
                }
    #pragma unroll
                for (int j = 0; j < NH; ++j) {
                    if (r >= n)
                        sc[0][0][j] = -INFINITY;
                    if (r + 8 >= n)
                        sc[0][1][j] = -INFINITY;
                }
                float pr[2][2][NH];
                float alpha[NH];
                softmax_step(sc, pr, alpha);                // rescales o_acc (the FP8 history) too
                {
                    const float2 al = make_float2(alpha[0], alpha[NH - 1]);
    #pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
    #pragma unroll
                        for (int k = 0; k < NO; ++k)
                            ores[mt][k] = __fmul2_rn(ores[mt][k], al);
                }
                // values: O^T[c][n] += V^T[c][16 tokens] . P[16 tokens][n]
                __syncwarp();                               // key tile fully read
                if (hist) {
                    stage_fp8(jh % C::STAGES, RT * D);
                    __syncwarp();                           // the raw tile is fully read
                    const bool go = lane == 0 && jh + C::STAGES < nhw;
                    fence_proxy_async_if(go);
                    issue_tile(jh + C::STAGES, go);
                } else {
                    stage_rows(a.vr, t0r, n);
                }
                __syncwarp();
                uint32_t b0, b1;
                if constexpr (GQ == 4) {
                    b0 = movmatrix_t(pack_f16(pr[0][0][0], 0.0f));
                    b1 = movmatrix_t(pack_f16(pr[0][1][0], 0.0f));
                } else {
                    b0 = movmatrix_t(pack_f16(pr[0][0][0], pr[0][0][NH - 1]));
                    b1 = movmatrix_t(pack_f16(pr[0][1][0], pr[0][1][NH - 1]));
                }
    #pragma unroll
                for (int m = 0; m < 8; ++m) {
                    uint32_t av[4];
                    ldmatrix_x4_trans(tst_s + ((lane & 7) + ((lane >> 4) & 1) * 8) * RS +
                                          (16 * m + ((lane >> 3) & 1) * 8) * 2, av);
                    float cv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    mma_f16(cv, av[0], av[1], av[2], av[3], b0, b1);
                    // FP8 history values (times v_scale at the end) go to o_acc,
                    // fp16 rows to ores; both in natural channel order here
                    const float2 c0 = GQ == 4 ? make_float2(cv[0], cv[2]) : make_float2(cv[0], cv[1]);
                    const float2 c1 = make_float2(cv[2], cv[3]);
                    if (F8 && hist) {
                        o_acc[m][0] = __fadd2_rn(o_acc[m][0], c0);
                        if constexpr (GQ == 8)
                            o_acc[m][NO - 1] = __fadd2_rn(o_acc[m][NO - 1], c1);
                    } else {
                        ores[m][0] = __fadd2_rn(ores[m][0], c0);
                        if constexpr (GQ == 8)
                            ores[m][NO - 1] = __fadd2_rn(ores[m][NO - 1], c1);
                    }
                }
            }
        }
    };
    // fp16 output of the tiles parked in the (then idle) staging region
    // through the history loop, so that it holds no registers there
    float4 *ores_park = reinterpret_cast<float4 *>(wbase + C::TSTOFF) + lane;
    float m_park[NH];    // running max when parked: the history rescales o_acc only
    if constexpr (C::TILES_FIRST) {
        run_tiles();     // overlaps the first history copy
#pragma unroll
        for (int j = 0; j < NH; ++j)
            m_park[j] = m_run[j];
        if (warp < ntile) {
            __syncwarp();                               // the staged tile is fully read
#pragma unroll
            for (int i = 0; i < 4 * NO; ++i) {
                const float2 lo = ores[i / NO * 2][i % NO], hi = ores[i / NO * 2 + 1][i % NO];
                ores_park[32 * i] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
    }

    float kscale = 1.0f;           // 2^(24 - E) of the current key group

    // unrolled by two: with two stages each copy of the body has a fixed
    // stage, so its stage offsets are constants
#pragma unroll 2
    for (int i = 0; i < nw; ++i) {
        const int stage = i % C::STAGES;
        if (!mbar_wait(bar0 + 8 * stage, (uint32_t)(i / C::STAGES) & 1u)) {
            // Give every copy this warp has in flight (the late stage i and
            // the ones after it) one more bounded wait, so that its stage
            // memory is normally quiet before the block exits; the block
            // then skips everything that would reuse shared memory and
            // writes empty partials.  The status bit marks the output of
            // this call as invalid.
            if (lane == 0) {
                atomicOr(a.status, kStatusWaitTimeout);
                s_failed = 1;
                for (int k = i; k < nw && k < (i == 0 ? 1 : i + C::STAGES); ++k)
                    mbar_wait(bar0 + 8 * (k % C::STAGES), (uint32_t)(k / C::STAGES) & 1u);
            }
            failed = true;
            break;
        }
        if (i == 0) {
            for (int k = 1; k < nw && k < C::STAGES; ++k)
                issue(k, lane == 0, 0u);
        }
        const unsigned char *st = wbase + stage * C::STAGE;
        const unsigned char *ks_s = st;                          // Ks, Kz (fp32 or fp16)
        const unsigned char *kz_s = st + RC::MW * D;
        const uint8_t *kc_s = st + RC::META + RC::KC;
        const uint8_t *vc_s = st + RC::META + RC::VC;
        const unsigned char *vs_s = st + RC::META + RC::VS;
        const unsigned char *vz_s = st + RC::META + RC::VZ;

        // ---- key B operand for a new group: fp16 hi/lo of q*s*2^(E - o) ---
        if (UG == 1 || i % UG == 0) {
            float sK[4], zK[4], smax = 0.0f;
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
                sK[i2] = meta_load<MF>(ks_s, ch[i2]);
                zK[i2] = meta_load<MF>(kz_s, ch[i2]);
                smax = fmaxf(smax, sK[i2]);
            }
            // scales are >= 0, so their bit patterns order like their values
            smax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(smax)));
            // |q*s| < 2^(eb + 1) for every entry; scale so that it stays < 2^15
            const float bound = smax * qmax;
            int E = 14 - (((__float_as_int(bound) >> 23) & 0xff) - 127);
            E = min(max(E, -100), 100);
            kscale = exp2i(24 - E);
            // v = q s 2^(E - o_k) exactly (power-of-two factors), and
            // v * z 2^(o_k - E) = q s z, the zero-point term, unscaled
            const float fE = exp2i(E), fz = exp2i(o_k - E);
            const float2 sK01 = __fmul2_rn(make_float2(sK[0], sK[1]), make_float2(fE, fE));
            const float2 sK23 = __fmul2_rn(make_float2(sK[2], sK[3]), make_float2(fE, fE));
            const float2 zK01 = __fmul2_rn(make_float2(zK[0], zK[1]), make_float2(fz, fz));
            const float2 zK23 = __fmul2_rn(make_float2(zK[2], zK[3]), make_float2(fz, fz));
            float zpart[GQ];
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
                const float2 v01 = __fmul2_rn(make_float2(qreg[hh][0], qreg[hh][1]), sK01);
                const float2 v23 = __fmul2_rn(make_float2(qreg[hh][2], qreg[hh][3]), sK23);
                const float2 zz = __ffma2_rn(v01, zK01, __fmul2_rn(v23, zK23));
                zpart[hh] = zz.x + zz.y;
                const float hi[4] = {trunc11(v01.x), trunc11(v01.y), trunc11(v23.x), trunc11(v23.y)};
                const float2 m1 = make_float2(-1.0f, -1.0f);
                const float2 lo01 = __ffma2_rn(make_float2(hi[0], hi[1]), m1, v01);   // exact: v - hi
                const float2 lo23 = __ffma2_rn(make_float2(hi[2], hi[3]), m1, v23);
                const float lo[4] = {lo01.x, lo01.y, lo23.x, lo23.y};
                unsigned char *base = bbuf + bs * C::BSTEP + bq * 4;
                if constexpr (GQ == 4) {
                    *reinterpret_cast<uint32_t *>(base + (2 * hh) * 16) = pack_f16(hi[0], hi[1]);
                    *reinterpret_cast<uint32_t *>(base + (2 * hh + 1) * 16) = pack_f16(lo[0], lo[1]);
                    *reinterpret_cast<uint32_t *>(base + 128 + (2 * hh) * 16) = pack_f16(hi[2], hi[3]);
                    *reinterpret_cast<uint32_t *>(base + 128 + (2 * hh + 1) * 16) = pack_f16(lo[2], lo[3]);
                } else {
                    *reinterpret_cast<uint32_t *>(base + hh * 16) = pack_f16(hi[0], hi[1]);
                    *reinterpret_cast<uint32_t *>(base + 128 + hh * 16) = pack_f16(hi[2], hi[3]);
                    *reinterpret_cast<uint32_t *>(base + 8 * C::BSTEP + hh * 16) = pack_f16(lo[0], lo[1]);
                    *reinterpret_cast<uint32_t *>(base + 8 * C::BSTEP + 128 + hh * 16) = pack_f16(lo[2], lo[3]);
                }
            }
            // sum zpart over all lanes; each lane ends with the heads it owns
            if constexpr (GQ == 4) {
                const bool u16 = lane & 16, u8 = lane & 8;
                float k0 = u16 ? zpart[2] : zpart[0], k1 = u16 ? zpart[3] : zpart[1];
                const float s0 = u16 ? zpart[0] : zpart[2], s1 = u16 ? zpart[1] : zpart[3];
                k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
                k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
                float kk = u8 ? k1 : k0;
                kk += __shfl_xor_sync(0xffffffffu, u8 ? k0 : k1, 8);
                kk += __shfl_xor_sync(0xffffffffu, kk, 4);
                kk += __shfl_xor_sync(0xffffffffu, kk, 2);
                kk += __shfl_xor_sync(0xffffffffu, kk, 1);
                // lane holds head ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1)
                zq[0] = __shfl_sync(0xffffffffu, kk, ((t >> 1) << 4) | ((t & 1) << 3));
            } else {
                const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
                float k4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float keep = u16 ? zpart[4 + e] : zpart[e];
                    const float send = u16 ? zpart[e] : zpart[4 + e];
                    k4[e] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
                float k2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float keep = u8 ? k4[2 + e] : k4[e];
                    const float send = u8 ? k4[e] : k4[2 + e];
                    k2[e] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                float kk = (u4 ? k2[1] : k2[0]) + __shfl_xor_sync(0xffffffffu, u4 ? k2[0] : k2[1], 4);
                kk += __shfl_xor_sync(0xffffffffu, kk, 2);
                kk += __shfl_xor_sync(0xffffffffu, kk, 1);
                // lane holds head ((lane>>4)&1)*4 + ((lane>>3)&1)*2 + ((lane>>2)&1)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hh = 2 * t + j;
                    zq[j] = __shfl_sync(0xffffffffu, kk, (((hh >> 2) & 1) << 4) | (((hh >> 1) & 1) << 3) |
                                                             ((hh & 1) << 2));
                }
            }
            __syncwarp();
        }

        // ---- scores of the 32 tokens: two 16-token k-tiles ----------------
        float sc[2][2][NH];     // [k-tile][row r / r+8][head slot]
        {
            uint32_t wa[2][RB / 16], wb[2][RB / 16];  // this thread's 32 channels, per k-tile
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
                const uint8_t *rowA = kc_s + (16 * kt + tau(r)) * RB;
                const uint8_t *rowB = kc_s + (16 * kt + tau(r + 8)) * RB;
                if constexpr (BITS == 2) {
                    const uint2 xa = *reinterpret_cast<const uint2 *>(rowA + 8 * t);
                    const uint2 xb = *reinterpret_cast<const uint2 *>(rowB + 8 * t);
                    wa[kt][0] = xa.x; wa[kt][1] = xa.y; wb[kt][0] = xb.x; wb[kt][1] = xb.y;
                } else {
                    const uint4 xa = *reinterpret_cast<const uint4 *>(rowA + 16 * t);
                    const uint4 xb = *reinterpret_cast<const uint4 *>(rowB + 16 * t);
                    wa[kt][0] = xa.x; wa[kt][1] = xa.y; wa[kt][2] = xa.z; wa[kt][3] = xa.w;
                    wb[kt][0] = xb.x; wb[kt][1] = xb.y; wb[kt][2] = xb.z; wb[kt][3] = xb.w;
                }
            }
            uint32_t sa[2][RB / 16], sb[2][RB / 16];  // the same words moved down by 8 bits
#pragma unroll
            for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                for (int e = 0; e < RB / 16; ++e) {
                    sa[kt][e] = down8(wa[kt][e]);
                    sb[kt][e] = down8(wb[kt][e]);
                }
            // one accumulator per k-tile; the B fragments serve both k-tiles
            float cacc[2][4];
#pragma unroll
            for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    cacc[kt][k] = 0.0f;
#pragma unroll
            for (int s = 0; s < 8; s += 2) {
                uint32_t bh[4], bl[4];
                const uint32_t baddr = bbuf_s + (s + ((lane >> 3) >> 1)) * C::BSTEP +
                                       ((lane >> 3) & 1) * 128 + (lane & 7) * 16;
                ldmatrix_x4(baddr, bh);
                if constexpr (GQ == 8)
                    ldmatrix_x4(baddr + 8 * C::BSTEP, bl);
#pragma unroll
                for (int ss = 0; ss < 2; ++ss) {
                    const int s2 = s + ss;
#pragma unroll
                    for (int kt = 0; kt < 2; ++kt) {
                        uint32_t a0, a1, a2, a3;
                        if constexpr (BITS == 2) {
                            a0 = code_pair_k<2>(wa[kt][0], sa[kt][0], 2 * s2);
                            a1 = code_pair_k<2>(wb[kt][0], sb[kt][0], 2 * s2);
                            a2 = code_pair_k<2>(wa[kt][1], sa[kt][1], 2 * s2);
                            a3 = code_pair_k<2>(wb[kt][1], sb[kt][1], 2 * s2);
                        } else {
                            const int q0 = 2 * (s2 >> 2), pos = 4 * (s2 & 3);
                            a0 = code_pair_k<4>(wa[kt][q0], sa[kt][q0], pos);
                            a1 = code_pair_k<4>(wb[kt][q0], sb[kt][q0], pos);
                            a2 = code_pair_k<4>(wa[kt][q0 + 1], sa[kt][q0 + 1], pos);
                            a3 = code_pair_k<4>(wb[kt][q0 + 1], sb[kt][q0 + 1], pos);
                        }
                        mma_f16(cacc[kt], a0, a1, a2, a3, bh[2 * ss], bh[2 * ss + 1]);
                        if constexpr (GQ == 8)
                            mma_f16(cacc[kt], a0, a1, a2, a3, bl[2 * ss], bl[2 * ss + 1]);
                    }
                }
            }
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
                const float *c = cacc[kt];
                if constexpr (GQ == 4) {
                    sc[kt][0][0] = fmaf(c[0] + c[1], kscale, -zq[0]);
                    sc[kt][1][0] = fmaf(c[2] + c[3], kscale, -zq[0]);
                } else {
                    sc[kt][0][0] = fmaf(c[0], kscale, -zq[0]);
                    sc[kt][0][NH - 1] = fmaf(c[1], kscale, -zq[NH - 1]);
                    sc[kt][1][0] = fmaf(c[2], kscale, -zq[0]);
                    sc[kt][1][NH - 1] = fmaf(c[3], kscale, -zq[NH - 1]);
                }
            }
        }

        // ---- online softmax over the 32 tokens (per warp) -----------------
        float pr[2][2][NH];
        float alpha[NH];
        softmax_step(sc, pr, alpha);

        // ---- values: O^T[c][n] += codes^T . (p*s) for both k-tiles --------
        // The mma accumulator rounds its fp32 sums toward zero, so a long
        // chain of small additions drifts low; and o = sum p s code - sum p s z
        // cancels heavily.  Each slice therefore starts a fresh mma
        // accumulator and is added into o_acc with round-to-nearest.
        //
        // Code operand: in the stored channel order each lane finds the runs
        // of all its value groups in CH consecutive bytes of a token row (its
        // channels G j + (G/8) r + e); the 16-bit halves of tokens k and k + 1
        // are paired with one prmt, each code pair is masked out as an fp16x2
        // of subnormals code * 2^(pos - 24) and moved to the top of the
        // mantissa (code * 2^(-14 - BITS)) with one exact fp16 multiply: the
        // tensor core aligns the products of an mma on the operands' exponent
        // fields, treating a subnormal as 2^-14, so a code low in the mantissa
        // would lose bits of its product.
        constexpr int TOP = 10 - BITS;                  // top of the fp16 mantissa
        constexpr int RL = G / 8;                       // codes per run
        constexpr int NHALF = CH / 2;                   // 16-bit halves per lane chunk
        // B operand (p*s) per k-tile: query group 4 puts value groups j and
        // j + 1 into columns 2 head and 2 head + 1 (one transpose serves two
        // groups), query group 8 one group per transpose with heads 2t, 2t+1
        constexpr int NB = GQ == 4 ? (VG + 1) / 2 : VG;
        uint32_t bb[2][NB][2];
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            const int tA = 16 * kt + tau(r), tB = 16 * kt + tau(r + 8);
            float sA[VG], sB[VG], zA[VG], zB[VG];
            if constexpr (!MF && VG == 4) {
                // one vector load per token for its four scales / zero points
                const float4 a4 = *reinterpret_cast<const float4 *>(vs_s + 16 * tA);
                const float4 b4 = *reinterpret_cast<const float4 *>(vs_s + 16 * tB);
                const float4 c4 = *reinterpret_cast<const float4 *>(vz_s + 16 * tA);
                const float4 d4 = *reinterpret_cast<const float4 *>(vz_s + 16 * tB);
                sA[0] = a4.x; sA[1] = a4.y; sA[2] = a4.z; sA[3] = a4.w;
                sB[0] = b4.x; sB[1] = b4.y; sB[2] = b4.z; sB[3] = b4.w;
                zA[0] = c4.x; zA[1] = c4.y; zA[2] = c4.z; zA[3] = c4.w;
                zB[0] = d4.x; zB[1] = d4.y; zB[2] = d4.z; zB[3] = d4.w;
            } else {
#pragma unroll
                for (int j = 0; j < VG; ++j) {
                    sA[j] = meta_load<MF>(vs_s, tA * VG + j);
                    sB[j] = meta_load<MF>(vs_s, tB * VG + j);
                    zA[j] = meta_load<MF>(vz_s, tA * VG + j);
                    zB[j] = meta_load<MF>(vz_s, tB * VG + j);
                }
            }
            if constexpr (GQ == 4 && VG % 2 == 0) {
                // value groups in pairs: (s_j, s_j+1) sit side by side in
                // the loaded metadata, so each product and each zero-point
                // update is one fp32x2 operation with no register moves
                // (per element the same roundings as the scalar form below)
                const float2 prA = make_float2(pr[kt][0][0], pr[kt][0][0]);
                const float2 prB = make_float2(pr[kt][1][0], pr[kt][1][0]);
#pragma unroll
                for (int jb = 0; jb < VG / 2; ++jb) {
                    const int j0 = 2 * jb, j1 = 2 * jb + 1;
                    const float2 pA = __fmul2_rn(prA, make_float2(sA[j0], sA[j1]));
                    const float2 pB = __fmul2_rn(prB, make_float2(sB[j0], sB[j1]));
                    float2 z = make_float2(zacc[j0][0], zacc[j1][0]);
                    z = __ffma2_rn(pA, make_float2(zA[j0], zA[j1]),
                                   __ffma2_rn(pB, make_float2(zB[j0], zB[j1]), z));
                    zacc[j0][0] = z.x;
                    zacc[j1][0] = z.y;
                    bb[kt][jb][0] = movmatrix_t(pack_f16(pA.x, pA.y));
                    bb[kt][jb][1] = movmatrix_t(pack_f16(pB.x, pB.y));
                }
            } else if constexpr (GQ == 4) {
                float pA[VG], pB[VG];
#pragma unroll
                for (int j = 0; j < VG; ++j) {
                    const float2 pAB = __fmul2_rn(make_float2(pr[kt][0][0], pr[kt][1][0]), make_float2(sA[j], sB[j]));
                    pA[j] = pAB.x;
                    pB[j] = pAB.y;
                    zacc[j][0] = fmaf(pAB.x, zA[j], fmaf(pAB.y, zB[j], zacc[j][0]));
                }
#pragma unroll
                for (int jb = 0; jb < NB; ++jb) {
                    const int j0 = 2 * jb, j1 = 2 * jb + 1;
                    bb[kt][jb][0] = movmatrix_t(pack_f16(pA[j0], j1 < VG ? pA[j1] : 0.0f));
                    bb[kt][jb][1] = movmatrix_t(pack_f16(pB[j0], j1 < VG ? pB[j1] : 0.0f));
                }
            } else if constexpr (VG % 2 == 0) {
                // query group 8, value groups in pairs: one fp32x2 product per
                // (token row, head, group pair); the packs take the heads of
                // one group from two products (same roundings per element
                // as the form below)
#pragma unroll
                for (int jb = 0; jb < VG / 2; ++jb) {
                    const int j0 = 2 * jb, j1 = 2 * jb + 1;
                    const float2 sA2 = make_float2(sA[j0], sA[j1]), sB2 = make_float2(sB[j0], sB[j1]);
                    const float2 zA2 = make_float2(zA[j0], zA[j1]), zB2 = make_float2(zB[j0], zB[j1]);
                    float2 pA[NH], pB[NH];
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        pA[hh] = __fmul2_rn(make_float2(pr[kt][0][hh], pr[kt][0][hh]), sA2);
                        pB[hh] = __fmul2_rn(make_float2(pr[kt][1][hh], pr[kt][1][hh]), sB2);
                        float2 z = make_float2(zacc[j0][hh], zacc[j1][hh]);
                        z = __ffma2_rn(pA[hh], zA2, __ffma2_rn(pB[hh], zB2, z));
                        zacc[j0][hh] = z.x;
                        zacc[j1][hh] = z.y;
                    }
                    bb[kt][j0][0] = movmatrix_t(pack_f16(pA[0].x, pA[NH - 1].x));
                    bb[kt][j0][1] = movmatrix_t(pack_f16(pB[0].x, pB[NH - 1].x));
                    bb[kt][j1][0] = movmatrix_t(pack_f16(pA[0].y, pA[NH - 1].y));
                    bb[kt][j1][1] = movmatrix_t(pack_f16(pB[0].y, pB[NH - 1].y));
                }
            } else {
#pragma unroll
                for (int j = 0; j < VG; ++j) {
                    const float2 pA = __fmul2_rn(make_float2(pr[kt][0][0], pr[kt][0][NH - 1]), make_float2(sA[j], sA[j]));
                    const float2 pB = __fmul2_rn(make_float2(pr[kt][1][0], pr[kt][1][NH - 1]), make_float2(sB[j], sB[j]));
                    float2 z2 = make_float2(zacc[j][0], zacc[j][NH - 1]);
                    z2 = __ffma2_rn(pA, make_float2(zA[j], zA[j]), __ffma2_rn(pB, make_float2(zB[j], zB[j]), z2));
                    zacc[j][0] = z2.x;
                    zacc[j][NH - 1] = z2.y;
                    bb[kt][j][0] = movmatrix_t(pack_f16(pA.x, pA.y));
                    bb[kt][j][1] = movmatrix_t(pack_f16(pB.x, pB.y));
                }
            }
        }
        // code words: [k-tile][token pair (2t, 2t+1) / (2t+8, 2t+9)][half]
        uint32_t xw[2][2][NHALF], xs[2][2][NHALF];
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
            uint32_t w[4][NHALF / 2];                   // tokens 2t, 2t+1, 2t+8, 2t+9
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = 2 * t + (q & 1) + 8 * (q >> 1);
                const uint8_t *row = vc_s + (16 * kt + tau(k)) * RB + CH * r;
                if constexpr (CH == 4) {
                    w[q][0] = *reinterpret_cast<const uint32_t *>(row);
                } else {
                    const uint2 x = *reinterpret_cast<const uint2 *>(row);
                    w[q][0] = x.x;
                    w[q][1] = x.y;
                }
            }
#pragma unroll
            for (int pr2 = 0; pr2 < 2; ++pr2)
#pragma unroll
                for (int hh = 0; hh < NHALF; ++hh) {
                    const uint32_t sel = (hh & 1) ? 0x7632u : 0x5410u;
                    xw[kt][pr2][hh] = prmt(w[2 * pr2][hh >> 1], w[2 * pr2 + 1][hh >> 1], sel);
                    xs[kt][pr2][hh] = down8(xw[kt][pr2][hh]);
                }
        }
        // the code pair of run position e of group j for a token pair
        auto vcode = [&](int kt, int pr2, int j, int e) -> uint32_t {
            const int bit = BITS * (RL * j + e);
            const int hh = bit / 16, pos = bit % 16;
            const uint32_t x = pos <= TOP ? xw[kt][pr2][hh] : xs[kt][pr2][hh];
            const int pp = pos <= TOP ? pos : pos - 8;
            const uint32_t m = x & ((((1u << BITS) - 1u) << pp) * 0x00010001u);
            if (pp == TOP)
                return m;
            const __half f = __ushort_as_half((unsigned short)((15 + TOP - pp) << 10));   // 2^(TOP - pp)
            return hmul2_u32(m, __halves2half2(f, f));
        };
#pragma unroll
        for (int j = 0; j < VG; ++j) {
#pragma unroll
            for (int km = 0; km < MT; ++km) {
                float cv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const uint32_t a0 = vcode(kt, 0, j, 2 * km);
                    const uint32_t a1 = vcode(kt, 0, j, 2 * km + 1);
                    const uint32_t a2 = vcode(kt, 1, j, 2 * km);
                    const uint32_t a3 = vcode(kt, 1, j, 2 * km + 1);
                    if constexpr (GQ == 4)
                        mma_f16(cv, a0, a1, a2, a3, bb[kt][j >> 1][0], bb[kt][j >> 1][1]);
                    else
                        mma_f16(cv, a0, a1, a2, a3, bb[kt][j][0], bb[kt][j][1]);
                }
                const int mt = j * MT + km;
                if constexpr (GQ == 4) {
                    // group j's columns: 2 head + (j & 1)
                    const float2 add = (j & 1) ? make_float2(cv[1], cv[3]) : make_float2(cv[0], cv[2]);
                    o_acc[mt][0] = __fadd2_rn(o_acc[mt][0], add);
                } else {
                    o_acc[mt][0] = __fadd2_rn(o_acc[mt][0], make_float2(cv[0], cv[1]));
                    o_acc[mt][1] = __fadd2_rn(o_acc[mt][1], make_float2(cv[2], cv[3]));
                }
            }
        }

        __syncwarp();   // every lane is done with this stage
        {
            const bool go = lane == 0 && i + C::STAGES < nw;
            fence_proxy_async_if(go);
            issue(i + C::STAGES, go, 0u);
        }
    }

    if constexpr (!C::TILES_FIRST)
        run_tiles();
    __syncthreads();
    if (s_failed) {
        // no shared-memory epilogue (a late copy may still land in a stage):
        // empty partials straight from registers; the host reads the status
        for (int hh = 0; hh < a.g; ++hh) {
            store_partial(a, qrow0 + hh, split, -INFINITY, 0.0f, 0.0f, tid);
            if (split == a.S - 1)
                store_partial(a, qrow0 + hh, a.S, -INFINITY, 0.0f, 0.0f, tid);
        }
        combine_if_last<(GQ > 4)>(a, p, &s_last);
        return;
    }

    // ---- per-warp epilogue: reduce over the 8 lanes sharing a head column -
    if constexpr (C::TILES_FIRST) {
        if (warp < ntile) {
            // to the final running max: 2^(max when parked - final max)
            const float2 f = make_float2(ex2_ftz(m_park[0] - m_run[0]), ex2_ftz(m_park[NH - 1] - m_run[NH - 1]));
#pragma unroll
            for (int i = 0; i < 4 * NO; ++i) {
                const float4 v = ores_park[32 * i];
                ores[i / NO * 2][i % NO] = __fmul2_rn(make_float2(v.x, v.y), f);
                ores[i / NO * 2 + 1][i % NO] = __fmul2_rn(make_float2(v.z, v.w), f);
            }
        }
    }
    float l_w[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        float l = l_part[j];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_w[j] = l;
#pragma unroll
        for (int v = 0; v < VG; ++v) {
            float z = zacc[v][j];
            z += __shfl_xor_sync(0xffffffffu, z, 4);
            z += __shfl_xor_sync(0xffffffffu, z, 8);
            z += __shfl_xor_sync(0xffffffffu, z, 16);
            zacc[v][j] = z;
        }
    }
    if (lane == 0)
        for (int s = 0; s < C::STAGES; ++s)
            mbar_inval(bar0 + 8 * s);
    __syncthreads();   // every warp has left its pipeline; its memory is free
    float *om = reinterpret_cast<float *>(smem);                 // [4 warps][GQ][D]
    float *mw = om + C::NWARP * GQ * D;                          // [4][GQ]
    float *lw = mw + C::NWARP * GQ;                              // [4][GQ]
    // undo the 2^(kCodeTop - 24) of the subnormal code operand
    const float fA = exp2i(24 - kCodeTop<BITS>), fB = fA;
    if constexpr (F8) {
        // FP8 history: natural channel order (16 m + r, + 8), times v_scale
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int jj = 0; jj < NH; ++jj) {
                const int hh = (GQ == 4) ? t : 2 * t + jj;
                float *row = om + (warp * GQ + hh) * D + 16 * m + r;
                if constexpr (GQ == 4) {
                    row[0] = o_acc[m][0].x * a.fp8_v_scale;
                    row[8] = o_acc[m][0].y * a.fp8_v_scale;
                } else {
                    row[0] = (jj == 0 ? o_acc[m][0].x : o_acc[m][0].y) * a.fp8_v_scale;
                    row[8] = (jj == 0 ? o_acc[m][1].x : o_acc[m][1].y) * a.fp8_v_scale;
                }
            }
    }
#pragma unroll
    for (int mt = 0; mt < 8 && !F8; ++mt) {
        const int j = mt / MT, km = mt % MT;
        const int chA = G * j + (G / 8) * r + 2 * km;            // row r; row r + 8 is chA + 1
#pragma unroll
        for (int jj = 0; jj < NH; ++jj) {
            const int hh = (GQ == 4) ? t : 2 * t + jj;
            float oA, oB;
            if constexpr (GQ == 4) {
                oA = o_acc[mt][0].x;
                oB = o_acc[mt][0].y;
            } else {
                oA = jj == 0 ? o_acc[mt][0].x : o_acc[mt][0].y;
                oB = jj == 0 ? o_acc[mt][NO - 1].x : o_acc[mt][NO - 1].y;
            }
            om[(warp * GQ + hh) * D + chA] = fmaf(oA, fA, -zacc[j][jj]);
            om[(warp * GQ + hh) * D + chA + 1] = fmaf(oB, fB, -zacc[j][jj]);
        }
    }
    if (warp < ntile) {            // residual outputs: channel 16m + r (+ 8)
        __syncwarp();
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int jj = 0; jj < NH; ++jj) {
                const int hh = (GQ == 4) ? t : 2 * t + jj;
                float *row = om + (warp * GQ + hh) * D + 16 * m + r;
                if constexpr (GQ == 4) {
                    row[0] += ores[m][0].x;
                    row[8] += ores[m][0].y;
                } else {
                    row[0] += jj == 0 ? ores[m][0].x : ores[m][0].y;
                    row[8] += jj == 0 ? ores[m][1].x : ores[m][1].y;
                }
            }
    }
    if (r == 0) {
#pragma unroll
        for (int jj = 0; jj < NH; ++jj) {
            const int hh = (GQ == 4) ? t : 2 * t + jj;
            mw[warp * GQ + hh] = m_run[jj];
            lw[warp * GQ + hh] = l_w[jj];
        }
    }
    __syncthreads();
    for (int hh = 0; hh < a.g; ++hh) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NWARP; ++w)
            M = fmaxf(M, mw[w * GQ + hh]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NWARP; ++w) {
                const float e = exp2f(mw[w * GQ + hh] - M);
                L = fmaf(lw[w * GQ + hh], e, L);
                O = fmaf(om[(w * GQ + hh) * D + tid], e, O);
            }
        }
        store_partial(a, qrow0 + hh, split, M, L, O, tid);
    }
    if (split == a.S - 1)                  // the residual went into partial S-1: slot S is empty
        for (int hh = 0; hh < a.g; ++hh)
            store_partial(a, qrow0 + hh, a.S, -INFINITY, 0.0f, 0.0f, tid);
    combine_if_last<(GQ > 4)>(a, p, &s_last);
}

__global__ void __launch_bounds__(kHeadDim) decode_combine_kernel(CombineArgs a)
{
    merge_row<1>(a.ws_m, a.ws_l, a.ws_o, a.out, blockIdx.x, a.S + 1, threadIdx.x);
}

// ------------------------------------------------------------ launchers ---

template <typename K>
cudaError_t prepare(K kernel, int smem)
{
    // opt in to more than 48 KB of dynamic shared memory (idempotent)
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// The opt-in to more than 48 KB of dynamic shared memory is a per-device
// attribute of the kernel: set it once on each device, from any host thread
// (one bit per device and kernel, set after the call succeeded; a second
// thread racing on the same device only repeats the idempotent call).
template <typename K>
cudaError_t prepare_on_device(K kernel, int smem, std::atomic<uint64_t> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    e = prepare(kernel, smem);
    if (e == cudaSuccess && bit)
        done.fetch_or(bit, std::memory_order_release);
    return e;
}

template <int BITS, int G, int GQ, int MF, int F8 = 0>
cudaError_t launch_mma(const DecodeArgs &a, int pairs, cudaStream_t s, int *blocks_per_sm)
{
    using C = MmaCfg<BITS, G, GQ, MF, F8>;
    static_assert(C::SMEM >= (kThreads / 32) * GQ * (kHeadDim + 2) * 4, "epilogue buffer");
    auto kernel = decode_split_mma<BITS, G, GQ, MF, F8>;
    static std::atomic<uint64_t> prepared{0};   // devices with the attribute set
    cudaError_t e = prepare_on_device(kernel, C::SMEM, prepared);
    if (e != cudaSuccess)
        return e;
    if (blocks_per_sm)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kernel, kThreads, C::SMEM);
    dim3 grid((unsigned)a.S, (unsigned)pairs);
    kernel<<<grid, kThreads, C::SMEM, s>>>(a);
    return cudaGetLastError();
}

template <int BITS, int G, int MAXG, int MF>
cudaError_t launch_simt(const DecodeArgs &a, int pairs, cudaStream_t s, int *blocks_per_sm)
{
    auto kernel = decode_split_simt<BITS, G, MAXG, MF>;
    if (blocks_per_sm)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kernel, kThreads, 0);
    dim3 grid((unsigned)a.S, (unsigned)pairs);
    kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int BITS, int G, int MF>
cudaError_t launch_bg(int g, const DecodeArgs &a, int pairs, cudaStream_t s, int *bps)
{
    if (G == 16) {
        if (g <= 1) return launch_simt<BITS, G, 1, MF>(a, pairs, s, bps);
        if (g <= 2) return launch_simt<BITS, G, 2, MF>(a, pairs, s, bps);
        if (g <= 4) return launch_simt<BITS, G, 4, MF>(a, pairs, s, bps);
        return launch_simt<BITS, G, 8, MF>(a, pairs, s, bps);
    }
    if (g <= 4)
        return launch_mma<BITS, (G < 32 ? 32 : G), 4, MF>(a, pairs, s, bps);
    return launch_mma<BITS, (G < 32 ? 32 : G), 8, MF>(a, pairs, s, bps);
}

// Every kernel for one metadata width: the caller picks by bits and G.
template <int MF>
cudaError_t launch_meta(int bits, int G, int g, const DecodeArgs &a, int pairs, cudaStream_t s,
                        int *bps)
{
    if (bits != 2 && bits != 4)
        return cudaErrorInvalidValue;
    switch (G * 8 + bits) {
    case 16 * 8 + 2: return launch_bg<2, 16, MF>(g, a, pairs, s, bps);
    case 32 * 8 + 2: return launch_bg<2, 32, MF>(g, a, pairs, s, bps);
    case 64 * 8 + 2: return launch_bg<2, 64, MF>(g, a, pairs, s, bps);
    case 128 * 8 + 2: return launch_bg<2, 128, MF>(g, a, pairs, s, bps);
    case 16 * 8 + 4: return launch_bg<4, 16, MF>(g, a, pairs, s, bps);
    case 32 * 8 + 4: return launch_bg<4, 32, MF>(g, a, pairs, s, bps);
    case 64 * 8 + 4: return launch_bg<4, 64, MF>(g, a, pairs, s, bps);
    case 128 * 8 + 4: return launch_bg<4, 128, MF>(g, a, pairs, s, bps);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace kivi
