// kivi_internal.cuh -- declarations shared by the CUDA translation units of
// libkivi (kernel argument blocks and launchers).  Not part of the C ABI.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kivi.h"

namespace kivi {

constexpr int kHeadDim = 128;   // d supported by this build
constexpr int kChunk = 128;     // quantised tokens per decode split unit
constexpr int kMaxGroupQ = 8;   // largest query group Hq / Hkv
constexpr int kSplitBlocksCap = 4096;  // (pair, split) blocks the workspace is sized for
constexpr size_t kWorkspaceHeader = 256;
constexpr int kMaxSink = 256;   // largest number of sink tokens

// Byte offsets inside one key-group record of the history buffer (see
// include/kivi.h): Ks[d] | Kz[d] | G / SL sub-slices of SL = min(G, 32) tokens,
// each Kc[SL][RB] | Vc[SL][RB] | Vs[SL][VG] | Vz[SL][VG]; scales and zero
// points are fp32 (MF = 0) or fp16 (MF = 1).
template <int BITS, int G, int MF = 0>
struct Rec {
    static constexpr int D = kHeadDim;
    static constexpr int RB = D * BITS / 8;                 // code bytes per token row
    static constexpr int VG = D / G;                        // value groups per token
    static constexpr int SL = G < 32 ? G : 32;              // tokens per sub-slice
    static constexpr int MW = MF ? 2 : 4;                   // bytes per scale / zero point
    static constexpr int META = 2 * MW * D;                 // Ks and Kz
    static constexpr int SUB = SL * (2 * RB + 2 * MW * VG); // one sub-slice
    static constexpr int BYTES = META + (G / SL) * SUB;     // the record
    static constexpr int KC = 0, VC = SL * RB, VS = 2 * SL * RB, VZ = 2 * SL * RB + MW * SL * VG;
    // byte offset of token t (0..G-1) of the record in the buffer part `part`
    __host__ __device__ static constexpr int64_t row(int t, int part_off, int width)
    {
        return META + (int64_t)(t / SL) * SUB + part_off + (int64_t)(t % SL) * width;
    }
};

// Scale / zero point i of a metadata array stored as fp32 or fp16.
template <int MF>
__device__ __forceinline__ float meta_load(const void *base, int i)
{
    if constexpr (MF)
        return __half2float(reinterpret_cast<const __half *>(base)[i]);
    else
        return reinterpret_cast<const float *>(base)[i];
}

template <int MF>
__device__ __forceinline__ void meta_store(void *base, int i, float v)
{
    if constexpr (MF)
        reinterpret_cast<__half *>(base)[i] = __float2half_rn(v);   // exact: v is a binary16
    else
        reinterpret_cast<float *>(base)[i] = v;
}

// fp16 row of fp16 token i (the sink rows first, then the residual ring from
// its oldest token).
__host__ __device__ __forceinline__ int fp16_row(int i, int n_sink, int Ns, int R, int head)
{
    if (i < n_sink)
        return i;
    const int slot = head + (i - n_sink);
    return Ns + (slot >= R ? slot - R : slot);
}

// Stored position of value channel c (include/kivi.h, "Stored value channel
// order"): runs of G/8 channels with the same index inside their group sit
// side by side; natural order when such a run is shorter than a byte.
template <int BITS, int G>
__host__ __device__ constexpr int value_pos(int c)
{
    return (G / 8) * BITS < 8 ? c
                              : 16 * ((c % G) / (G / 8)) + (G / 8) * (c / G) + (c % G) % (G / 8);
}

// Streaming quantisation of nq_new tokens.  The tokens are the concatenation
// [old residual (n_old tokens), new input tokens from input token `skip` on];
// quantised tokens go to records n_quant / G .. of every pair.
struct QuantArgs {
    const __half *k_in, *v_in;        // new tokens
    int64_t in_sb, in_sh, in_st;      // element strides: batch, kv head, token
    int64_t skip;                     // input tokens taken by the sink before these
    const __half *k_res, *v_res;      // fp16 rows [P][rows][D]
    int rows;                         // fp16 rows per pair: Ns sink rows + R slots
    int Ns;                           // residual slot s is row Ns + s
    int R;
    int head;                         // slot of the oldest residual token (a ring)
    int n_old;
    int Hkv;
    int64_t n_quant;
    int64_t nq_new;
    int64_t cap;
    uint8_t *hist;                    // history records
    float fp8_k_scale, fp8_v_scale;   // FP8 KV only
    int v8;                           // inputs and fp16 rows 32-byte aligned
};

// Copy ntok input tokens starting at src_tok0 into fp16 rows of every pair:
// rows dst_row0 + i (ring = 0: sink rows), or the residual ring slots
// dst_row0 + (slot0 + i) mod ring.
struct ResidArgs {
    const __half *k_in, *v_in;
    int64_t in_sb, in_sh, in_st;
    __half *k_res, *v_res;
    int rows;
    int Hkv;
    int64_t src_tok0;
    int dst_row0;
    int ring;
    int slot0;
    int ntok;
};

// One split-K decode launch over all pairs.
struct DecodeArgs {
    const uint8_t *hist;              // history records
    const __half *kr, *vr;            // fp16 rows [P][rows][D]
    const __half *q;                  // [B][Hq][D]
    float *ws_m, *ws_l, *ws_o;        // [B*Hq][S+1], [B*Hq][S+1], [B*Hq][S+1][D]
    unsigned *status;                 // workspace status word (error bits)
    unsigned *counters;               // [pairs] blocks finished per pair (fused combine)
    __half *out;                      // [B][Hq][D]; nullptr: partials only
    int64_t cap;
    int64_t n_quant;
    int n_fp16;                       // fp16 tokens: the sink rows, then the residual ring
    int n_sink;                       // sink rows 0 .. n_sink - 1
    int Ns;                           // residual slot s is row Ns + s
    int R;
    int head;                         // slot of the oldest residual token
    int rows;                         // fp16 rows per pair
    int Hkv;
    int g;                            // query heads per kv head
    int S;                            // blocks (history splits) per pair; partial S = fp16 rows
    float scale_log2;                 // softmax scale * log2(e)
    float fp8_k_scale, fp8_v_scale;   // FP8 KV only
    int poison_first_copy;            // test hook: see kivi_test_decode_wait_timeout
};

struct CombineArgs {
    const float *ws_m, *ws_l, *ws_o;
    __half *out;                      // [B*Hq][D]
    int S;                            // history splits; S + 1 partials per row
};

cudaError_t launch_quantize(int bits, int G, int meta, const QuantArgs &a, int pairs, cudaStream_t s);
cudaError_t launch_quantize_fp8(int fmt, const QuantArgs &a, int pairs, cudaStream_t s);
cudaError_t launch_residual_copy(const ResidArgs &a, int pairs, cudaStream_t s);
cudaError_t launch_decode_partial(int bits, int G, int meta, const DecodeArgs &a, int pairs,
                                  cudaStream_t s);
// Resident (pair, split) blocks per SM of the history kernel launch_decode_partial uses.
cudaError_t decode_blocks_per_sm(int bits, int G, int meta, int g, int *blocks);
// FP8 KV decode (kivi_decode_fp8.cu); blocks_per_sm set: occupancy query only.
cudaError_t launch_decode_fp8(int fmt, const DecodeArgs &a, int pairs, cudaStream_t s,
                              int *blocks_per_sm);
// The fp16-metadata instantiations (kivi_decode_f16.cu).
cudaError_t launch_decode_partial_f16(int bits, int G, const DecodeArgs &a, int pairs,
                                      cudaStream_t s, int *blocks_per_sm);
cudaError_t launch_decode_combine(const CombineArgs &a, int rows, cudaStream_t s);

}  // namespace kivi
