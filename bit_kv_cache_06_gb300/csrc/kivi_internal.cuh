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
constexpr int kSplitBlocksCap = 1024;  // (pair, split) blocks the workspace is sized for
constexpr size_t kWorkspaceHeader = 256;

// Streaming quantisation of nq_new tokens.  The tokens are the concatenation
// [old residual (n_old tokens), new input tokens]; quantised rows go to
// [n_quant, n_quant + nq_new) of every pair.
struct QuantArgs {
    const __half *k_in, *v_in;        // new tokens
    int64_t in_sb, in_sh, in_st;      // element strides: batch, kv head, token
    const __half *k_res, *v_res;      // residual [P][R][D]
    int n_old;
    int R;
    int Hkv;
    int64_t n_quant;
    int64_t nq_new;
    int64_t cap;
    uint8_t *kc, *vc;
    float *ks, *kz, *vs, *vz;
};

// Copy ntok input tokens starting at src_tok0 into residual slots
// [dst_slot0, dst_slot0 + ntok) of every pair.
struct ResidArgs {
    const __half *k_in, *v_in;
    int64_t in_sb, in_sh, in_st;
    __half *k_res, *v_res;
    int R;
    int Hkv;
    int64_t src_tok0;
    int dst_slot0;
    int ntok;
};

// One split-K decode launch over all pairs.
struct DecodeArgs {
    const uint8_t *kc, *vc;
    const float *ks, *kz, *vs, *vz;
    const __half *kr, *vr;
    const __half *q;                  // [B][Hq][D]
    float *ws_m, *ws_l, *ws_o;        // [B*Hq][S+1], [B*Hq][S+1], [B*Hq][S+1][D]
    unsigned *status;                 // workspace status word (error bits)
    unsigned *counters;               // [pairs] blocks finished per pair (fused combine)
    __half *out;                      // [B][Hq][D]; nullptr: partials only
    int64_t cap;
    int64_t n_quant;
    int n_resid;
    int R;
    int Hkv;
    int g;                            // query heads per kv head
    int S;                            // blocks (history splits) per pair; partial S = residual
    float scale_log2;                 // softmax scale * log2(e)
};

struct CombineArgs {
    const float *ws_m, *ws_l, *ws_o;
    __half *out;                      // [B*Hq][D]
    int S;                            // history splits; S + 1 partials per row
};

cudaError_t launch_quantize(int bits, int G, const QuantArgs &a, int pairs, cudaStream_t s);
cudaError_t launch_residual_copy(const ResidArgs &a, int pairs, cudaStream_t s);
cudaError_t launch_decode_partial(int bits, int G, const DecodeArgs &a, int pairs, cudaStream_t s);
// Resident (pair, split) blocks per SM of the history kernel launch_decode_partial uses.
cudaError_t decode_blocks_per_sm(int bits, int G, int g, int *blocks);
cudaError_t launch_decode_combine(const CombineArgs &a, int rows, cudaStream_t s);

}  // namespace kivi
