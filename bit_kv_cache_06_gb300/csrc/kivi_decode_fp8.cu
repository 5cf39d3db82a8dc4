// kivi_decode_fp8.cu -- decode over an FP8 KV history (E4M3 or E5M2, one
// scale per tensor): the split-K tensor-core kernel in its FP8 mode, compiled
// apart from the packed-code kernels.
#include "kivi_decode_kernels.cuh"

namespace kivi {

cudaError_t launch_decode_fp8(int fmt, const DecodeArgs &a, int pairs, cudaStream_t s,
                              int *blocks_per_sm)
{
    // the packed-code template arguments (2-bit, G = 32) only size the
    // per-warp stage buffers, which the FP8 mode uses for its staged tiles
    if (fmt == KIVI_FP8_E4M3)
        return a.g <= 4 ? launch_mma<2, 32, 4, 0, KIVI_FP8_E4M3>(a, pairs, s, blocks_per_sm)
                        : launch_mma<2, 32, 8, 0, KIVI_FP8_E4M3>(a, pairs, s, blocks_per_sm);
    if (fmt == KIVI_FP8_E5M2)
        return a.g <= 4 ? launch_mma<2, 32, 4, 0, KIVI_FP8_E5M2>(a, pairs, s, blocks_per_sm)
                        : launch_mma<2, 32, 8, 0, KIVI_FP8_E5M2>(a, pairs, s, blocks_per_sm);
    return cudaErrorInvalidValue;
}

}  // namespace kivi
