// kivi_decode_f16.cu -- the decode kernels for caches whose scales and zero
// points are stored as fp16 (KIVI_META_FP16), compiled apart from the fp32
// ones.
#include "kivi_decode_kernels.cuh"

namespace kivi {

cudaError_t launch_decode_partial_f16(int bits, int G, const DecodeArgs &a, int pairs,
                                      cudaStream_t s, int *blocks_per_sm)
{
    return launch_meta<1>(bits, G, a.g, a, pairs, s, blocks_per_sm);
}

}  // namespace kivi
