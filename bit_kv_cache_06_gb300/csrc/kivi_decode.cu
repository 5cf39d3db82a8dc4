// kivi_decode.cu -- the decode entry points of the library (fp32-metadata
// kernels; the fp16-metadata ones are instantiated in kivi_decode_f16.cu).
#include "kivi_decode_kernels.cuh"

namespace kivi {

cudaError_t launch_decode_partial(int bits, int G, int meta, const DecodeArgs &a, int pairs,
                                  cudaStream_t s)
{
    if (meta)
        return launch_decode_partial_f16(bits, G, a, pairs, s, nullptr);
    return launch_meta<0>(bits, G, a.g, a, pairs, s, nullptr);
}

cudaError_t decode_blocks_per_sm(int bits, int G, int meta, int g, int *blocks)
{
    DecodeArgs dummy{};
    dummy.g = g;
    if (meta)
        return launch_decode_partial_f16(bits, G, dummy, 0, nullptr, blocks);
    return launch_meta<0>(bits, G, g, dummy, 0, nullptr, blocks);
}

cudaError_t launch_decode_combine(const CombineArgs &a, int rows, cudaStream_t s)
{
    decode_combine_kernel<<<(unsigned)rows, kHeadDim, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kivi
