// Receiver launches for the default record geometry (4096-value chunks, k = 64), and the
// dispatch of the other geometries to decode_aggregate_variants.cu.
#include "decode_aggregate.cuh"

namespace spl {

cudaError_t launch_decode_aggregate(const DecodeTable& tab, const Codec& cd, int P, int64_t n,
                                    float* mean, float* theta, float lr, bool validate,
                                    PeerStats* stats, uint32_t* flags, cudaStream_t stream) {
    if (cd.chunk == kChunk && cd.topk == kTopK)
        return launch_geometry<DefaultGeometry>(tab, P, n, mean, theta, lr, validate, stats, flags,
                                                stream);
    return launch_decode_aggregate_variant(tab, cd, P, n, mean, theta, lr, validate, stats, flags,
                                           stream);
}

#if SPL_CHECKED
SPL_DEBUG_READER(debug_read_decode)
#endif

}  // namespace spl
