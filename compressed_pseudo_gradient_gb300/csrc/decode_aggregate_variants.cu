// Receiver launches for the record geometries of the codec variants (other chunk lengths and
// k).  The kernel is the one in decode_aggregate.cuh.
#include "decode_aggregate.cuh"

namespace spl {

cudaError_t launch_decode_aggregate_variant(const DecodeTable& tab, const Codec& cd, int P,
                                            int64_t n, float* mean, float* theta, float lr,
                                            bool validate, PeerStats* stats, uint32_t* flags,
                                            cudaStream_t stream) {
    const int L = cd.chunk, K = cd.topk;
    if (L == 4096 && K == 32)
        return launch_geometry<Geometry<4096, 32>>(tab, P, n, mean, theta, lr, validate,
                                                         stats, flags, stream);
    if (L == 4096 && K == 128)
        return launch_geometry<Geometry<4096, 128>>(tab, P, n, mean, theta, lr, validate,
                                                         stats, flags, stream);
    if (L == 2048 && K == 32)
        return launch_geometry<Geometry<2048, 32>>(tab, P, n, mean, theta, lr, validate,
                                                         stats, flags, stream);
    if (L == 8192 && K == 128)
        return launch_geometry<Geometry<8192, 128>>(tab, P, n, mean, theta, lr, validate,
                                                         stats, flags, stream);
    return cudaErrorNotSupported;
}

#if SPL_CHECKED
SPL_DEBUG_READER(debug_read_decode_variants)
#endif

}  // namespace spl
