// Sender launches for the default codec (4096-value chunks, k = 64, max-abs scale), and the
// dispatch of every other codec to ef_compress_variants.cu.
#include "ef_compress.cuh"

namespace spl {

cudaError_t launch_ef_compress(const CompressTable& tab, const Codec& cd, bool bf16, bool ef_host,
                               float beta, uint8_t* payload, float* scales, uint32_t* flags,
                               cudaStream_t stream) {
    if (is_default_codec(cd))
        return launch_codec<DefaultGeometry, kScaleMax>(tab, bf16, ef_host, beta, payload, scales,
                                                        flags, stream);
    return launch_ef_compress_variant(tab, cd, bf16, ef_host, beta, payload, scales, flags, stream);
}

#if SPL_CHECKED
SPL_DEBUG_READER(debug_read_compress)
#endif

}  // namespace spl
