// Sender launches for the codec variants: other chunk lengths and k, and the mean-abs scale
// rule (device-resident error buffers only).  The kernel is the one in ef_compress.cuh.
#include "ef_compress.cuh"

namespace spl {

namespace {

template <int L, int K>
cudaError_t launch_rule(const CompressTable& tab, int rule, bool bf16, bool ef_host, float beta,
                        uint8_t* payload, float* scales, uint32_t* flags, cudaStream_t stream) {
    using Geo = Geometry<L, K>;
    if (rule == kScaleMax)
        return launch_codec<Geo, kScaleMax>(tab, bf16, ef_host, beta, payload, scales, flags, stream);
    return launch_codec<Geo, kScaleMeanAbs>(tab, bf16, ef_host, beta, payload, scales, flags, stream);
}

}  // namespace

cudaError_t launch_ef_compress_variant(const CompressTable& tab, const Codec& cd, bool bf16,
                                       bool ef_host, float beta, uint8_t* payload, float* scales,
                                       uint32_t* flags, cudaStream_t stream) {
    if (codec_record_bytes(cd) == 0) return cudaErrorNotSupported;
    const int L = cd.chunk, K = cd.topk, R = cd.rule;
    if (L == 4096 && K == 64 && R == kScaleMeanAbs)
        return launch_codec<DefaultGeometry, kScaleMeanAbs>(tab, bf16, ef_host, beta, payload,
                                                            scales, flags, stream);
    if (L == 4096 && K == 32)
        return launch_rule<4096, 32>(tab, R, bf16, ef_host, beta, payload, scales, flags, stream);
    if (L == 4096 && K == 128)
        return launch_rule<4096, 128>(tab, R, bf16, ef_host, beta, payload, scales, flags, stream);
    if (L == 2048 && K == 32)
        return launch_rule<2048, 32>(tab, R, bf16, ef_host, beta, payload, scales, flags, stream);
    if (L == 8192 && K == 128)
        return launch_rule<8192, 128>(tab, R, bf16, ef_host, beta, payload, scales, flags, stream);
    return cudaErrorNotSupported;
}

#if SPL_CHECKED
SPL_DEBUG_READER(debug_read_compress_variants)
#endif

}  // namespace spl
