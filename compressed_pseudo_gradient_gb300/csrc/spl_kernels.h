// Host-side declarations of the kernel launchers behind the C ABI (internal header).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace spl {

constexpr int kMaxTensorsPerLaunch = 64;
constexpr int kMaxPeers = 256;

// A codec: chunk length L, entries per record k, scale rule (0: max |a| / 1.5, the default;
// 1: mean-abs).
struct Codec {
    int chunk;
    int topk;
    int rule;
};

// The record geometries (L, k) with kernels in this library; the first is the default.
constexpr int kNumGeometries = 5;
constexpr int kGeometries[kNumGeometries][2] = {
    {4096, 64}, {4096, 32}, {4096, 128}, {2048, 32}, {8192, 128}};

inline bool is_default_codec(const Codec& cd) {
    return cd.chunk == 4096 && cd.topk == 64 && cd.rule == 0;
}

// Bytes of one record of a supported codec (k x (2 + log2 L) bits), or 0 when the library
// has no kernels for it.
inline int64_t codec_record_bytes(const Codec& cd) {
    if (cd.rule != 0 && cd.rule != 1) return 0;
    for (int i = 0; i < kNumGeometries; ++i) {
        if (kGeometries[i][0] != cd.chunk || kGeometries[i][1] != cd.topk) continue;
        int bits = 0;
        while ((1 << bits) < cd.chunk) ++bits;
        return static_cast<int64_t>(cd.topk) * (2 + bits) / 8;
    }
    return 0;
}

// A table of tensors compressed in one launch; chunk_begin holds prefix sums of the
// per-tensor chunk counts (chunk_begin[num] = chunks in this launch).
struct CompressTable {
    const void* delta[kMaxTensorsPerLaunch];
    float* ef[kMaxTensorsPerLaunch];
    int64_t n[kMaxTensorsPerLaunch];
    int64_t chunk_begin[kMaxTensorsPerLaunch + 1];
    int num;
};

struct DecodeTable {
    const uint8_t* payload[kMaxPeers];
    const float* scale[kMaxPeers];
};

// ef_host: the tensors' error buffers are pinned host memory, read and written over the host
// link with plain accesses (delta stays in device memory; default codec only).  The table's
// chunk_begin counts chunks of the codec's length.
cudaError_t launch_ef_compress(const CompressTable& tab, const Codec& cd, bool bf16, bool ef_host,
                               float beta, uint8_t* payload, float* scales, uint32_t* flags,
                               cudaStream_t stream);
// The same for a codec other than the default (cudaErrorNotSupported for an unknown one).
cudaError_t launch_ef_compress_variant(const CompressTable& tab, const Codec& cd, bool bf16,
                                       bool ef_host, float beta, uint8_t* payload, float* scales,
                                       uint32_t* flags, cudaStream_t stream);

// Per-peer statistics (same layout as spl_peer_stats in spl.h), accumulated by the kernel.
struct PeerStats {
    uint32_t rejected;
    uint32_t big;
    uint32_t negative;
    float max_scale;
    double sumsq;
};

// validate: check every record (strictly ascending indices, a finite non-negative scale) and
// leave out the ones that fail; always on when stats is given.
cudaError_t launch_decode_aggregate(const DecodeTable& tab, const Codec& cd, int P, int64_t n,
                                    float* mean, float* theta, float lr, bool validate,
                                    PeerStats* stats, uint32_t* flags, cudaStream_t stream);
// The same for a record geometry other than the default (the scale rule does not matter to
// the receiver).
cudaError_t launch_decode_aggregate_variant(const DecodeTable& tab, const Codec& cd, int P,
                                            int64_t n, float* mean, float* theta, float lr,
                                            bool validate, PeerStats* stats, uint32_t* flags,
                                            cudaStream_t stream);

cudaError_t launch_pack(const uint16_t* idx, const uint8_t* codes, int64_t C,
                        uint8_t* payload, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* payload, int64_t C, uint16_t* idx, uint8_t* codes,
                          cudaStream_t stream);

// Chunks per CTA in the codec kernels' wave schedule (spl_device.cuh, cta_chunks): fewer keep
// the chunks in flight closer together, more spread each CTA's start-up and final work (the
// sender's last record, the receiver's first copies and accumulator clear) over more chunks.
// Measured at 2^30 values: the sender 1.860 ms at 16 (1.860 at 8 and 12, 1.867-1.869 at 24
// and 32; at 24 the decoder layer's multi-tensor round gains 0.8 % and the flat one loses
// 0.5 %), the 24-peer receiver 2.032-2.050 ms at 32 (2.078 at 8, 2.057 at 16, 2.052 at 24,
// 2.094 at 48, 2.077 at 64; its lean 8-peer mean of 2^27 values 0.0961 ms at 32 and 16,
// 0.0967 at 8).
constexpr int kSendChunksPerCta = 16;
constexpr int kSendChunksPerCtaBf16 = 24;   // a bf16 delta: 2^27 heavy-tailed values 0.2260
                                            // ms at 24, 0.2290 at 16, 0.2301 at 32
constexpr int kRecvChunksPerCta = 32;

// The grid that covers `total` chunks in waves of `resident` CTAs taking `per_cta` chunks
// each: one partial wave when everything fits in one, else whole waves (the last one's
// surplus CTAs exit at once).
inline int wave_grid(int64_t total, int resident, int per_cta) {
    const int64_t per_wave = static_cast<int64_t>(resident) * per_cta;
    const int64_t waves = (total + per_wave - 1) / per_wave;
    return static_cast<int>(waves <= 1 ? (total < resident ? total : resident) : waves * resident);
}

// Data-movement reference kernels (spl_calib.h), C chunks of 4,096 values: sender = the
// sender's movement (out0 = in0 + in1), otherwise the receiver's (out0 = -in0, out1 = in0);
// the codec kernels' wave schedule, or one persistent wave.
cudaError_t launch_calib_moves(bool sender, const float* in0, const float* in1, float* out0,
                               float* out1, int64_t C, bool persistent, uint32_t* flags,
                               cudaStream_t stream);

#if SPL_CHECKED
// Checked build only: each translation unit's debug array (see spl_device.cuh), copied to out
// (kDebugWords words) and cleared when reset is set.
cudaError_t debug_read_compress(uint32_t* out, bool reset);
cudaError_t debug_read_compress_variants(uint32_t* out, bool reset);
cudaError_t debug_read_decode(uint32_t* out, bool reset);
cudaError_t debug_read_decode_variants(uint32_t* out, bool reset);
cudaError_t debug_read_pack(uint32_t* out, bool reset);
#endif

// Resident-CTA count used to size persistent grids: SMs x blocks per SM for the kernel.
int persistent_grid(const void* kernel, int threads, size_t dyn_smem);

}  // namespace spl
