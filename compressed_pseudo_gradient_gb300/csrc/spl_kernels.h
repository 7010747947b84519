// Host-side declarations of the kernel launchers behind the C ABI (internal header).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace spl {

constexpr int kMaxTensorsPerLaunch = 64;
constexpr int kMaxPeers = 256;

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
// link with plain accesses (delta stays in device memory).
cudaError_t launch_ef_compress(const CompressTable& tab, bool bf16, bool ef_host, float beta,
                               uint8_t* payload, float* scales, uint32_t* flags,
                               cudaStream_t stream);

// Per-peer statistics (same layout as spl_peer_stats in spl.h), accumulated by the kernel.
struct PeerStats {
    uint32_t rejected;
    uint32_t big;
    uint32_t negative;
    float max_scale;
    double sumsq;
};

cudaError_t launch_decode_aggregate(const DecodeTable& tab, int P, int64_t n, float* mean,
                                    float* theta, float lr, PeerStats* stats, uint32_t* flags,
                                    cudaStream_t stream);

cudaError_t launch_pack(const uint16_t* idx, const uint8_t* codes, int64_t C,
                        uint8_t* payload, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* payload, int64_t C, uint16_t* idx, uint8_t* codes,
                          cudaStream_t stream);

// Resident-CTA count used to size persistent grids: SMs x blocks per SM for the kernel.
int persistent_grid(const void* kernel, int threads, size_t dyn_smem);

}  // namespace spl
