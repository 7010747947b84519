// Record layout kernels: (idx[C][64], codes[C][64]) <-> payload[C][112].
//
// Layout: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
// Pre-Training", "SparseLoCo: Three Compression Levers in One Pass", per-chunk equation
// (64 fields, each a 2-bit value and a 12-bit index: 896 bits, 112 bytes).  Entry r is the
// field code | idx << 2 at bits [14r, 14r + 14), least significant bit first.
//
// One warp per record, grid-stride: lane l handles entries l and l + 32; record words are
// assembled (or taken apart) with shuffles and moved as 16-byte vectors.
#include "spl_device.cuh"
#include "spl_kernels.h"

namespace spl {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
k_pack(const uint16_t* __restrict__ idx, const uint8_t* __restrict__ codes, int64_t C,
       uint8_t* __restrict__ payload) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t c = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5; c < C;
         c += warps) {
        const int64_t e = c * kTopK;
        if (!SPL_CHECK(c < C, kSitePack, c)) continue;
        const uint32_t f0 = (codes[e + lane] & 3u) | ((idx[e + lane] & 0xfffu) << 2);
        const uint32_t f1 = (codes[e + lane + 32] & 3u) | ((idx[e + lane + 32] & 0xfffu) << 2);
        store_record(payload + c * kRecordBytes, record_word(f0, f1, lane), lane);
    }
}

__global__ void __launch_bounds__(kThreads)
k_unpack(const uint8_t* __restrict__ payload, int64_t C, uint16_t* __restrict__ idx,
         uint8_t* __restrict__ codes) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t c = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5; c < C;
         c += warps) {
        if (!SPL_CHECK(c < C, kSitePack, c)) continue;
        const uint32_t* words = reinterpret_cast<const uint32_t*>(payload + c * kRecordBytes);
        const uint32_t mine = lane < kRecordWords ? words[lane] : 0u;
        const int64_t e = c * kTopK;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = lane + 32 * h;
            const int bit = kFieldBits * r;
            const int w = bit >> 5;
            const int off = bit & 31;
            const uint32_t lo = __shfl_sync(0xffffffffu, mine, w);
            const uint32_t hi = __shfl_sync(0xffffffffu, mine, (w + 1) & 31);
            uint32_t f = lo >> off;
            if (off > 32 - kFieldBits) f |= hi << (32 - off);
            f &= (1u << kFieldBits) - 1u;
            codes[e + r] = static_cast<uint8_t>(f & 3u);
            idx[e + r] = static_cast<uint16_t>(f >> 2);
        }
    }
}

int warp_grid(int64_t C) {
    const int64_t ctas = (C + (kThreads / 32) - 1) / (kThreads / 32);
    const int cap = persistent_grid(reinterpret_cast<const void*>(&k_pack), kThreads, 0);
    return static_cast<int>(ctas < cap ? ctas : cap);
}

}  // namespace

#if SPL_CHECKED
SPL_DEBUG_READER(debug_read_pack)
#endif

cudaError_t launch_pack(const uint16_t* idx, const uint8_t* codes, int64_t C, uint8_t* payload,
                        cudaStream_t stream) {
    if (C == 0) return cudaSuccess;
    const int grid = warp_grid(C);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    k_pack<<<grid, kThreads, 0, stream>>>(idx, codes, C, payload);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* payload, int64_t C, uint16_t* idx, uint8_t* codes,
                          cudaStream_t stream) {
    if (C == 0) return cudaSuccess;
    const int grid = warp_grid(C);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    k_unpack<<<grid, kThreads, 0, stream>>>(payload, C, idx, codes);
    return cudaGetLastError();
}

}  // namespace spl
