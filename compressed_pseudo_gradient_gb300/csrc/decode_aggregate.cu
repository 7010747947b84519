// Receiver kernel of the SparseLoCo codec: decode P peers' records, take their mean, and
// optionally apply the outer step theta <- theta - lr * mean, in one pass over HBM.
//
// Method: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
// Pre-Training", "SparseLoCo: Three Compression Levers in One Pass" (item 3: the receiver
// rebuilds positions from the 12-bit indices) and "Why Extreme Sparsity Doesn't Break
// Convergence" ("Sparse aggregation can improve model quality": the peers' sparse updates
// are aggregated); "Why DiLoCo Alone Isn't Enough" for the pseudo-gradient's sign.
//
// Design (HBM-bound: P x 116 B read per chunk, 16 KB of mean written, 32 KB of theta read and
// written when the outer step is fused):
//   - one 256-thread CTA per chunk, grid-stride over chunks with a persistent grid; the
//     chunk's accumulator is 16 KB of shared memory, so the dense output is written exactly
//     once and nothing is zero-filled or atomically added in global memory;
//   - all P records (7 x 16 B each) and scales are fetched by all threads at once, together
//     with the chunk's theta, so their latencies overlap;
//   - one warp adds the peers into the accumulator in peer order (each lane owns entries r
//     and r + 32; indices inside a valid record are strictly ascending, hence distinct), which
//     fixes the fp32 summation order; it also checks each record and skips malformed ones;
//   - the dense pass reads the accumulator, divides by P, stores the mean and the updated
//     theta with streaming stores, and clears the accumulator for the next chunk.
#include <cfloat>

#include "spl_device.cuh"
#include "spl_kernels.h"

namespace spl {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = kChunk / kThreads;   // 16
constexpr int kVec = kPer / 4;

__global__ void __launch_bounds__(kThreads)
k_decode_aggregate(const DecodeTable tab, int P, int64_t n, float* __restrict__ mean,
                   float* __restrict__ theta, float neg_lr, uint32_t* __restrict__ flags) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* acc = reinterpret_cast<float*>(smem_raw);                             // 4096
    uint4* rec = reinterpret_cast<uint4*>(smem_raw + kChunk * sizeof(float));    // P x 7
    float* sc = reinterpret_cast<float*>(rec + P * kRecordVec);                  // P

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t C = (n + kChunk - 1) / kChunk;
    const float pf = static_cast<float>(P);
    bool bad = false;

#pragma unroll
    for (int v = 0; v < kVec; ++v)
        reinterpret_cast<float4*>(acc)[v * (kThreads) + tid] = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int64_t c = blockIdx.x; c < C; c += gridDim.x) {
        const int64_t base = c * kChunk;
        const bool full = base + kChunk <= n;
        const int valid = full ? kChunk : static_cast<int>(n - base);

        float4 th[kVec];
        if (theta != nullptr && full) {
#pragma unroll
            for (int v = 0; v < kVec; ++v) th[v] = ld_stream_f4(theta + base + v * 1024 + 4 * tid);
        }
        for (int i = tid; i < P * kRecordVec; i += kThreads) {
            const int p = i / kRecordVec;
            const int w = i - p * kRecordVec;
            rec[i] = __ldcs(reinterpret_cast<const uint4*>(tab.payload[p] + c * kRecordBytes) + w);
        }
        for (int p = tid; p < P; p += kThreads) sc[p] = __ldcs(tab.scale[p] + c);
        __syncthreads();

        if (warp == 0) {
            for (int p = 0; p < P; ++p) {
                const uint32_t* words = reinterpret_cast<const uint32_t*>(rec + p * kRecordVec);
                const uint32_t f0 = record_field(words, lane);
                const uint32_t f1 = record_field(words, lane + 32);
                const uint32_t i0 = f0 >> 2;
                const uint32_t i1 = f1 >> 2;
                const uint32_t first_hi = __shfl_sync(0xffffffffu, i1, 0);
                uint32_t next0 = __shfl_down_sync(0xffffffffu, i0, 1);
                const uint32_t next1 = __shfl_down_sync(0xffffffffu, i1, 1);
                if (lane == 31) next0 = first_hi;
                const float s = sc[p];
                const bool ok = i0 < next0 && (lane == 31 || i1 < next1) && s >= 0.0f &&
                                s <= FLT_MAX;
                if (!__all_sync(0xffffffffu, ok)) {
                    bad = true;
                    continue;
                }
                if (base + i0 < n) acc[i0] = __fadd_rn(acc[i0], level_value(f0 & 3u, s));
                if (base + i1 < n) acc[i1] = __fadd_rn(acc[i1], level_value(f1 & 3u, s));
                __syncwarp();
            }
        }
        __syncthreads();

#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            const int j0 = v * 1024 + 4 * tid;
            float4 s4 = reinterpret_cast<float4*>(acc)[j0 >> 2];
            reinterpret_cast<float4*>(acc)[j0 >> 2] = make_float4(0.f, 0.f, 0.f, 0.f);
            s4.x = __fdiv_rn(s4.x, pf);
            s4.y = __fdiv_rn(s4.y, pf);
            s4.z = __fdiv_rn(s4.z, pf);
            s4.w = __fdiv_rn(s4.w, pf);
            if (full) {
                st_stream_f4(mean + base + j0, s4);
                if (theta != nullptr) {
                    float4 t4 = th[v];
                    t4.x = __fmaf_rn(neg_lr, s4.x, t4.x);
                    t4.y = __fmaf_rn(neg_lr, s4.y, t4.y);
                    t4.z = __fmaf_rn(neg_lr, s4.z, t4.z);
                    t4.w = __fmaf_rn(neg_lr, s4.w, t4.w);
                    st_stream_f4(theta + base + j0, t4);
                }
            } else {
                const float m[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = j0 + u;
                    if (j < valid) {
                        mean[base + j] = m[u];
                        if (theta != nullptr)
                            theta[base + j] = __fmaf_rn(neg_lr, m[u], theta[base + j]);
                    }
                }
            }
        }
    }
    if (bad && flags != nullptr) atomicOr(flags, kFlagBadRecord);
}

}  // namespace

cudaError_t launch_decode_aggregate(const DecodeTable& tab, int P, int64_t n, float* mean,
                                    float* theta, float lr, uint32_t* flags,
                                    cudaStream_t stream) {
    const int64_t C = (n + kChunk - 1) / kChunk;
    if (C == 0) return cudaSuccess;
    const size_t smem = kChunk * sizeof(float) + static_cast<size_t>(P) * (kRecordBytes + 4);
    const int resident = persistent_grid(reinterpret_cast<const void*>(&k_decode_aggregate),
                                         kThreads, smem);
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    const int grid = static_cast<int>(C < resident ? C : resident);
    k_decode_aggregate<<<grid, kThreads, smem, stream>>>(tab, P, n, mean, theta, -lr, flags);
    return cudaGetLastError();
}

}  // namespace spl
