// Data-movement reference kernels (declared in include/spl_calib.h): the codec kernels' byte
// movement with none of their arithmetic, so that the time each takes is the floor that the
// codec kernel's own access pattern sets.  Not part of the codec.
#include "spl_device.cuh"
#include "spl_kernels.h"

namespace spl {
namespace {

constexpr int kCalibChunk = 4096;
constexpr int kCalibThreads = 256;
constexpr int kCalibCtasPerSm = 4;   // as the codec kernels run: 4 resident CTAs per SM

// kSender: stage = [in0 chunk | in1 chunk], out0 = in0 + in1 with plain stores.
// receiver: stage = [in0 chunk], out0 = -in0 and out1 = in0 with plain stores.
// Each thread handles 16 values, 4 vectors of 4 at j = v * 1024 + 4 * tid, as the codec
// kernels do.
template <bool kSender>
__global__ void __launch_bounds__(kCalibThreads, kCalibCtasPerSm)
k_calib_moves(const float* __restrict__ in0, const float* __restrict__ in1,
              float* __restrict__ out0, float* __restrict__ out1, int64_t C,
              uint32_t* __restrict__ flags, int ctas, int per_cta) {
    constexpr int kArrays = kSender ? 2 : 1;
    constexpr uint32_t kBytes = kCalibChunk * 4;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* stage = reinterpret_cast<float*>(smem_raw);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + kArrays * kBytes);
    const int tid = threadIdx.x;
    const int64_t G = ctas;
    const ChunkSpan span = cta_chunks(C, ctas, per_cta, blockIdx.x);
    if (span.first >= span.end) return;
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_expect_tx(bar, kArrays * kBytes);
        bulk_load(stage, in0 + span.first * kCalibChunk, kBytes, bar);
        if constexpr (kSender)
            bulk_load(stage + kCalibChunk, in1 + span.first * kCalibChunk, kBytes, bar);
    }
    __syncthreads();
    uint32_t parity = 0;
    bool aborted = false;
    for (int64_t c = span.first; c < span.end; c += G) {
        const bool timed_out = !mbar_wait(bar, parity);
        if (__syncthreads_or(timed_out)) {
            aborted = true;
            break;
        }
        float4 r0[4], r1[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int j = v * 1024 + 4 * tid;
            const float4 x = *reinterpret_cast<const float4*>(stage + j);
            if constexpr (kSender) {
                const float4 y = *reinterpret_cast<const float4*>(stage + kCalibChunk + j);
                r0[v] = make_float4(__fadd_rn(x.x, y.x), __fadd_rn(x.y, y.y), __fadd_rn(x.z, y.z),
                                    __fadd_rn(x.w, y.w));
            } else {
                r0[v] = make_float4(-x.x, -x.y, -x.z, -x.w);
                r1[v] = x;
            }
        }
        parity ^= 1u;
        // the sender stores its values right after reading them, before the barrier that
        // frees the stage; the receiver stores at the end of its chunk, after the next copies
        // have started
        if constexpr (kSender) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                *reinterpret_cast<float4*>(out0 + c * kCalibChunk + v * 1024 + 4 * tid) = r0[v];
        }
        __syncthreads();   // the stage has been read: the next chunk's copies may land in it
        if (tid == 0 && c + G < span.end) {
            fence_async_smem();
            mbar_expect_tx(bar, kArrays * kBytes);
            bulk_load(stage, in0 + (c + G) * kCalibChunk, kBytes, bar);
            if constexpr (kSender)
                bulk_load(stage + kCalibChunk, in1 + (c + G) * kCalibChunk, kBytes, bar);
        }
        if constexpr (!kSender) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int64_t i = c * kCalibChunk + v * 1024 + 4 * tid;
                *reinterpret_cast<float4*>(out0 + i) = r0[v];
                *reinterpret_cast<float4*>(out1 + i) = r1[v];
            }
        }
    }
    if (aborted && tid == 0) {
        // the copy that timed out may still land: wait for it (bounded) before the CTA's
        // shared memory is released, and report it if that wait runs out too
        const bool pending = !mbar_wait(bar, parity);
        if (flags != nullptr) atomicOr(flags, kFlagTimeout | (pending ? kFlagCopyPending : 0u));
    }
}

template <bool kSender>
cudaError_t launch_calib(const float* in0, const float* in1, float* out0, float* out1, int64_t C,
                         bool persistent, uint32_t* flags, cudaStream_t stream) {
    const void* kern = reinterpret_cast<const void*>(&k_calib_moves<kSender>);
    const size_t smem = (kSender ? 2 : 1) * kCalibChunk * 4 + 16;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int resident = sms * kCalibCtasPerSm;
    // persistent: one wave of resident CTAs, each taking every resident-th chunk
    const int per_cta =
        persistent ? static_cast<int>((C + resident - 1) / resident)
                   : (kSender ? kSendChunksPerCta : kRecvChunksPerCta);
    const int grid = wave_grid(C, resident, per_cta);
    k_calib_moves<kSender><<<grid, kCalibThreads, smem, stream>>>(in0, in1, out0, out1, C, flags,
                                                                  resident, per_cta);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_calib_moves(bool sender, const float* in0, const float* in1, float* out0,
                               float* out1, int64_t C, bool persistent, uint32_t* flags,
                               cudaStream_t stream) {
    return sender ? launch_calib<true>(in0, in1, out0, nullptr, C, persistent, flags, stream)
                  : launch_calib<false>(in0, nullptr, out0, out1, C, persistent, flags, stream);
}

}  // namespace spl
