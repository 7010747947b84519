// Fused sender kernel of the SparseLoCo codec: error feedback, chunk top-64, 2-bit quantise,
// 14-bit field packing and the error-feedback residual, in one pass over HBM.
//
// Method: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
// Pre-Training", "SparseLoCo: Three Compression Levers in One Pass" (items 1-3, per-chunk
// equation) and "Why Extreme Sparsity Doesn't Break Convergence" ("Error feedback
// accumulation": what is not sent stays in the buffer for the next round).
//
// Design (HBM-bound: 8 B read + 4 B written per fp32 value, 116 B written per chunk):
//   - one 256-thread CTA per 4096-value chunk, grid-stride over chunks with a grid of
//     SMs x resident CTAs; each thread keeps 16 values in registers, loaded as four 16-byte
//     vectors at chunk offsets v*1024 + 4*tid (v = 0..3), so every warp access is 512
//     contiguous bytes; the error buffer is read and written exactly once, with streaming
//     cache hints;
//   - the 64th-largest |a| is found by a radix select on the 31-bit magnitude keys:
//     shared-memory histograms of key bits [30:20], [19:9] and [8:0], each restricted to the
//     keys that match the digits found so far, stopping early once the boundary bin is taken
//     whole; no sort and no global scratch;
//   - keys above the threshold, and threshold ties in index order, are marked in a 4096-bit
//     shared bitmap, so one warp compacts the 64 indices in ascending order with popc scans;
//   - the threads that own the chosen values compute their codes and residuals in registers
//     and store the whole chunk of the error buffer once; one warp packs the 64 fields into
//     the 112-byte record with shuffles and 16-byte stores.
#include "spl_device.cuh"
#include "spl_kernels.h"

namespace spl {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = kChunk / kThreads;    // 16 values per thread
constexpr int kVec = kPer / 4;             // 4 vectors of 4 per thread
constexpr int kBitmapWords = kChunk / 32;  // 128

struct Smem {
    uint32_t hist[2][2048];
    uint32_t sel_bm[kBitmapWords];  // keys strictly above the threshold prefix
    uint32_t eq_bm[kBitmapWords];   // keys equal to the threshold prefix (tie candidates)
    uint32_t fin_bm[kBitmapWords];  // the 64 chosen positions
    uint32_t warp_tot[kWarps];
    uint32_t warp_max[kWarps];
    uint32_t bcast[3];              // digit, count above the digit's bin, count in the bin
    float scale;
    uint16_t sel_idx[kTopK];
    uint8_t code_at[kChunk];
};

// Block-wide search of the bin holding the need-th largest key (counting from the top bin).
// Thread t owns bins [kBinsPer*t, kBinsPer*t + kBinsPer).  Writes sm.bcast; the caller
// synchronises before reading it.
template <int kBins>
__device__ __forceinline__ void find_digit(Smem& sm, const uint32_t* hist, uint32_t need,
                                           int tid, int lane, int warp) {
    constexpr int kBinsPer = kBins / kThreads;
    uint32_t h[kBinsPer];
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < kBinsPer; ++i) {
        h[i] = hist[kBinsPer * tid + i];
        sum += h[i];
    }
    uint32_t incl = sum;   // suffix sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
    }
    if (lane == 0) sm.warp_tot[warp] = incl;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        if (w > warp) incl += sm.warp_tot[w];
    const uint32_t excl = incl - sum;
    if (excl < need && incl >= need) {
        uint32_t run = excl;
#pragma unroll
        for (int i = kBinsPer - 1; i >= 0; --i) {
            if (run + h[i] >= need) {
                sm.bcast[0] = kBinsPer * tid + i;
                sm.bcast[1] = run;
                sm.bcast[2] = h[i];
                break;
            }
            run += h[i];
        }
    }
}

template <bool kBf16>
__device__ __forceinline__ void load_accumulate(const void* delta, const float* ef, int valid,
                                                bool full, float beta, int tid,
                                                float (&a)[kPer]) {
    if (full) {
        float4 e4[kVec];
#pragma unroll
        for (int v = 0; v < kVec; ++v) e4[v] = ld_stream_f4(ef + v * 1024 + 4 * tid);
        if constexpr (kBf16) {
            uint2 d2[kVec];
            const uint16_t* d = static_cast<const uint16_t*>(delta);
#pragma unroll
            for (int v = 0; v < kVec; ++v) d2[v] = ld_stream_u2(d + v * 1024 + 4 * tid);
#pragma unroll
            for (int v = 0; v < kVec; ++v) {
                a[4 * v + 0] = __fmaf_rn(beta, e4[v].x, bf16_bits_to_float(d2[v].x & 0xffffu));
                a[4 * v + 1] = __fmaf_rn(beta, e4[v].y, bf16_bits_to_float(d2[v].x >> 16));
                a[4 * v + 2] = __fmaf_rn(beta, e4[v].z, bf16_bits_to_float(d2[v].y & 0xffffu));
                a[4 * v + 3] = __fmaf_rn(beta, e4[v].w, bf16_bits_to_float(d2[v].y >> 16));
            }
        } else {
            float4 d4[kVec];
            const float* d = static_cast<const float*>(delta);
#pragma unroll
            for (int v = 0; v < kVec; ++v) d4[v] = ld_stream_f4(d + v * 1024 + 4 * tid);
#pragma unroll
            for (int v = 0; v < kVec; ++v) {
                a[4 * v + 0] = __fmaf_rn(beta, e4[v].x, d4[v].x);
                a[4 * v + 1] = __fmaf_rn(beta, e4[v].y, d4[v].y);
                a[4 * v + 2] = __fmaf_rn(beta, e4[v].z, d4[v].z);
                a[4 * v + 3] = __fmaf_rn(beta, e4[v].w, d4[v].w);
            }
        }
    } else {
#pragma unroll
        for (int v = 0; v < kVec; ++v)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = v * 1024 + 4 * tid + u;
                float d = 0.0f, e = 0.0f;
                if (j < valid) {
                    e = ef[j];
                    d = kBf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(delta)[j])
                              : static_cast<const float*>(delta)[j];
                }
                a[4 * v + u] = j < valid ? __fmaf_rn(beta, e, d) : 0.0f;   // pads are +0
            }
    }
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 3)
k_ef_compress(const CompressTable tab, float beta, uint8_t* __restrict__ payload,
              float* __restrict__ scales, uint32_t* __restrict__ flags) {
    __shared__ __align__(16) Smem sm;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t total = tab.chunk_begin[tab.num];
    bool nonfinite = false;

    for (int64_t c = blockIdx.x; c < total; c += gridDim.x) {
        int t = 0;
        {
            int hi = tab.num;
            while (hi - t > 1) {
                const int mid = (t + hi) >> 1;
                if (tab.chunk_begin[mid] <= c) t = mid; else hi = mid;
            }
        }
        const int64_t base = (c - tab.chunk_begin[t]) * kChunk;
        const int64_t n = tab.n[t];
        float* ef = tab.ef[t] + base;
        const void* delta = kBf16
            ? static_cast<const void*>(static_cast<const uint16_t*>(tab.delta[t]) + base)
            : static_cast<const void*>(static_cast<const float*>(tab.delta[t]) + base);
        const bool full = base + kChunk <= n;
        const int valid = full ? kChunk : static_cast<int>(n - base);

        // ---- a = beta * e + delta, and the magnitude keys --------------------------------
        float a[kPer];
        load_accumulate<kBf16>(delta, ef, valid, full, beta, tid, a);
        uint32_t key[kPer];
        uint32_t kmax = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            key[i] = mag_key(a[i]);
            kmax = max(kmax, key[i]);
        }
        nonfinite |= kmax >= kKeyInf;

        // ---- clear the histograms and bitmaps; chunk max --------------------------------
        {
            uint4* h4 = reinterpret_cast<uint4*>(&sm.hist[0][0]);
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < 4; ++i) h4[tid + i * kThreads] = z;   // 2 x 2048 words
            if (tid < kBitmapWords) sm.sel_bm[tid] = 0;
            else sm.eq_bm[tid - kBitmapWords] = 0;
            kmax = __reduce_max_sync(0xffffffffu, kmax);
            if (lane == 0) sm.warp_max[warp] = kmax;
        }
        __syncthreads();
        uint32_t mkey = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mkey = max(mkey, sm.warp_max[w]);

        // ---- radix select of the 64th largest key ---------------------------------------
#pragma unroll
        for (int i = 0; i < kPer; ++i) atomicAdd(&sm.hist[0][key[i] >> 20], 1u);
        __syncthreads();
        find_digit<2048>(sm, sm.hist[0], kTopK, tid, lane, warp);
        __syncthreads();
        uint32_t need = kTopK - sm.bcast[1];
        uint32_t prefix = sm.bcast[0] << 20;
        uint32_t pmask = 0x7ffu << 20;
        bool done = sm.bcast[2] == need;

        if (!done) {
            // hist[0] is free again: clear the 512 bins the last pass uses
            sm.hist[0][tid] = 0;
            sm.hist[0][tid + kThreads] = 0;
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if ((key[i] & pmask) == prefix) atomicAdd(&sm.hist[1][(key[i] >> 9) & 0x7ffu], 1u);
            __syncthreads();
            find_digit<2048>(sm, sm.hist[1], need, tid, lane, warp);
            __syncthreads();
            need -= sm.bcast[1];
            prefix |= sm.bcast[0] << 9;
            pmask |= 0x7ffu << 9;
            done = sm.bcast[2] == need;
        }
        if (!done) {
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if ((key[i] & pmask) == prefix) atomicAdd(&sm.hist[0][key[i] & 0x1ffu], 1u);
            __syncthreads();
            find_digit<512>(sm, sm.hist[0], need, tid, lane, warp);
            __syncthreads();
            need -= sm.bcast[1];
            prefix |= sm.bcast[0];
            pmask = 0x7fffffffu;
        }

        // ---- mark keys above the threshold prefix, and the tie candidates ---------------
#pragma unroll
        for (int v = 0; v < kVec; ++v)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t mk = key[4 * v + u] & pmask;
                const int j = v * 1024 + 4 * tid + u;
                if (mk > prefix) atomicOr(&sm.sel_bm[j >> 5], 1u << (j & 31));
                else if (mk == prefix) atomicOr(&sm.eq_bm[j >> 5], 1u << (j & 31));
            }
        __syncthreads();

        // ---- one warp: take the first `need` ties, compact the 64 indices ascending ------
        if (warp == 0) {
            uint32_t eqw[4];
            uint32_t cnt = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                eqw[q] = sm.eq_bm[4 * lane + q];
                cnt += __popc(eqw[q]);
            }
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t before = incl - cnt;
            uint32_t take = need > before ? min(need - before, cnt) : 0u;
            uint32_t fin[4];
            uint32_t fcnt = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w = eqw[q];
                uint32_t kept = 0;
                while (take != 0u && w != 0u) {
                    const uint32_t low = w & (0u - w);
                    kept |= low;
                    w ^= low;
                    --take;
                }
                fin[q] = sm.sel_bm[4 * lane + q] | kept;
                sm.fin_bm[4 * lane + q] = fin[q];
                fcnt += __popc(fin[q]);
            }
            uint32_t pos = fcnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, pos, o);
                if (lane >= o) pos += y;
            }
            pos -= fcnt;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w = fin[q];
                while (w != 0u) {
                    const int b = __ffs(w) - 1;
                    if (pos < kTopK) sm.sel_idx[pos] = static_cast<uint16_t>(128 * lane + 32 * q + b);
                    ++pos;
                    w &= w - 1u;
                }
            }
            if (lane == 0) sm.scale = __fdiv_rn(__uint_as_float(mkey), 1.5f);
        }
        __syncthreads();

        // ---- owners: codes and residuals; store the error buffer once -------------------
        const float s = sm.scale;
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            const int j0 = v * 1024 + 4 * tid;
            const uint32_t bits = sm.fin_bm[j0 >> 5] >> (j0 & 31);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if ((bits >> u) & 1u) {
                    const uint32_t code = quant_code(a[4 * v + u], s);
                    a[4 * v + u] = __fsub_rn(a[4 * v + u], level_value(code, s));
                    sm.code_at[j0 + u] = static_cast<uint8_t>(code);
                }
            }
        }
        if (full) {
#pragma unroll
            for (int v = 0; v < kVec; ++v)
                st_stream_f4(ef + v * 1024 + 4 * tid,
                             make_float4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]));
        } else {
#pragma unroll
            for (int v = 0; v < kVec; ++v)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = v * 1024 + 4 * tid + u;
                    if (j < valid) ef[j] = a[4 * v + u];
                }
        }
        __syncthreads();

        // ---- one warp: pack the record and write the scale ------------------------------
        if (warp == 0) {
            const uint32_t i0 = sm.sel_idx[lane];
            const uint32_t i1 = sm.sel_idx[lane + 32];
            const uint32_t f0 = sm.code_at[i0] | (i0 << 2);
            const uint32_t f1 = sm.code_at[i1] | (i1 << 2);
            const uint32_t word = record_word(f0, f1, lane);
            store_record(payload + c * kRecordBytes, word, lane);
            if (lane == 0) scales[c] = s;
        }
    }
    if (nonfinite && flags != nullptr) atomicOr(flags, kFlagNonFinite);
}

}  // namespace

cudaError_t launch_ef_compress(const CompressTable& tab, bool bf16, float beta,
                               uint8_t* payload, float* scales, uint32_t* flags,
                               cudaStream_t stream) {
    const int64_t total = tab.chunk_begin[tab.num];
    if (total == 0) return cudaSuccess;
    const void* kern = bf16 ? reinterpret_cast<const void*>(&k_ef_compress<true>)
                            : reinterpret_cast<const void*>(&k_ef_compress<false>);
    const int resident = persistent_grid(kern, kThreads, 0);
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    const int grid = static_cast<int>(total < resident ? total : resident);
    if (bf16)
        k_ef_compress<true><<<grid, kThreads, 0, stream>>>(tab, beta, payload, scales, flags);
    else
        k_ef_compress<false><<<grid, kThreads, 0, stream>>>(tab, beta, payload, scales, flags);
    return cudaGetLastError();
}

}  // namespace spl
