// Fused sender kernel of the SparseLoCo codec: error feedback, chunk top-64, 2-bit quantise,
// 14-bit field packing and the error-feedback residual, in one pass over HBM.  Templated on
// the codec (chunk length L, k, scale rule), the delta type and where the error buffer lives;
// the translation units that include this header instantiate it (the default codec in
// ef_compress.cu, the variants in ef_compress_variants.cu).
//
// Method: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
// Pre-Training", "SparseLoCo: Three Compression Levers in One Pass" (items 1-3, per-chunk
// equation) and "Why Extreme Sparsity Doesn't Break Convergence" ("Error feedback
// accumulation": what is not sent stays in the buffer for the next round).
//
// Design (HBM-bound: 8 B read + 4 B written per fp32 value, 116 B written per chunk):
//   - one 256-thread CTA per 4096-value chunk (L values for a variant; the figures below are
//     the default codec's), grid-stride over chunks with a persistent grid
//     (SMs x resident CTAs); while a chunk is worked on, the next chunk's error buffer and
//     delta fly into a shared-memory stage as two 1-D bulk copies (TMA, no multicast, no
//     cluster) completing on an mbarrier, whose wait is bounded in time;
//   - each thread takes 16 values from the stage into registers (four 16-byte vectors at
//     chunk offsets v*1024 + 4*tid), forms a = fma(beta, e, delta) and the 31-bit magnitude
//     keys, and keeps them there for the whole chunk; the error buffer is written back once,
//     from registers, with streaming stores;
//   - the 64th-largest key: a shared-memory histogram of 2048 bins of 1/128 octave over the
//     16 octaves below the chunk's largest key; warp 0 finds the bin holding the 64th key
//     among the top 512 bins (a block-wide search over all 2048 runs only when those hold
//     fewer than 64 keys); keys above that bin are marked chosen, and the bin's own keys are
//     taken whole or, up to 64 of them, ranked by warp 0 (magnitude, then index); any other
//     chunk (a non-finite value, the 64th key more than 16 octaves below the largest, more
//     than 64 keys in its bin) takes an out-of-line radix select over key bits [30:20],
//     [19:9] and [8:0] with ties to the lowest indices; the chosen positions end up in a
//     4096-bit shared bitmap;
//   - one warp turns the bitmap into per-word prefix counts, from which every thread that
//     owns a chosen value knows its rank in ascending index order; it writes the value and
//     its position to shared memory by rank, and every thread stores its error-buffer values
//     unchanged; the last warp, at the top of the next iteration behind the barrier that
//     already follows the owner step (overlapping the histogram), codes the 64 entries,
//     writes their residuals over the stored values, assembles the 112-byte record (28
//     words) and stores it as seven 16-byte vectors; five block barriers per chunk in all;
//   - mean-abs scale (variant): the same, the last warp first forming the scale (pairwise sum
//     in ascending index order, divided by k);
//   - error buffer in host memory, and k = 128 under the max-abs rule: the owners code their
//     values and form the residuals in registers instead (the host buffer then crosses the
//     link once, in whole vectors; the packing warp's work stays short).
#pragma once

#include <type_traits>

#include "spl_device.cuh"
#include "spl_kernels.h"

namespace spl {
namespace {

constexpr uint32_t kWindow = (2048u << 16) - 1u;   // 16 octaves of magnitude keys: 2048 bins
constexpr uint32_t kNotFound = 0xffffffffu;

// Per-codec sizes of the sender.  A CTA of L / 16 threads works on one chunk, 16 values per
// thread (default: 256 threads, 4 vectors per thread, 128 bitmap words, 4 per lane of warp 0),
// and 1024 / threads CTAs share an SM (64 registers per thread, 32 warps per SM).
template <class Geo>
struct SendShape {
    static constexpr int kChunk = Geo::kChunk;
    static constexpr int kTopK = Geo::kTopK;
    static constexpr int kThreads = kChunk / 16;
    static constexpr int kWarps = kThreads / 32;
    static constexpr int kPer = kChunk / kThreads;       // values per thread
    static constexpr int kVec = kPer / 4;                // vectors of 4 per thread
    static constexpr int kStride = 4 * kThreads;         // between a thread's vectors
    static constexpr int kBitmapWords = kChunk / 32;
    static constexpr int kWordsPerLane = kBitmapWords / 32;
    static constexpr int kMinBlocks = 1024 / kThreads;
    static_assert(kPer % 4 == 0 && kThreads % 32 == 0 && 2048 % kThreads == 0, "sender shape");
};

template <class Geo, int kRule>
struct Smem {
    using S = SendShape<Geo>;
    float stage_e[S::kChunk];          // prefetched error-buffer chunk (bulk copy)
    uint32_t stage_d[S::kChunk];       // prefetched delta chunk: fp32, or bf16 in the first half
    uint32_t hist[2048];               // histogram bins (one select pass at a time)
    uint32_t sel_bm[S::kBitmapWords];  // chosen positions (complete once the select is done)
    uint32_t eq_bm[S::kBitmapWords];   // ties at the final threshold (many-candidate path)
    uint32_t warp_tot[S::kWarps];
    uint32_t warp_max[S::kWarps];
    uint32_t bcast[3];                 // digit, count above the digit's bin, count in the bin
    uint2 cand[64];                    // (key, index) of the keys in the boundary bin
    uint32_t ncand;
    uint16_t fields[S::kTopK];         // the record's fields, in ascending index order
    float vals[S::kTopK];              // the chosen a by rank (coded once the record is packed)
    uint32_t full_scan;                // the k-th key lies below the top 512 bins
    alignas(16) uint16_t pre[S::kBitmapWords];   // chosen positions before each bitmap word
    uint64_t bar;                      // completes when the stage's bulk copies have landed
};

// Block-wide search of the bin holding the need-th largest key (counting from the top bin).
// Thread t owns bins [kBinsPer*t, kBinsPer*t + kBinsPer).  Writes sm.bcast; the caller
// synchronises before reading it.
template <int kBins, class S, class Sm>
__device__ __forceinline__ void find_digit(Sm& sm, const uint32_t* hist, uint32_t need,
                                           int tid, int lane, int warp) {
    constexpr int kWarps = S::kWarps;
    constexpr int kBinsPer = kBins / S::kThreads;
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

// Warp 0: the bin holding the need-th largest key, searched among the top 512 of the 2048
// bins (the 4 octaves below the largest key), where it lies for all but very heavy-tailed
// chunks.  Writes sm.bcast and returns true, or returns false (for the whole warp) when those
// bins hold fewer than need keys.  Spares the block-wide search and its two barriers.
template <class Sm>
__device__ __forceinline__ bool top_digit(Sm& sm, uint32_t need, int lane) {
    constexpr int kTop = 512;
    constexpr int kBase = 2048 - kTop;
    constexpr int kPerLane = kTop / 32;
    uint32_t h[kPerLane];
    uint32_t sum = 0;
    const uint4* h4 = reinterpret_cast<const uint4*>(&sm.hist[kBase + kPerLane * lane]);
#pragma unroll
    for (int q = 0; q < kPerLane / 4; ++q) {
        const uint4 v = h4[q];
        h[4 * q + 0] = v.x;
        h[4 * q + 1] = v.y;
        h[4 * q + 2] = v.z;
        h[4 * q + 3] = v.w;
        sum += v.x + v.y + v.z + v.w;
    }
    uint32_t incl = sum;   // suffix sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
    }
    if (__shfl_sync(0xffffffffu, incl, 0) < need) return false;
    const uint32_t excl = incl - sum;
    if (excl < need && incl >= need) {
        uint32_t run = excl;
#pragma unroll
        for (int i = kPerLane - 1; i >= 0; --i) {
            if (run + h[i] >= need) {
                sm.bcast[0] = kBase + kPerLane * lane + i;
                sm.bcast[1] = run;
                sm.bcast[2] = h[i];
                break;
            }
            run += h[i];
        }
    }
    return true;
}

// The chunk a CTA works on: its tensor's pointers advanced to the chunk, and its extent.
struct ChunkRef {
    const void* delta;
    float* ef;
    int valid;
    bool full;
};

template <int kChunk, bool kBf16>
__device__ __forceinline__ ChunkRef locate(const CompressTable& tab, int64_t c) {
    int t = 0;
    int hi = tab.num;
    while (hi - t > 1) {
        const int mid = (t + hi) >> 1;
        if (tab.chunk_begin[mid] <= c) t = mid; else hi = mid;
    }
    const int64_t base = (c - tab.chunk_begin[t]) * kChunk;
    const int64_t n = tab.n[t];
    ChunkRef r;
    r.ef = tab.ef[t] + base;
    r.delta = kBf16
        ? static_cast<const void*>(static_cast<const uint16_t*>(tab.delta[t]) + base)
        : static_cast<const void*>(static_cast<const float*>(tab.delta[t]) + base);
    r.full = base + kChunk <= n;
    r.valid = r.full ? kChunk : static_cast<int>(n - base);
    return r;
}

// One thread: start the bulk copies of a full chunk's error buffer and delta into the stage.
// With the error buffer in host memory (kEfHost) only delta is staged: the buffer is read and
// written over the host link with plain 16-byte accesses.
template <int kChunk, bool kBf16, bool kEfHost, class Sm>
__device__ __forceinline__ void prefetch(Sm& sm, const ChunkRef& r) {
    constexpr uint32_t kDeltaBytes = kChunk * (kBf16 ? 2 : 4);
    fence_async_smem();
    mbar_expect_tx(&sm.bar, (kEfHost ? 0u : kChunk * 4u) + kDeltaBytes);
    if constexpr (!kEfHost) bulk_load(sm.stage_e, r.ef, kChunk * 4, &sm.bar);
    bulk_load(sm.stage_d, r.delta, kDeltaBytes, &sm.bar);
}

// a = fmaf(beta, e, delta) for this thread's 16 values, from the stage (full chunks); with
// the error buffer in host memory, e comes straight from there.
template <class S, bool kBf16, bool kEfHost, class Sm>
__device__ __forceinline__ void accumulate_from_stage(const Sm& sm, const ChunkRef& r,
                                                      float beta, int tid, float (&a)[S::kPer]) {
    constexpr int kVec = S::kVec;
    float4 eh[kVec];
    if constexpr (kEfHost) {
#pragma unroll
        for (int v = 0; v < kVec; ++v) eh[v] = ld_stream_f4(r.ef + v * S::kStride + 4 * tid);
    }
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
        const int j0 = v * S::kStride + 4 * tid;
        const float4 e4 = kEfHost ? eh[v] : *reinterpret_cast<const float4*>(&sm.stage_e[j0]);
        float d[4];
        if constexpr (kBf16) {
            const uint2 d2 = *reinterpret_cast<const uint2*>(
                reinterpret_cast<const uint16_t*>(sm.stage_d) + j0);
            d[0] = bf16_bits_to_float(d2.x & 0xffffu);
            d[1] = bf16_bits_to_float(d2.x >> 16);
            d[2] = bf16_bits_to_float(d2.y & 0xffffu);
            d[3] = bf16_bits_to_float(d2.y >> 16);
        } else {
            const float4 d4 = *reinterpret_cast<const float4*>(&sm.stage_d[j0]);
            d[0] = d4.x; d[1] = d4.y; d[2] = d4.z; d[3] = d4.w;
        }
        a[4 * v + 0] = __fmaf_rn(beta, e4.x, d[0]);
        a[4 * v + 1] = __fmaf_rn(beta, e4.y, d[1]);
        a[4 * v + 2] = __fmaf_rn(beta, e4.z, d[2]);
        a[4 * v + 3] = __fmaf_rn(beta, e4.w, d[3]);
    }
}

// The same for a tail chunk, straight from global memory; pads are +0.
template <class S, bool kBf16>
__device__ __forceinline__ void accumulate_tail(const ChunkRef& r, float beta, int tid,
                                                float (&a)[S::kPer]) {
#pragma unroll
    for (int v = 0; v < S::kVec; ++v)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = v * S::kStride + 4 * tid + u;
            float d = 0.0f, e = 0.0f;
            if (j < r.valid) {
                e = r.ef[j];
                d = kBf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(r.delta)[j])
                          : static_cast<const float*>(r.delta)[j];
            }
            a[4 * v + u] = j < r.valid ? __fmaf_rn(beta, e, d) : 0.0f;
        }
}

// Generic select (any data): radix passes on key bits [30:20], [19:9] and [8:0], each over
// the keys matching the digits found so far, stopping once the boundary bin is taken whole;
// ties at the final threshold go to the lowest indices.  Marks the 64 chosen positions in
// sm.sel_bm.  Entered by all threads with sm.sel_bm/eq_bm cleared; clears hist itself.
template <class Geo, class Sm>
__device__ __noinline__ void generic_select(Sm& sm, const uint32_t (&key)[SendShape<Geo>::kPer],
                                            int tid, int lane, int warp) {
    using S = SendShape<Geo>;
    constexpr int kPer = S::kPer;
    constexpr int kVec = S::kVec;
    constexpr int kThreads = S::kThreads;
    constexpr int kStride = S::kStride;
    constexpr uint32_t kTopK = S::kTopK;
    {
        uint4* h4 = reinterpret_cast<uint4*>(&sm.hist[0]);
#pragma unroll
        for (int i = 0; i < 512 / kThreads; ++i) h4[tid + i * kThreads] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPer; ++i) atomicAdd(&sm.hist[key[i] >> 20], 1u);
    __syncthreads();
    find_digit<2048, S>(sm, sm.hist, kTopK, tid, lane, warp);
    __syncthreads();
    uint32_t need = kTopK - sm.bcast[1];      // keys still to take from bin D
    const uint32_t dig = sm.bcast[0];
    const uint32_t in_bin = sm.bcast[2];

    if (in_bin == need) {
        // ---- bin D is taken whole: every key at or above it is in -------------------
#pragma unroll
        for (int v = 0; v < kVec; ++v)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = v * kStride + 4 * tid + u;
                if ((key[4 * v + u] >> 20) >= dig) atomicOr(&sm.sel_bm[j >> 5], 1u << (j & 31));
            }
        __syncthreads();
    } else {
        // ---- resolve bin D: radix passes on key bits [19:9] and [8:0] ---------------
        uint32_t prefix = dig << 20;
        uint32_t pmask = 0x7ffu << 20;
        {   // the first pass's bins have been read: clear them for the second pass
            uint4* h4 = reinterpret_cast<uint4*>(&sm.hist[0]);
#pragma unroll
            for (int i = 0; i < 512 / kThreads; ++i) h4[tid + i * kThreads] = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if ((key[i] & pmask) == prefix) atomicAdd(&sm.hist[(key[i] >> 9) & 0x7ffu], 1u);
        __syncthreads();
        find_digit<2048, S>(sm, sm.hist, need, tid, lane, warp);
        __syncthreads();
        need -= sm.bcast[1];
        prefix |= sm.bcast[0] << 9;
        pmask |= 0x7ffu << 9;
        if (sm.bcast[2] != need) {
#pragma unroll
            for (int i = 0; i < 512 / kThreads; ++i)   // the second pass's bins have been read
                sm.hist[tid + i * kThreads] = 0;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if ((key[i] & pmask) == prefix) atomicAdd(&sm.hist[key[i] & 0x1ffu], 1u);
            __syncthreads();
            find_digit<512, S>(sm, sm.hist, need, tid, lane, warp);
            __syncthreads();
            need -= sm.bcast[1];
            prefix |= sm.bcast[0];
            pmask = 0x7fffffffu;
        }
        // keys above the final prefix are in; ties at it go by index, lowest first
#pragma unroll
        for (int v = 0; v < kVec; ++v)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t mk = key[4 * v + u] & pmask;
                const int j = v * kStride + 4 * tid + u;
                if (mk > prefix) atomicOr(&sm.sel_bm[j >> 5], 1u << (j & 31));
                else if (mk == prefix) atomicOr(&sm.eq_bm[j >> 5], 1u << (j & 31));
            }
        __syncthreads();
        if (warp == 0) {
            constexpr int kWpl = S::kWordsPerLane;
            uint32_t eqw[kWpl];
            uint32_t cnt = 0;
#pragma unroll
            for (int qq = 0; qq < kWpl; ++qq) {
                eqw[qq] = sm.eq_bm[kWpl * lane + qq];
                cnt += __popc(eqw[qq]);
            }
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t before = incl - cnt;
            uint32_t take = need > before ? min(need - before, cnt) : 0u;
#pragma unroll
            for (int qq = 0; qq < kWpl; ++qq) {
                uint32_t w = eqw[qq];
                uint32_t kept = 0;
                while (take != 0u && w != 0u) {
                    const uint32_t low = w & (0u - w);
                    kept |= low;
                    w ^= low;
                    --take;
                }
                sm.sel_bm[kWpl * lane + qq] |= kept;
            }
        }
        __syncthreads();
    }
}

// Writes a record of kWords words held one per lane (word w0 + lane) at rec + 4 * w0: as
// 16-byte vectors when records are 16-byte aligned, else as words.  Called by all 32 lanes.
template <int kWords, bool kVec>
__device__ __forceinline__ void store_words(uint8_t* rec, int w0, uint32_t word, int lane) {
    const int cnt = kWords - w0 < 32 ? kWords - w0 : 32;
    if constexpr (kVec) {
        const int nv = cnt / 4;
        const int b = 4 * (lane < nv ? lane : 0);
        uint4 v;
        v.x = __shfl_sync(0xffffffffu, word, b + 0);
        v.y = __shfl_sync(0xffffffffu, word, b + 1);
        v.z = __shfl_sync(0xffffffffu, word, b + 2);
        v.w = __shfl_sync(0xffffffffu, word, b + 3);
        if (lane < nv) reinterpret_cast<uint4*>(rec + 4 * w0)[lane] = v;
    } else {
        if (lane < cnt) reinterpret_cast<uint32_t*>(rec)[w0 + lane] = word;
    }
}

// One warp: assemble a record from the fields in shared memory and store it with its scale.
template <class Geo, class Sm>
__device__ __forceinline__ void pack_record(const Sm& sm, uint8_t* __restrict__ payload,
                                            float* __restrict__ scales, int64_t c, float s,
                                            int lane) {
    constexpr int kFieldBits = Geo::kFieldBits;
    constexpr int kRecordWords = Geo::kRecordWords;
#pragma unroll
    for (int w0 = 0; w0 < kRecordWords; w0 += 32) {
        const int w = w0 + lane < kRecordWords ? w0 + lane : kRecordWords - 1;
        const int r_first = (32 * w) / kFieldBits;
        const int r_last = (32 * w + 31) / kFieldBits;
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {   // a word touches at most 4 fields of >= 13 bits
            const int r = r_first + k;
            if (r <= r_last) {
                const uint32_t f = sm.fields[r];
                const int off = kFieldBits * r - 32 * w;
                word |= off >= 0 ? (f << off) : (f >> (-off));
            }
        }
        store_words<kRecordWords, Geo::kVecRecords>(payload + c * Geo::kRecordBytes, w0, word,
                                                     lane);
    }
    if (lane == 0) scales[c] = s;
}

// One warp: the scale, each chosen entry's code, its residual written over the error-buffer
// value stored earlier (pads excluded), and the record.  The scale comes from the chosen
// values: max-abs from the largest magnitude key among them (the chunk's largest key is always
// chosen, so this is the chunk maximum, NaN included); mean-abs from the pairwise sum of |a|
// over ranks 0..k-1 in ascending index order, divided by k (lane l first sums its k/32
// consecutive ranks the same way, then the lanes combine as a tree).  Runs after a barrier
// that follows the chunk's owner step and its error-buffer stores, so the residuals land last.
template <class Geo, int kRule, class Sm>
__device__ __forceinline__ void finish_record(Sm& sm, uint8_t* __restrict__ payload,
                                              float* __restrict__ scales, int64_t c, float* ef,
                                              int valid, int lane) {
    constexpr int kTopK = Geo::kTopK;
    constexpr int kPerLane = kTopK / 32;
    float x[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) x[i] = sm.vals[kPerLane * lane + i];
    float s;
    if constexpr (kRule == kScaleMax) {
        uint32_t kmax = 0;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) kmax = max(kmax, mag_key(x[i]));
        s = __fdiv_rn(__uint_as_float(__reduce_max_sync(0xffffffffu, kmax)), 1.5f);
    } else {
        float t[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) t[i] = fabsf(x[i]);
#pragma unroll
        for (int w = 1; w < kPerLane; w <<= 1)
#pragma unroll
            for (int i = 0; i + w < kPerLane; i += 2 * w) t[i] = __fadd_rn(t[i], t[i + w]);
        float sum = t[0];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
            sum = __fadd_rn(sum, __shfl_down_sync(0xffffffffu, sum, o));
        s = __fdiv_rn(__shfl_sync(0xffffffffu, sum, 0), static_cast<float>(kTopK));
    }
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int r = kPerLane * lane + i;
        const uint32_t code = quant_code(x[i], s);
        const uint32_t pos = static_cast<uint32_t>(sm.fields[r]) >> 2;
        sm.fields[r] = static_cast<uint16_t>(code | (pos << 2));
        if (static_cast<int>(pos) < valid) ef[pos] = __fsub_rn(x[i], level_value(code, s));
    }
    __syncwarp();
    pack_record<Geo>(sm, payload, scales, c, s, lane);
}

template <class Geo, int kRule, bool kBf16, bool kEfHost>
__global__ void __launch_bounds__(SendShape<Geo>::kThreads, SendShape<Geo>::kMinBlocks)
k_ef_compress(const CompressTable tab, float beta, uint8_t* __restrict__ payload,
              float* __restrict__ scales, uint32_t* __restrict__ flags) {
    using S = SendShape<Geo>;
    constexpr int kChunk = S::kChunk;
    constexpr int kTopK = S::kTopK;
    constexpr int kThreads = S::kThreads;
    constexpr int kWarps = S::kWarps;
    constexpr int kPer = S::kPer;
    constexpr int kVec = S::kVec;
    constexpr int kStride = S::kStride;
    constexpr int kBitmapWords = S::kBitmapWords;
    constexpr int kFieldBits = Geo::kFieldBits;
    constexpr int kRecordWords = Geo::kRecordWords;
    constexpr int kRecordBytes = Geo::kRecordBytes;
    // max-abs scale: the packing warp codes the chosen values and writes their residuals
    // (it overlaps the histogram), except where the owners do it cheaper in registers: with
    // the error buffer in host memory (k scattered 4-byte writes per chunk would cost the
    // host link more than the divergent owner step costs) and for k = 128 (four entries per
    // lane of the packing warp then outlast the histogram: +1 % at L = 4096, +4 % at 8192)
    constexpr bool kCodeInPlace = kRule == kScaleMax && (kEfHost || kTopK > 64);
    // the out-of-line select takes the keys through memory.  Handing it a copy made on that
    // path keeps the key registers from also being stored to the stack on every chunk (-4.5 %
    // at k = 64); where registers are scarcer (k = 128, a host error buffer) the copy makes
    // the compiler spill more in the loop instead, so there the keys are passed directly
    constexpr bool kCopyKeys = kTopK <= 64 && !kEfHost;
    using Sm = Smem<Geo, kRule>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t total = tab.chunk_begin[tab.num];
    if (static_cast<int64_t>(blockIdx.x) >= total) return;

    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        const ChunkRef r0 = locate<kChunk, kBf16>(tab, blockIdx.x);
        if (r0.full) prefetch<kChunk, kBf16, kEfHost>(sm, r0);
    }
    __syncthreads();

    uint32_t parity = 0;
    bool nonfinite = false;
    bool aborted = false;
    int64_t pend_c = -1;     // the chunk whose record the last warp still has to pack
    float pend_s = 0.0f;
    float* pend_ef = nullptr;   // mean-abs: that chunk's error buffer and extent
    int pend_valid = 0;

    for (int64_t c = blockIdx.x; c < total; c += gridDim.x) {
        const ChunkRef r = locate<kChunk, kBf16>(tab, c);

        // ---- a = beta * e + delta (from the prefetched stage), and the magnitude keys -----
        float a[kPer];
        bool timed_out = false;
        if (r.full) {
            timed_out = !mbar_wait(&sm.bar, parity);
            parity ^= 1u;
            accumulate_from_stage<S, kBf16, kEfHost>(sm, r, beta, tid, a);
        } else {
            accumulate_tail<S, kBf16>(r, beta, tid, a);
        }
        uint32_t key[kPer];
        uint32_t kmax = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            key[i] = mag_key(a[i]);
            kmax = max(kmax, key[i]);
        }
        nonfinite |= kmax >= kKeyInf;

        // ---- clear the histogram; chunk max ----------------------------------------------
        // (the previous chunk's select is done, and nothing reads the histogram after it)
        {
            uint4* h4 = reinterpret_cast<uint4*>(&sm.hist[0]);
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < 512 / kThreads; ++i) h4[tid + i * kThreads] = z;   // 2048 words
            if (tid == 0) {
                sm.ncand = 0;
                sm.bcast[0] = kNotFound;
            }
            kmax = __reduce_max_sync(0xffffffffu, kmax);
            if (lane == 0) sm.warp_max[warp] = kmax;
        }
        if (__syncthreads_or(timed_out)) {
            aborted = true;
            break;
        }
        // the stage has been read by every thread: start the next chunk's copies
        if (tid == 0 && c + gridDim.x < total) {
            const ChunkRef rn = locate<kChunk, kBf16>(tab, c + gridDim.x);
            if (rn.full) prefetch<kChunk, kBf16, kEfHost>(sm, rn);
        }
        // the previous chunk's owners have read the bitmaps (the barrier above follows their
        // step): clear them for this chunk's select, which first writes them two barriers on
        if constexpr (2 * kBitmapWords == kThreads) {
            if (tid < kBitmapWords) sm.sel_bm[tid] = 0;
            else sm.eq_bm[tid - kBitmapWords] = 0;
        } else {
            for (int i = tid; i < 2 * kBitmapWords; i += kThreads) {
                if (i < kBitmapWords) sm.sel_bm[i] = 0;
                else sm.eq_bm[i - kBitmapWords] = 0;
            }
        }
        // the last warp packs the previous chunk's record: its fields are complete (the
        // barrier above follows that chunk's owner step) and are next written after this
        // chunk's select
        if (warp == kWarps - 1 && pend_c >= 0) {
            if constexpr (kCodeInPlace)
                pack_record<Geo>(sm, payload, scales, pend_c, pend_s, lane);
            else
                finish_record<Geo, kRule>(sm, payload, scales, pend_c, pend_ef, pend_valid, lane);
        }
        uint32_t mkey = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mkey = max(mkey, sm.warp_max[w]);

        // ---- select, fast path: 2048 bins of 1/128 octave over the 16 octaves below the
        //      largest key; the 64th key almost always falls inside, and its bin holds only a
        //      few keys, which warp 0 ranks directly.  Otherwise: the generic radix select.
        //      (A narrower first window does not pay: with ~10 % of the keys inside it, nearly
        //      every warp still has a lane that takes the in-window path.)
        // lo_key puts the largest key exactly in the top bin, so no key needs clamping
        const bool windowed = mkey < kKeyInf;
        const uint32_t lo_key = mkey > kWindow ? mkey - kWindow : 0u;
        if (windowed) {
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if (key[i] >= lo_key) atomicAdd(&sm.hist[(key[i] - lo_key) >> 16], 1u);
        }
        __syncthreads();
        if (windowed && warp == 0) {
            const bool found = top_digit(sm, kTopK, lane);
            if (lane == 0) sm.full_scan = found ? 0u : 1u;
        }
        __syncthreads();
        if (windowed && sm.full_scan != 0u) {   // uniform: every thread read the same flag
            find_digit<2048, S>(sm, sm.hist, kTopK, tid, lane, warp);
            __syncthreads();
        }
        bool selected = false;
        if (windowed && sm.bcast[0] != kNotFound) {
            const uint32_t need = kTopK - sm.bcast[1];
            const uint32_t dig = sm.bcast[0];
            const uint32_t in_bin = sm.bcast[2];
            if (in_bin == need || in_bin <= 64u) {
                const bool rank_bin = in_bin != need;
                // bin D as a key range [k_lo, k_hi): keys at or above k_hi are in, keys in the
                // range are in when the bin is taken whole, else they are the candidates
                const uint32_t k_lo = lo_key + (dig << 16);
                const uint32_t k_hi = k_lo + (1u << 16);
                const uint32_t k_in = rank_bin ? k_hi : k_lo;
#pragma unroll
                for (int v = 0; v < kVec; ++v) {
                    // a vector's four positions share one bitmap word: one OR per vector
                    const int j0 = v * kStride + 4 * tid;
                    uint32_t nib = 0;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t kk = key[4 * v + u];
                        if (kk >= k_in) {
                            nib |= 1u << u;
                        } else if (kk >= k_lo) {
                            const uint32_t slot = atomicAdd(&sm.ncand, 1u);
                            if (slot < 64u) sm.cand[slot] = make_uint2(kk, static_cast<uint32_t>(j0 + u));
                        }
                    }
                    if (nib != 0u) atomicOr(&sm.sel_bm[j0 >> 5], nib << (j0 & 31));
                }
                __syncthreads();
                if (rank_bin && warp == 0) {
                    // rank each candidate among the bin's keys (magnitude, then index)
                    if (in_bin <= 32u) {
                        const uint2 me = static_cast<uint32_t>(lane) < in_bin ? sm.cand[lane] : make_uint2(0u, 0u);
                        uint32_t rank = 0;
                        for (uint32_t o = 0; o < in_bin; ++o) {
                            const uint32_t ok = __shfl_sync(0xffffffffu, me.x, o);
                            const uint32_t oj = __shfl_sync(0xffffffffu, me.y, o);
                            rank += (ok > me.x || (ok == me.x && oj < me.y)) ? 1u : 0u;
                        }
                        if (static_cast<uint32_t>(lane) < in_bin && rank < need)
                            atomicOr(&sm.sel_bm[me.y >> 5], 1u << (me.y & 31));
                    } else {   // 33..64 candidates (dense tops): two per lane
                        const uint2 m0 = sm.cand[lane];
                        const uint2 m1 = static_cast<uint32_t>(lane) + 32u < in_bin ? sm.cand[lane + 32] : make_uint2(0u, 0u);
                        uint32_t r0 = 0, r1 = 0;
                        for (uint32_t o = 0; o < in_bin; ++o) {
                            const uint32_t src = o & 31u;
                            const uint32_t k0 = __shfl_sync(0xffffffffu, m0.x, src);
                            const uint32_t j0 = __shfl_sync(0xffffffffu, m0.y, src);
                            const uint32_t k1 = __shfl_sync(0xffffffffu, m1.x, src);
                            const uint32_t j1 = __shfl_sync(0xffffffffu, m1.y, src);
                            const uint32_t ok = o < 32u ? k0 : k1;
                            const uint32_t oj = o < 32u ? j0 : j1;
                            r0 += (ok > m0.x || (ok == m0.x && oj < m0.y)) ? 1u : 0u;
                            r1 += (ok > m1.x || (ok == m1.x && oj < m1.y)) ? 1u : 0u;
                        }
                        if (r0 < need) atomicOr(&sm.sel_bm[m0.y >> 5], 1u << (m0.y & 31));
                        if (static_cast<uint32_t>(lane) + 32u < in_bin && r1 < need)
                            atomicOr(&sm.sel_bm[m1.y >> 5], 1u << (m1.y & 31));
                    }
                    __syncwarp();
                }
                selected = true;
            }
        }
        if (!selected) {
            if constexpr (kCopyKeys) {
                uint32_t key_mem[kPer];
#pragma unroll
                for (int i = 0; i < kPer; ++i) key_mem[i] = key[i];
                generic_select<Geo>(sm, key_mem, tid, lane, warp);
            } else {
                generic_select<Geo>(sm, key, tid, lane, warp);
            }
        }

        // ---- warp 0: chosen positions before each bitmap word ----------------------------
        if (warp == 0) {
            if constexpr (S::kWordsPerLane == 4) {
                const uint4 w4 = *reinterpret_cast<const uint4*>(&sm.sel_bm[4 * lane]);
                const uint32_t c0 = __popc(w4.x), c1 = __popc(w4.y), c2 = __popc(w4.z);
                const uint32_t mine = c0 + c1 + c2 + __popc(w4.w);
                uint32_t incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t p0 = incl - mine;
                *reinterpret_cast<uint2*>(&sm.pre[4 * lane]) =
                    make_uint2(p0 | ((p0 + c0) << 16), (p0 + c0 + c1) | ((p0 + c0 + c1 + c2) << 16));
            } else {
                constexpr int kWpl = S::kWordsPerLane;
                uint32_t cnt[kWpl];
                uint32_t mine = 0;
#pragma unroll
                for (int q = 0; q < kWpl; ++q) {
                    cnt[q] = __popc(sm.sel_bm[kWpl * lane + q]);
                    mine += cnt[q];
                }
                uint32_t incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                uint32_t run = incl - mine;
#pragma unroll
                for (int q = 0; q < kWpl; ++q) {
                    sm.pre[kWpl * lane + q] = static_cast<uint16_t>(run);
                    run += cnt[q];
                }
            }
        }
        __syncthreads();

        // ---- owners: rank and value of each chosen value (the last warp codes them and
        //      writes their residuals; with a host error buffer, code and residual here) -----
        float s = 0.0f;   // coding in place: the max-abs scale
        if constexpr (kCodeInPlace) s = __fdiv_rn(__uint_as_float(mkey), 1.5f);
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            const int j0 = v * kStride + 4 * tid;
            const uint32_t word = sm.sel_bm[j0 >> 5];
            const int sh = j0 & 31;
            if (((word >> sh) & 0xfu) == 0u) continue;
            const uint32_t base_rank = sm.pre[j0 >> 5];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if ((word >> (sh + u)) & 1u) {
                    const uint32_t rank = base_rank + __popc(word & ((1u << (sh + u)) - 1u));
                    if constexpr (kCodeInPlace) {
                        const uint32_t code = quant_code(a[4 * v + u], s);
                        a[4 * v + u] = __fsub_rn(a[4 * v + u], level_value(code, s));
                        if (rank < kTopK)
                            sm.fields[rank] = static_cast<uint16_t>(code | (static_cast<uint32_t>(j0 + u) << 2));
                    } else if (rank < kTopK) {
                        sm.vals[rank] = a[4 * v + u];
                        sm.fields[rank] = static_cast<uint16_t>(static_cast<uint32_t>(j0 + u) << 2);
                    }
                }
            }
        }
        if (r.full) {
#pragma unroll
            for (int v = 0; v < kVec; ++v)
                st_stream_f4(r.ef + v * kStride + 4 * tid,
                             make_float4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]));
        } else {
#pragma unroll
            for (int v = 0; v < kVec; ++v)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = v * kStride + 4 * tid + u;
                    if (j < r.valid) r.ef[j] = a[4 * v + u];
                }
        }

        // ---- the record is packed by the last warp at the top of the next iteration ------
        pend_c = c;
        pend_s = s;
        pend_ef = r.ef;
        pend_valid = r.valid;
    }
    __syncthreads();   // the last chunk's fields (and error-buffer stores) are complete
    if (warp == kWarps - 1 && pend_c >= 0) {
        if constexpr (kCodeInPlace)
            pack_record<Geo>(sm, payload, scales, pend_c, pend_s, lane);
        else
            finish_record<Geo, kRule>(sm, payload, scales, pend_c, pend_ef, pend_valid, lane);
    }
    bool copy_pending = false;
    if (aborted && tid == 0) {
        // the copy that did not complete may still land: wait once more (bounded) before
        // the CTA's shared memory is released; if that wait runs out too, the block exits with
        // the copy possibly in flight, which the flags report
        copy_pending = !mbar_wait(&sm.bar, parity ^ 1u);
    }
    if (flags != nullptr) {
        if (nonfinite) atomicOr(flags, kFlagNonFinite);
        if (aborted && tid == 0) atomicOr(flags, kFlagTimeout | (copy_pending ? kFlagCopyPending : 0u));
    }
}

template <class Geo, int kRule, bool kBf16, bool kEfHost>
cudaError_t launch_compress(const CompressTable& tab, int64_t total, float beta, uint8_t* payload,
                            float* scales, uint32_t* flags, cudaStream_t stream) {
    const void* kern = reinterpret_cast<const void*>(&k_ef_compress<Geo, kRule, kBf16, kEfHost>);
    const size_t smem = sizeof(Smem<Geo, kRule>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    constexpr int kThreads = SendShape<Geo>::kThreads;
    const int resident = persistent_grid(kern, kThreads, smem);
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    const int grid = static_cast<int>(total < resident ? total : resident);
    k_ef_compress<Geo, kRule, kBf16, kEfHost><<<grid, kThreads, smem, stream>>>(tab, beta, payload,
                                                                                scales, flags);
    return cudaGetLastError();
}

// Launch for one codec (geometry and scale rule), over the delta type and error-buffer kind.
template <class Geo, int kRule>
cudaError_t launch_codec(const CompressTable& tab, bool bf16, bool ef_host, float beta,
                         uint8_t* payload, float* scales, uint32_t* flags, cudaStream_t stream) {
    const int64_t total = tab.chunk_begin[tab.num];
    if (total == 0) return cudaSuccess;
    if (ef_host) {
        if constexpr (std::is_same_v<Geo, DefaultGeometry> && kRule == kScaleMax) {
            return bf16 ? launch_compress<Geo, kRule, true, true>(tab, total, beta, payload, scales, flags, stream)
                        : launch_compress<Geo, kRule, false, true>(tab, total, beta, payload, scales, flags, stream);
        }
        return cudaErrorNotSupported;   // host-resident error buffers: default codec only
    }
    return bf16 ? launch_compress<Geo, kRule, true, false>(tab, total, beta, payload, scales, flags, stream)
                : launch_compress<Geo, kRule, false, false>(tab, total, beta, payload, scales, flags, stream);
}

}  // namespace
}  // namespace spl
