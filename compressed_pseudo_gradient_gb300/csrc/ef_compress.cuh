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
//     the default codec's) at a time, four resident per SM; the grid runs in waves of the
//     resident CTAs, each CTA taking 16 chunks spaced a wave apart, so the chunks in flight
//     stay close together in memory (1.86 ms per 2^30 values against 2.00 ms with one
//     persistent wave); while a chunk is worked on, the next chunk's error buffer and delta
//     fly into a shared-memory stage as two 1-D bulk copies (TMA, no multicast, no cluster)
//     completing on an mbarrier, whose wait is bounded in time;
//   - each thread takes 16 values from the stage into registers (four 16-byte vectors at
//     chunk offsets v*1024 + 4*tid), forms a = fma(beta, e, delta) and the 31-bit magnitude
//     keys, and stores a to the error buffer at once, unchanged (plain stores: the lines stay
//     in L2 for the read-back below); only the keys stay in registers;
//   - the 64th-largest key: a shared-memory histogram of 2048 bins of 1/128 octave over the
//     16 octaves below the chunk's largest key (one unconditional atomic per key); warp 0
//     finds the bin holding the 64th key among the top 512 bins (a block-wide search over all
//     2048 runs only when those hold fewer than 64 keys); marking is branch-free: keys above
//     that bin go into a 4096-bit chosen bitmap with predicated ORs, and the bin's own keys
//     are taken whole or, up to 64 of them, recorded in a tie bitmap and a key buffer and
//     ranked by warp 0 (magnitude, then index); any other chunk (a non-finite value, the 64th
//     key more than 16 octaves below the largest, more than 64 keys in its bin) takes an
//     out-of-line radix select over key bits [30:20], [19:9] and [8:0] with ties to the
//     lowest indices;
//   - the finish of a chunk overlaps the next chunk's select on warp groups: beside warp 0's
//     bin search the gather group turns the previous chunk's bitmap into positions by rank and
//     reads the chosen values back from the error buffer (cp.async, from L2); beside warp 0's
//     ranking the packing group codes them, writes their residuals over the stored values and
//     packs the record with shuffles (the mean-abs rule first forms the scale as a pairwise
//     sum in ascending index order); four block barriers per chunk;
//   - error buffer in host memory: only delta is staged, the buffer crosses the link once in
//     whole vectors, and the owners of the chosen values code them and form the residuals in
//     registers before that one store (k scattered writes per chunk over the link would cost
//     more); five barriers per chunk.
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

// kFast: the select's marking pass keeps the boundary bin's keys by position (keybuf) for the
// warp that ranks them, and the packing warp finds the chosen positions itself (no owner step).
template <class Geo, int kRule, bool kFast>
struct Smem {
    using S = SendShape<Geo>;
    float stage_e[S::kChunk];          // prefetched error-buffer chunk (bulk copy)
    uint32_t stage_d[S::kChunk];       // prefetched delta chunk: fp32, or bf16 in the first half
    uint32_t hist[2048];               // histogram bins (one select pass at a time)
    // chosen positions (complete once the select is done); kFast alternates two, one per
    // chunk, so the packing warp reads the previous chunk's while this chunk's is marked
    uint32_t sel_bm[kFast ? 2 : 1][S::kBitmapWords];
    uint32_t eq_bm[S::kBitmapWords];   // ties at the final threshold (many-candidate path)
    uint32_t warp_tot[S::kWarps];
    uint32_t warp_max[S::kWarps];
    uint32_t bcast[3];                 // digit, count above the digit's bin, count in the bin
    uint2 cand[64];                    // (key, index) of the keys in the boundary bin
    uint32_t ncand;
    uint16_t fields[S::kTopK];         // the record's fields, in ascending index order
    float vals[S::kTopK];              // kFast: the chosen values by rank, read back
    uint32_t gcount[8];                // kFast: chosen positions per gather warp
    float psum[4];                     // kFast, mean-abs: each packing warp's partial sum
    uint32_t full_scan;                // the k-th key lies below the top 512 bins
    alignas(16) uint16_t pre[S::kBitmapWords];   // chosen positions before each bitmap word
    // boundary-bin keys by position, as offsets from the bin's lowest key (kFast only)
    alignas(16) uint16_t keybuf[kFast ? S::kChunk : 8];
    const void* next_delta;            // the next chunk of this CTA, located by thread 0
    float* next_ef;
    int next_valid;
    int next_tensor;                   // thread 0: the tensor of the last chunk it located
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

// t: the tensor of the last chunk located by this caller; a CTA visits its chunks in
// increasing order, so the tensor index only moves forward (past empty tensors too).
template <int kChunk, bool kBf16>
__device__ __forceinline__ ChunkRef locate(const CompressTable& tab, int64_t c, int& t) {
    while (t + 1 < tab.num && tab.chunk_begin[t + 1] <= c) ++t;
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
    if (!SPL_CHECK(r.full, kSiteBulk, r.valid)) return;
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
        if (!SPL_CHECK(j0 + 3 < S::kChunk, kSiteStage, j0)) continue;
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
            if (j < r.valid && SPL_CHECK(r.valid <= S::kChunk, kSiteTail, r.valid)) {
                e = r.ef[j];
                d = kBf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(r.delta)[j])
                          : static_cast<const float*>(r.delta)[j];
            }
            a[4 * v + u] = j < r.valid ? __fmaf_rn(beta, e, d) : 0.0f;
        }
}

// Shared-memory OR of v into *w when v is nonzero, as one predicated instruction (no branch:
// the marking pass runs it for every vector of four values).
__device__ __forceinline__ void red_or_nonzero(uint32_t* w, uint32_t v) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "@p red.shared.or.b32 [%0], %1;\n\t}" ::"r"(smem_addr(w)), "r"(v)
        : "memory");
}

// Shared-memory 16-bit store of v when keep is set, as one predicated instruction.
__device__ __forceinline__ void st_u16_if(uint16_t* p, uint32_t v, bool keep) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t"
        "@p st.shared.u16 [%0], %1;\n\t}" ::"r"(smem_addr(p)), "h"(static_cast<uint16_t>(v)),
        "r"(keep ? 1u : 0u)
        : "memory");
}

// This thread's 16 values of a chunk's error buffer (a tail chunk's pads are not stored).
template <class S, bool kEvictFirst>
__device__ __forceinline__ void store_error_buffer(const ChunkRef& r, const float (&a)[S::kPer],
                                                   int tid) {
    if (r.full) {
        // in HBM, plain stores, not evict-first ones: the fast flow's gather group reads the
        // 64 chosen values back one chunk later, and keeping the lines in L2 for that is worth
        // 1.3 % of the compress (2.012 -> 1.986 ms at 2^30); a host buffer is streamed
#pragma unroll
        for (int v = 0; v < S::kVec; ++v) {
            if (!SPL_CHECK(v * S::kStride + 4 * tid + 3 < S::kChunk, kSiteEfStore, 4 * tid)) continue;
            const float4 x = make_float4(a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
            if constexpr (kEvictFirst)
                st_stream_f4(r.ef + v * S::kStride + 4 * tid, x);
            else
                *reinterpret_cast<float4*>(r.ef + v * S::kStride + 4 * tid) = x;
        }
    } else {
#pragma unroll
        for (int v = 0; v < S::kVec; ++v)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = v * S::kStride + 4 * tid + u;
                if (j < r.valid && SPL_CHECK(r.valid <= S::kChunk, kSiteEfStore, r.valid))
                    r.ef[j] = a[4 * v + u];
            }
    }
}

// Generic select (any data): radix passes on key bits [30:20], [19:9] and [8:0], each over
// the keys matching the digits found so far, stopping once the boundary bin is taken whole;
// ties at the final threshold go to the lowest indices.  Marks the 64 chosen positions in
// sm.sel_bm[cur].  Entered by all threads with it and sm.eq_bm cleared; clears hist itself.
template <class Geo, class Sm>
__device__ __noinline__ void generic_select(Sm& sm, int cur,
                                            const uint32_t (&key)[SendShape<Geo>::kPer],
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
    for (int i = 0; i < kPer; ++i)
        if (SPL_CHECK((key[i] >> 20) < 2048u, kSiteGenericHist, key[i]))
            atomicAdd(&sm.hist[key[i] >> 20], 1u);
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
                if ((key[4 * v + u] >> 20) >= dig &&
                    SPL_CHECK((j >> 5) < S::kBitmapWords, kSiteBitmap, j))
                    atomicOr(&sm.sel_bm[cur][j >> 5], 1u << (j & 31));
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
                if (!SPL_CHECK((j >> 5) < S::kBitmapWords, kSiteBitmap, j)) continue;
                if (mk > prefix) atomicOr(&sm.sel_bm[cur][j >> 5], 1u << (j & 31));
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
                sm.sel_bm[cur][kWpl * lane + qq] |= kept;
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

// Named barrier among `threads` threads (a multiple of 32) of the CTA; ids 1.. (0 is
// __syncthreads).
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// kFast sizes: the gather group (the last kChunk / 1024 warps: one bitmap word per lane) turns
// a finished chunk's bitmap into positions by rank; the packing group (the last k / 32 warps:
// one rank per lane) codes and packs the record, warp p forming words [p b, p b + b) of the
// record from ranks [32 p, 32 p + 32), b the field width (32 fields of b bits fill b words).
template <class Geo>
struct FinishShape {
    static constexpr int kWarps = SendShape<Geo>::kWarps;
    static constexpr int kGatherWarps = SendShape<Geo>::kBitmapWords / 32;
    static constexpr int kPackWarps = Geo::kTopK / 32;
    static_assert(kGatherWarps < kWarps && kPackWarps < kWarps, "warp 0 is never in a group");
};

constexpr int kBarGather = 1;   // named barrier ids
constexpr int kBarPack = 2;

// kFast, the gather group (called by its warps only, g = the warp's index in the group): the
// positions of a finished chunk's chosen entries into sm.fields by rank (ascending position),
// from its bitmap sm.sel_bm[which] (complete behind a barrier that precedes this call), and
// asynchronous copies of their values, read back from the error buffer (where every thread
// stored the chunk's accumulated values unchanged), into sm.vals by rank; pads (past `valid`)
// are +0.  Clears the bitmap for a later chunk.  The copies are this thread's own: it waits for
// them (cp.async.wait_all) before the barrier after which the packing group reads them.
template <class Geo, class Sm>
__device__ __forceinline__ void gather_chosen(Sm& sm, int which, const float* ef, int valid,
                                              int g, int lane) {
    using F = FinishShape<Geo>;
    const int w = 32 * g + lane;
    uint32_t word = sm.sel_bm[which][w];
    sm.sel_bm[which][w] = 0u;
    const uint32_t cnt = __popc(word);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm.gcount[g] = incl;
    named_sync(kBarGather, 32 * F::kGatherWarps);
    uint32_t rank = incl - cnt;
    for (int h = 0; h < g; ++h) rank += sm.gcount[h];
    while (word != 0u) {
        const int b = __ffs(word) - 1;
        word &= word - 1u;
        const int pos = 32 * w + b;
        if (SPL_CHECK(rank < static_cast<uint32_t>(Geo::kTopK), kSiteFields, rank)) {
            sm.fields[rank] = static_cast<uint16_t>(pos);
            if (pos < valid) cp_async4(&sm.vals[rank], ef + pos);
            else sm.vals[rank] = 0.0f;
        }
        ++rank;
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// kFast, the packing group (called by its warps only, p = the warp's index in the group): rank
// r = 32 p + lane's code, its residual written over the stored value (pads excluded), and
// record words [p b, p b + b).  The scale: max-abs from the chunk's largest key (always among
// the chosen); mean-abs from the pairwise sum of |a| over ranks 0..k-1 in ascending order
// divided by k: each warp sums its 32 ranks pairwise (the tree over lanes), and the group
// combines the warps' sums as the upper levels of the same tree.
template <class Geo, int kRule, class Sm>
__device__ __forceinline__ void code_and_pack(Sm& sm, uint8_t* __restrict__ payload,
                                              float* __restrict__ scales, int64_t c, float* ef,
                                              int valid, uint32_t mkey, int p, int lane) {
    using F = FinishShape<Geo>;
    constexpr int kTopK = Geo::kTopK;
    constexpr int kB = Geo::kFieldBits;
    const int r = 32 * p + lane;
    const float x = sm.vals[r];
    const uint32_t pos = sm.fields[r];
    float s;
    if constexpr (kRule == kScaleMax) {
        s = __fdiv_rn(__uint_as_float(mkey), 1.5f);
    } else {
        float sum = fabsf(x);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
            sum = __fadd_rn(sum, __shfl_down_sync(0xffffffffu, sum, o));
        if constexpr (F::kPackWarps > 1) {
            if (lane == 0) sm.psum[p] = sum;
            named_sync(kBarPack, 32 * F::kPackWarps);
            float t[F::kPackWarps];
#pragma unroll
            for (int q = 0; q < F::kPackWarps; ++q) t[q] = sm.psum[q];
#pragma unroll
            for (int wdt = 1; wdt < F::kPackWarps; wdt <<= 1)
#pragma unroll
                for (int q = 0; q + wdt < F::kPackWarps; q += 2 * wdt) t[q] = __fadd_rn(t[q], t[q + wdt]);
            sum = t[0];
        } else {
            sum = __shfl_sync(0xffffffffu, sum, 0);
        }
        s = __fdiv_rn(sum, static_cast<float>(kTopK));
    }
    const uint32_t code = quant_code(x, s);
    if (static_cast<int>(pos) < valid &&
        SPL_CHECK(valid <= SendShape<Geo>::kChunk, kSiteEfStore, pos))
        ef[pos] = __fsub_rn(x, level_value(code, s));
    const uint32_t field = code | (pos << 2);
    // word p b + k (k < b) holds bits [32 k, 32 k + 32) of this warp's 32 fields: field j at
    // bits [b j, b j + b); a word touches at most 4 fields of >= 13 bits
    const int k = lane < kB ? lane : kB - 1;
    const int j_first = (32 * k) / kB;
    const int j_last = (32 * k + 31) / kB;
    uint32_t word = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int j = j_first + q;
        const uint32_t f = __shfl_sync(0xffffffffu, field, j < 32 ? j : 31);
        if (j <= j_last) {
            const int off = kB * j - 32 * k;
            word |= off >= 0 ? (f << off) : (f >> (-off));
        }
    }
    uint32_t* rec = reinterpret_cast<uint32_t*>(payload + c * Geo::kRecordBytes);
    if (lane < kB && SPL_CHECK(kB * p + lane < Geo::kRecordWords, kSiteRecord, kB * p + lane))
        rec[kB * p + lane] = word;
    if (p == 0 && lane == 0) scales[c] = s;
}

template <class Geo, int kRule, bool kBf16, bool kEfHost>
__global__ void __launch_bounds__(SendShape<Geo>::kThreads, SendShape<Geo>::kMinBlocks)
k_ef_compress(const CompressTable tab, float beta, uint8_t* __restrict__ payload,
              float* __restrict__ scales, uint32_t* __restrict__ flags, int ctas, int per_cta) {
    using S = SendShape<Geo>;
    constexpr int kChunk = S::kChunk;
    constexpr int kTopK = S::kTopK;
    constexpr int kThreads = S::kThreads;
    constexpr int kWarps = S::kWarps;
    constexpr int kPer = S::kPer;
    constexpr int kVec = S::kVec;
    constexpr int kStride = S::kStride;
    constexpr int kBitmapWords = S::kBitmapWords;
    constexpr int kWpl = S::kWordsPerLane;
    using F = FinishShape<Geo>;
    constexpr int kGatherFirst = kWarps - F::kGatherWarps;   // first warp of the gather group
    constexpr int kPackFirst = kWarps - F::kPackWarps;       // first warp of the packing group
    // Two ways to finish a chunk once its positions are chosen:
    //   - kFast (the usual one): every thread stores its accumulated values unchanged; in the
    //     next iteration the gather group turns the chunk's bitmap into positions by rank and
    //     reads their values back (still in L2) beside warp 0's bin search, and the packing
    //     group codes them, writes their residuals over them and packs the record beside warp
    //     0's boundary-bin ranking.  No owner step and no prefix barrier: four block barriers
    //     per chunk.
    //   - coding in place (the error buffer in host memory, where k scattered writes per
    //     chunk would cost the host link more than the owner step costs): warp 0 forms prefix
    //     counts of the bitmap, and the owners code their chosen values and form the residuals
    //     in registers before the one store; five barriers per chunk.
    constexpr bool kCodeInPlace = kEfHost;
    constexpr bool kFast = !kCodeInPlace;
    // the out-of-line select takes the keys through memory.  Handing it a copy made on that
    // path keeps the key registers from also being stored to the stack on every chunk (-4.5 %
    // at k = 64); with a host error buffer, where registers are scarcer, the copy makes the
    // compiler spill more in the loop instead, so there the keys are passed directly
    constexpr bool kCopyKeys = !kEfHost;
    using Sm = Smem<Geo, kRule, kFast>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t total = tab.chunk_begin[tab.num];
    const ChunkSpan span = cta_chunks(total, ctas, per_cta, blockIdx.x);
    if (span.first >= span.end) return;

    // thread 0 locates each chunk once, when it starts the chunk's copies, and leaves it in
    // shared memory for the CTA
    if constexpr (kFast) {   // the packing warp clears each bitmap after use; start clean
        for (int i = tid; i < 2 * kBitmapWords; i += kThreads)
            sm.sel_bm[i / kBitmapWords][i % kBitmapWords] = 0;
    }
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        sm.next_tensor = 0;
        const ChunkRef r0 = locate<kChunk, kBf16>(tab, span.first, sm.next_tensor);
        sm.next_delta = r0.delta;
        sm.next_ef = r0.ef;
        sm.next_valid = r0.valid;
        if (r0.full) prefetch<kChunk, kBf16, kEfHost>(sm, r0);
    }
    __syncthreads();

    uint32_t parity = 0;
    bool nonfinite = false;
    bool aborted = false;
    int pend_c = -1;         // the chunk whose record the last warp still has to pack
    float pend_s = 0.0f;     // coding in place: its scale
    uint32_t pend_mkey = 0;  // kFast: its largest key
    float* pend_ef = nullptr;   // its error buffer and extent
    int pend_valid = 0;

    // chunk indices stay below 2^31 (the host checks), so they are 32-bit here
    const int end32 = static_cast<int>(span.end);
    int it = 0;   // this CTA's iteration: kFast alternates the bitmaps by its parity
    for (int c = static_cast<int>(span.first); c < end32; c += ctas, ++it) {
        const int cur = kFast ? (it & 1) : 0;   // this chunk's bitmap: sm.sel_bm[cur]
        ChunkRef r;
        r.delta = sm.next_delta;
        r.ef = sm.next_ef;
        r.valid = sm.next_valid;
        r.full = r.valid == kChunk;

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
        if constexpr (kFast) {
            // the accumulated values go to the error buffer now, unchanged (the packing group
            // writes the chosen ones' residuals over them in the next iteration): from here on
            // only the keys stay in registers
            store_error_buffer<S, false>(r, a, tid);
        }

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
        // the stage has been read by every thread: start the next chunk's copies (and every
        // thread has read this chunk's location: replace it with the next one's)
        if (tid == 0 && c + ctas < end32) {
            const ChunkRef rn = locate<kChunk, kBf16>(tab, c + ctas, sm.next_tensor);
            sm.next_delta = rn.delta;
            sm.next_ef = rn.ef;
            sm.next_valid = rn.valid;
            if (rn.full) prefetch<kChunk, kBf16, kEfHost>(sm, rn);
        }
        if constexpr (!kFast) {
            // the previous chunk's owners have read the bitmaps (the barrier above follows
            // their step): clear them for this chunk's select, which first writes them two
            // barriers on
            if constexpr (2 * kBitmapWords == kThreads) {
                if (tid < kBitmapWords) sm.sel_bm[cur][tid] = 0;
                else sm.eq_bm[tid - kBitmapWords] = 0;
            } else {
                for (int i = tid; i < 2 * kBitmapWords; i += kThreads) {
                    if (i < kBitmapWords) sm.sel_bm[cur][i] = 0;
                    else sm.eq_bm[i - kBitmapWords] = 0;
                }
            }
            // the last warp packs the previous chunk's record: its fields are complete (the
            // barrier above follows that chunk's owner step) and are next written after this
            // chunk's select
            if (warp == kWarps - 1 && pend_c >= 0)
                pack_record<Geo>(sm, payload, scales, pend_c, pend_s, lane);
        }
        uint32_t mkey = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mkey = max(mkey, sm.warp_max[w]);

        // ---- select, fast path: 2048 bins of 1/128 octave over the 16 octaves below the
        //      largest key; the 64th key almost always falls inside, and its bin holds only a
        //      few keys, which warp 0 ranks directly.  Otherwise: the generic radix select.
        //      (A narrower first window does not pay: with ~10 % of the keys inside it, nearly
        //      every warp still has a lane that takes the in-window path.)
        // lo_key puts the largest key exactly in the top bin; a key below the window counts
        // in bin 0 (one unconditional atomic per key, no branch), so bin 0 is exact only when
        // nothing lies below the window (lo_key = 0), and a boundary bin of 0 otherwise
        // takes the generic select
        const bool windowed = mkey < kKeyInf;
        const uint32_t lo_key = mkey > kWindow ? mkey - kWindow : 0u;
        if (windowed) {
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const uint32_t bin = (max(key[i], lo_key) - lo_key) >> 16;
                if (SPL_CHECK(bin < 2048u, kSiteHist, bin)) atomicAdd(&sm.hist[bin], 1u);
            }
        }
        __syncthreads();
        if (windowed && warp == 0) {
            const bool found = top_digit(sm, kTopK, lane);
            if (lane == 0) sm.full_scan = found ? 0u : 1u;
        }
        if constexpr (kFast) {
            // beside warp 0's bin search: the gather group takes the previous chunk's chosen
            // positions from its bitmap (complete: a barrier follows that chunk's select),
            // clears that bitmap and starts reading the chosen values back; the warps between
            // clear the tie bitmap (warp 0 read it before the previous barrier) for this
            // chunk's marking, one barrier on
            if (warp >= kGatherFirst) {
                if (pend_c >= 0)   // the previous chunk's bitmap is the other one
                    gather_chosen<Geo>(sm, (it + 1) & 1, pend_ef, pend_valid, warp - kGatherFirst,
                                       lane);
            } else {
                for (int i = tid - 32; i >= 0 && i < kBitmapWords; i += 32 * (kGatherFirst - 1))
                    sm.eq_bm[i] = 0;
            }
        }
        __syncthreads();
        if (windowed && sm.full_scan != 0u) {   // uniform: every thread read the same flag
            if (tid == 0) SPL_COUNT(kDbgFullScan);
            find_digit<2048, S>(sm, sm.hist, kTopK, tid, lane, warp);
            __syncthreads();
        }
        if (tid == 0) SPL_COUNT(kDbgChunks);
        bool selected = false;
        if (windowed && sm.bcast[0] != kNotFound && (sm.bcast[0] != 0u || lo_key == 0u)) {
            const uint32_t need = kTopK - sm.bcast[1];
            const uint32_t dig = sm.bcast[0];
            const uint32_t in_bin = sm.bcast[2];
            if (in_bin == need || in_bin <= 64u) {
                const bool rank_bin = in_bin != need;
                if (tid == 0) SPL_COUNT(rank_bin ? (in_bin <= 32u ? kDbgRank32 : kDbgRank64) : kDbgWhole);
                // bin D as a key range [k_lo, k_hi): keys at or above k_hi are in, keys in the
                // range are in when the bin is taken whole, else they are the candidates
                const uint32_t k_lo = lo_key + (dig << 16);
                const uint32_t k_hi = k_lo + (1u << 16);
                const uint32_t k_in = rank_bin ? k_hi : k_lo;
                if constexpr (kFast) {
                    // branch-free marking: one predicated OR per vector of four (its positions
                    // share a bitmap word); a candidate's key offset is kept by position
                    if (rank_bin) {
#pragma unroll
                        for (int v = 0; v < kVec; ++v) {
                            const int j0 = v * kStride + 4 * tid;
                            uint32_t nib = 0, nib_cd = 0;
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint32_t kk = key[4 * v + u];
                                const uint32_t d = kk - k_lo;
                                const bool cd = d < (1u << 16);
                                nib |= (kk >= k_hi ? 1u : 0u) << u;
                                nib_cd |= (cd ? 1u : 0u) << u;
                                if (SPL_CHECK(j0 + u < kChunk, kSiteKeybuf, j0 + u))
                                    st_u16_if(&sm.keybuf[j0 + u], d, cd);
                            }
                            if (SPL_CHECK((j0 >> 5) < kBitmapWords, kSiteBitmap, j0)) {
                                red_or_nonzero(&sm.sel_bm[cur][j0 >> 5], nib << (j0 & 31));
                                red_or_nonzero(&sm.eq_bm[j0 >> 5], nib_cd << (j0 & 31));
                            }
                        }
                    } else {
#pragma unroll
                        for (int v = 0; v < kVec; ++v) {
                            const int j0 = v * kStride + 4 * tid;
                            uint32_t nib = 0;
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                nib |= (key[4 * v + u] >= k_lo ? 1u : 0u) << u;
                            if (SPL_CHECK((j0 >> 5) < kBitmapWords, kSiteBitmap, j0))
                                red_or_nonzero(&sm.sel_bm[cur][j0 >> 5], nib << (j0 & 31));
                        }
                    }
                    // the gather group's read-back copies have landed before the barrier
                    // after which the packing group reads them
                    if (warp >= kGatherFirst) asm volatile("cp.async.wait_all;" ::: "memory");
                } else {
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
                        if (nib != 0u && SPL_CHECK((j0 >> 5) < kBitmapWords, kSiteBitmap, j0))
                            atomicOr(&sm.sel_bm[cur][j0 >> 5], nib << (j0 & 31));
                    }
                }
                __syncthreads();
                if (rank_bin && warp == 0) {
                    if constexpr (kFast) {
                        // the candidates in ascending position order, from the tie bitmap
                        uint32_t w[kWpl];
                        uint32_t mine = 0;
#pragma unroll
                        for (int q = 0; q < kWpl; ++q) {
                            w[q] = sm.eq_bm[kWpl * lane + q];
                            mine += __popc(w[q]);
                        }
                        uint32_t incl = mine;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += y;
                        }
                        uint32_t slot = incl - mine;
#pragma unroll
                        for (int q = 0; q < kWpl; ++q) {
                            uint32_t bitsq = w[q];
                            while (bitsq != 0u) {
                                const int b = __ffs(bitsq) - 1;
                                bitsq &= bitsq - 1u;
                                const uint32_t pos = 32 * (kWpl * lane + q) + b;
                                if (SPL_CHECK(slot < 64u && pos < static_cast<uint32_t>(kChunk), kSiteCand, slot))
                                    sm.cand[slot] = make_uint2(k_lo + sm.keybuf[pos], pos);
                                ++slot;
                            }
                        }
                        __syncwarp();
                    }
                    // rank each candidate among the bin's keys (magnitude, then index)
                    if (in_bin <= 32u) {
                        const uint2 me = static_cast<uint32_t>(lane) < in_bin ? sm.cand[lane] : make_uint2(0u, 0u);
                        uint32_t rank = 0;
                        for (uint32_t o = 0; o < in_bin; ++o) {
                            const uint32_t ok = __shfl_sync(0xffffffffu, me.x, o);
                            const uint32_t oj = __shfl_sync(0xffffffffu, me.y, o);
                            rank += (ok > me.x || (ok == me.x && oj < me.y)) ? 1u : 0u;
                        }
                        if (static_cast<uint32_t>(lane) < in_bin && rank < need &&
                            SPL_CHECK((me.y >> 5) < kBitmapWords, kSiteBitmap, me.y))
                            atomicOr(&sm.sel_bm[cur][me.y >> 5], 1u << (me.y & 31));
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
                        if (r0 < need && SPL_CHECK((m0.y >> 5) < kBitmapWords, kSiteBitmap, m0.y))
                            atomicOr(&sm.sel_bm[cur][m0.y >> 5], 1u << (m0.y & 31));
                        if (static_cast<uint32_t>(lane) + 32u < in_bin && r1 < need &&
                            SPL_CHECK((m1.y >> 5) < kBitmapWords, kSiteBitmap, m1.y))
                            atomicOr(&sm.sel_bm[cur][m1.y >> 5], 1u << (m1.y & 31));
                    }
                    __syncwarp();
                }
                selected = true;
            }
        }
        if (!selected) {
            if (tid == 0) SPL_COUNT(kDbgGeneric);
            if (kFast && warp >= kGatherFirst) asm volatile("cp.async.wait_all;" ::: "memory");
            if constexpr (kCopyKeys) {
                uint32_t key_mem[kPer];
#pragma unroll
                for (int i = 0; i < kPer; ++i) key_mem[i] = key[i];
                generic_select<Geo>(sm, cur, key_mem, tid, lane, warp);
            } else {
                generic_select<Geo>(sm, cur, key, tid, lane, warp);
            }
        }
        // kFast: the packing group codes and packs the previous chunk's record while warp 0
        // ranks this chunk's boundary bin
        if constexpr (kFast) {
            if (warp >= kPackFirst && pend_c >= 0)
                code_and_pack<Geo, kRule>(sm, payload, scales, pend_c, pend_ef, pend_valid,
                                          pend_mkey, warp - kPackFirst, lane);
        }

        float s = 0.0f;   // coding in place: the max-abs scale
        if constexpr (!kFast) {
            // ---- warp 0: chosen positions before each bitmap word ------------------------
            if (warp == 0) {
                if constexpr (kWpl == 4) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(&sm.sel_bm[cur][4 * lane]);
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
                    uint32_t cnt[kWpl];
                    uint32_t mine = 0;
#pragma unroll
                    for (int q = 0; q < kWpl; ++q) {
                        cnt[q] = __popc(sm.sel_bm[cur][kWpl * lane + q]);
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

            // ---- owners: code each chosen value, form its residual in place, and write its
            //      field by rank ------------------------------------------------------------
            s = __fdiv_rn(__uint_as_float(mkey), 1.5f);
#pragma unroll
            for (int v = 0; v < kVec; ++v) {
                const int j0 = v * kStride + 4 * tid;
                const uint32_t word = sm.sel_bm[cur][j0 >> 5];
                const int sh = j0 & 31;
                if (((word >> sh) & 0xfu) == 0u) continue;
                const uint32_t base_rank = sm.pre[j0 >> 5];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if ((word >> (sh + u)) & 1u) {
                        const uint32_t rank = base_rank + __popc(word & ((1u << (sh + u)) - 1u));
                        const uint32_t code = quant_code(a[4 * v + u], s);
                        a[4 * v + u] = __fsub_rn(a[4 * v + u], level_value(code, s));
                        if (rank < kTopK)
                            sm.fields[rank] = static_cast<uint16_t>(code | (static_cast<uint32_t>(j0 + u) << 2));
                    }
                }
            }
        }
        // ---- coding in place: the error buffer, stored once, with the residuals ----------
        if constexpr (!kFast) store_error_buffer<S, kEfHost>(r, a, tid);

        // ---- the record is packed by the last warp in the next iteration ------------------
        pend_c = c;
        pend_s = s;
        pend_mkey = mkey;
        pend_ef = r.ef;
        pend_valid = r.valid;
    }
    __syncthreads();   // the last chunk's select (and error-buffer stores) are complete
    if constexpr (kFast) {
        if (pend_c >= 0) {   // uniform
            if (warp >= kGatherFirst) {
                gather_chosen<Geo>(sm, (it - 1) & 1, pend_ef, pend_valid, warp - kGatherFirst,
                                   lane);
                asm volatile("cp.async.wait_all;" ::: "memory");
            }
            __syncthreads();
            if (warp >= kPackFirst)
                code_and_pack<Geo, kRule>(sm, payload, scales, pend_c, pend_ef, pend_valid,
                                          pend_mkey, warp - kPackFirst, lane);
        }
    } else {
        if (warp == kWarps - 1 && pend_c >= 0)
            pack_record<Geo>(sm, payload, scales, pend_c, pend_s, lane);
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
    constexpr bool kFast = !kEfHost;
    const size_t smem = sizeof(Smem<Geo, kRule, kFast>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    constexpr int kThreads = SendShape<Geo>::kThreads;
    const int resident = persistent_grid(kern, kThreads, smem);
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    constexpr int kPerCta = kBf16 ? kSendChunksPerCtaBf16 : kSendChunksPerCta;
    const int grid = wave_grid(total, resident, kPerCta);
    k_ef_compress<Geo, kRule, kBf16, kEfHost><<<grid, kThreads, smem, stream>>>(
        tab, beta, payload, scales, flags, resident, kPerCta);
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
