// Device-side constants and helpers shared by the codec's kernels (sm_103a).
//
// Format: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
// Pre-Training", section "SparseLoCo: Three Compression Levers in One Pass": chunks of 4096,
// top-64 by |value|, 2-bit values, 12-bit indices, 64 x 14 bits = 112 bytes per chunk.
// Codec variants keep the layout with another chunk length L or k: fields of
// 2 + log2(L) bits, k of them per record.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace spl {

constexpr int kChunk = 4096;
constexpr int kTopK = 64;
constexpr int kFieldBits = 14;
constexpr int kRecordBytes = 112;
constexpr int kRecordWords = kRecordBytes / 4;   // 28
constexpr int kRecordVec = kRecordBytes / 16;    // 7 x 16 bytes

// Scale rules: s = max |a| / 1.5 (the default), or the pairwise sum of the k chosen |a| in
// ascending index order divided by k (mean-abs, a variant).
constexpr int kScaleMax = 0;
constexpr int kScaleMeanAbs = 1;

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }

// A codec's record geometry: chunk length L (a power of two), k entries per record, each a
// field of 2 + log2(L) bits; the supported geometries fill whole 32-bit words.
template <int L, int K>
struct Geometry {
    static constexpr int kChunk = L;
    static constexpr int kTopK = K;
    static constexpr int kFieldBits = 2 + ilog2(L);
    static constexpr int kRecordWords = K * kFieldBits / 32;
    static constexpr int kRecordBytes = 4 * kRecordWords;
    static constexpr bool kVecRecords = kRecordBytes % 16 == 0;   // records stay 16-B aligned
    static_assert((L & (L - 1)) == 0 && L >= 2048 && L <= 8192, "chunk length");
    static_assert(K % 32 == 0 && K >= 32 && K <= 128, "entries per record");
    static_assert(K * kFieldBits % 32 == 0, "records fill whole words");
};
using DefaultGeometry = Geometry<kChunk, kTopK>;
static_assert(DefaultGeometry::kRecordBytes == kRecordBytes, "default record size");

constexpr uint32_t kFlagNonFinite = 1u;
constexpr uint32_t kFlagBadRecord = 2u;
constexpr uint32_t kFlagTimeout = 4u;
constexpr uint32_t kFlagCopyPending = 8u;   // after a timeout, the copy's own wait ran out too

// ---- checked build (compiled with -DSPL_CHECKED=1 into a library of its own) ---------------
// Every shared- and global-memory index of the kernels is tested before the access; an index
// out of range is recorded in a device debug array of this translation unit and the access is
// skipped (nothing traps).  The same array counts which select path each chunk took.  In the
// normal build SPL_CHECK is the constant true and SPL_COUNT nothing, so the code is unchanged.
constexpr int kDebugWords = 16;
enum DebugWord : int {
    kDbgSites = 0,        // OR of 1 << site over failed checks
    kDbgFirstSite = 1,    // site + 1 of the first failed check (0: none)
    kDbgFirstIndex = 2,   // its index (low 32 bits)
    kDbgFailures = 3,     // failed checks
    kDbgChunks = 8,       // sender chunks (fast-flow kernels)
    kDbgWhole = 9,        // ... whose boundary bin was taken whole
    kDbgRank32 = 10,      // ... whose boundary bin (<= 32 keys) was ranked
    kDbgRank64 = 11,      // ... whose boundary bin (33..64 keys) was ranked
    kDbgFullScan = 12,    // ... whose bin search went past the top 512 bins
    kDbgGeneric = 13      // ... that took the generic radix select
};
enum CheckSite : uint32_t {
    kSiteStage = 0, kSiteTail, kSiteHist, kSiteKeybuf, kSiteBitmap, kSiteCand, kSiteFields,
    kSiteEfStore, kSiteRecord, kSiteBulk, kSiteGenericHist, kSiteRecStage, kSiteAcc, kSiteEnt,
    kSiteMean, kSiteRecCopy, kSiteScale, kSiteStats, kSitePack
};

#if SPL_CHECKED
namespace {   // one array per translation unit
__device__ uint32_t g_debug[kDebugWords];
__device__ __noinline__ bool spl_check_failed(uint32_t site, uint64_t index) {
    atomicOr(&g_debug[kDbgSites], 1u << (site & 31u));
    atomicAdd(&g_debug[kDbgFailures], 1u);
    if (atomicCAS(&g_debug[kDbgFirstSite], 0u, site + 1u) == 0u)
        g_debug[kDbgFirstIndex] = static_cast<uint32_t>(index);
    return false;
}
}  // namespace
#define SPL_CHECK(cond, site, index) ((cond) ? true : ::spl::spl_check_failed((site), (index)))
#define SPL_COUNT(word) atomicAdd(&::spl::g_debug[(word)], 1u)
// Host side, one per translation unit: copy (and optionally clear) this unit's debug array.
#define SPL_DEBUG_READER(fn)                                                                  \
    cudaError_t fn(uint32_t* out, bool reset) {                                               \
        cudaError_t e = cudaMemcpyFromSymbol(out, g_debug, sizeof(uint32_t) * kDebugWords);  \
        if (e == cudaSuccess && reset) {                                                      \
            const uint32_t zero[kDebugWords] = {0};                                           \
            e = cudaMemcpyToSymbol(g_debug, zero, sizeof zero);                               \
        }                                                                                     \
        return e;                                                                             \
    }
#else
#define SPL_CHECK(cond, site, index) true
#define SPL_COUNT(word) ((void)0)
#endif

// Upper bound on any wait for an asynchronous copy: a healthy copy lands in microseconds.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// |a| as an ordered integer key: for non-NaN floats, unsigned order of (bits & 0x7fffffff)
// equals order of |a|.  Every NaN maps to one key just above +Inf, so NaNs rank first and
// tie among themselves (then the lower index wins, as for any tie).
constexpr uint32_t kKeyInf = 0x7f800000u;
constexpr uint32_t kKeyNaN = 0x7f800001u;

__device__ __forceinline__ uint32_t mag_key(float a) {
    return min(__float_as_uint(a) & 0x7fffffffu, kKeyNaN);
}

// 2-bit code and decoded value.  mag is set only strictly above s: a value exactly at the
// midpoint s of the two levels 0.5s and 1.5s takes the smaller one.
__device__ __forceinline__ uint32_t quant_code(float v, float s) {
    const uint32_t sign = v < 0.0f ? 1u : 0u;
    const uint32_t mag = fabsf(v) > s ? 1u : 0u;
    return (sign << 1) | mag;
}

__device__ __forceinline__ float level_value(uint32_t code, float s) {
    const float q = (code & 1u) ? __fmul_rn(1.5f, s) : __fmul_rn(0.5f, s);
    return (code & 2u) ? -q : q;
}

// x / d rounded to nearest, given rd = RN(1 / d): Markstein's correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): q0 = RN(x * rd), the remainder x - q0 * d is exact in one fma, and
// RN(q0 + rem * rd) is the correctly rounded quotient.  The tests compare it with the
// correctly rounded division for every divisor 1..256 over every significand, over every
// dividend below 2^-111 (quotients near and below the normal range), and on zeros,
// infinities and NaN.
// The correction is exact while q0 is zero or a normal number: a zero quotient is q0 itself
// (keeping its sign), and tiny nonzero quotients (and infinities or NaN, for which the
// remainder is NaN) take the correctly rounded division, on a branch that is rarely taken.
__device__ __forceinline__ float div_rn(float x, float d, float rd) {
    const float q0 = __fmul_rn(x, rd);
    const float rem = __fmaf_rn(-q0, d, x);
    const float q = __fmaf_rn(rem, rd, q0);
    const float aq = fabsf(q0);
    if ((aq < 2.3509887e-38f && aq != 0.0f) || !(aq <= 3.402823466e38f))  // 2^-125, FLT_MAX
        return __fdiv_rn(x, d);
    return aq == 0.0f ? q0 : q;
}

// 16-byte streaming accesses: the codec touches every dense byte exactly once.
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
    return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ void st_stream_f4(float* p, float4 v) {
    __stcs(reinterpret_cast<float4*>(p), v);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h16) {
    return __uint_as_float(h16 << 16);
}

// ---- which chunks a CTA works on ------------------------------------------------------------
// A launch is a sequence of waves of `ctas` CTAs (as many as are resident on the GPU at once);
// CTA b of wave w takes chunks w ctas K + b + j ctas for j = 0 .. K - 1 (K = per_cta), below
// `total`, in that order.  The CTAs on the GPU at any moment thus work on one compact range of
// chunks that advances through memory, and a CTA that runs ahead or behind can drift by at
// most K chunks.  (With one persistent wave, CTAs drift apart over hundreds of chunks, the
// addresses in flight spread over a wide range, and DRAM delivers less for the same bytes:
// spl_calib_moves measures both schedules.)
struct ChunkSpan {
    int64_t first;   // this CTA's first chunk (none if >= end)
    int64_t end;     // one past the last chunk of its wave; its chunks are first + j ctas < end
};

__host__ __device__ __forceinline__ ChunkSpan cta_chunks(int64_t total, int ctas, int per_cta,
                                                         int64_t block) {
    const int64_t w = block / ctas;
    const int64_t base = w * ctas * per_cta;
    const int64_t wave_end = base + static_cast<int64_t>(ctas) * per_cta;
    ChunkSpan s;
    s.first = base + block % ctas;
    s.end = wave_end < total ? wave_end : total;
    return s;
}

// ---- 1-D bulk copies (TMA, no multicast, no cluster launch) completed on an mbarrier ------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later bulk copies.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Global -> shared copy of `bytes` (a multiple of 16; both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 16-byte global -> shared copy (cp.async) whose completion is later reported to an mbarrier.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

// The same for 4 bytes (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

// One arrival on the mbarrier once all of this thread's earlier cp.async copies have landed
// (counted against the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0u;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase with the given parity to complete, for at most kWaitLimitNs.
// Returns false on timeout (the caller reports kFlagTimeout and stops).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// Builds record word w (0..27) of a chunk from the 64 fields held by one warp: lane l holds
// field l in f_lo and field l + 32 in f_hi.  Must be called by all 32 lanes; lanes >= 28
// return an unused value.  Field r sits at bits [14r, 14r + 14) of the 896-bit record.
__device__ __forceinline__ uint32_t record_word(uint32_t f_lo, uint32_t f_hi, int lane) {
    const int w = lane < kRecordWords ? lane : kRecordWords - 1;
    const int r_first = (32 * w) / kFieldBits;
    const int r_last = (32 * w + 31) / kFieldBits;
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {   // a 32-bit word touches at most 4 fields of 14 bits
        const int r = min(r_first + k, kTopK - 1);
        const uint32_t lo = __shfl_sync(0xffffffffu, f_lo, r & 31);
        const uint32_t hi = __shfl_sync(0xffffffffu, f_hi, r & 31);
        const uint32_t f = r < 32 ? lo : hi;
        if (r_first + k <= r_last) {
            const int off = kFieldBits * r - 32 * w;   // -12 .. 31
            word |= off >= 0 ? (f << off) : (f >> (-off));
        }
    }
    return word;
}

// Stores the 28 words held by lanes 0..27 as seven 16-byte vectors (record is 16-B aligned).
__device__ __forceinline__ void store_record(uint8_t* rec, uint32_t word, int lane) {
    const int b = 4 * (lane < kRecordVec ? lane : 0);
    uint4 v;
    v.x = __shfl_sync(0xffffffffu, word, b + 0);
    v.y = __shfl_sync(0xffffffffu, word, b + 1);
    v.z = __shfl_sync(0xffffffffu, word, b + 2);
    v.w = __shfl_sync(0xffffffffu, word, b + 3);
    if (lane < kRecordVec) reinterpret_cast<uint4*>(rec)[lane] = v;
}

// The same with one funnel shift, for fields of kBits bits.  Reads words[w + 1] even when
// the field ends inside words[w] (its bits are masked off), so the word after the record must
// be readable shared memory.
template <int kBits = kFieldBits>
__device__ __forceinline__ uint32_t record_field_fs(const uint32_t* words, int r) {
    const int bit = kBits * r;
    const int w = bit >> 5;
    return __funnelshift_r(words[w], words[w + 1], bit & 31) & ((1u << kBits) - 1u);
}

}  // namespace spl
