// Device-side constants and helpers shared by the codec's kernels (sm_103a).
//
// Format: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
// Pre-Training", section "SparseLoCo: Three Compression Levers in One Pass": chunks of 4096,
// top-64 by |value|, 2-bit values, 12-bit indices, 64 x 14 bits = 112 bytes per chunk.
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

constexpr uint32_t kFlagNonFinite = 1u;
constexpr uint32_t kFlagBadRecord = 2u;

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

// Field r (0..63) of a record held as 28 words in shared memory.
__device__ __forceinline__ uint32_t record_field(const uint32_t* words, int r) {
    const int bit = kFieldBits * r;
    const int w = bit >> 5;
    const int off = bit & 31;
    uint32_t v = words[w] >> off;
    if (off > 32 - kFieldBits) v |= words[w + 1] << (32 - off);
    return v & ((1u << kFieldBits) - 1u);
}

}  // namespace spl
