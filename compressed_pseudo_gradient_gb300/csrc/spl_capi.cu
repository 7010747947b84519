// C ABI of the codec (declared in include/spl.h): argument checks on the host, then
// stream-ordered kernel launches.  Nothing here allocates device memory or synchronises.
#include <cmath>
#include <cstring>
#include <mutex>

#include "spl.h"
#include "spl_calib.h"
#include "spl_device.cuh"
#include "spl_kernels.h"
#if SPL_CHECKED
#include "spl_checked.h"
#endif

namespace {

thread_local int g_last_cuda_error = 0;

spl_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SPL_OK;
    g_last_cuda_error = static_cast<int>(e);
    return SPL_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Byte ranges [p, p + n) and [q, q + m) share a byte.
bool overlap(const void* p, size_t n, const void* q, size_t m) {
    if (p == nullptr || q == nullptr || n == 0 || m == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + m && b < a + n;
}

constexpr size_t kMaxChunks = 0x7fffffff;   // chunk indices stay below 2^31

// CUDA memory type of a pointer (cudaMemoryTypeDevice, cudaMemoryTypeHost for pinned host
// memory, ...), or -1 when the runtime cannot tell (the error is cleared).
int memory_type(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return static_cast<int>(at.type);
}

}  // namespace

namespace spl {

// Resident CTAs of a kernel on the current device (SMs x blocks per SM).  The device's SM
// count is read once per device; the occupancy query is a host-side computation.
int persistent_grid(const void* kernel, int threads, size_t dyn_smem) {
    static std::mutex mu;
    static int sm_count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    int sms;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (sm_count[dev] == 0 &&
            cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess)
            return -1;
        sms = sm_count[dev];
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem) !=
        cudaSuccess)
        return -1;
    return sms * (per_sm > 0 ? per_sm : 1);
}

}  // namespace spl

extern "C" {

size_t spl_num_chunks(size_t n) { return n / SPL_CHUNK + (n % SPL_CHUNK != 0); }

const char* spl_status_string(int status) {
    switch (status) {
        case SPL_OK: return "ok";
        case SPL_ERR_INVALID_ARG: return "invalid argument";
        case SPL_ERR_ALIGNMENT: return "misaligned pointer";
        case SPL_ERR_CUDA: return "CUDA error";
        case SPL_ERR_NONFINITE: return "non-finite accumulated value";
        case SPL_ERR_BAD_PAYLOAD: return "rejected record";
        case SPL_ERR_TIMEOUT: return "kernel stopped on a bounded wait";
        default: return "unknown status";
    }
}

spl_status spl_flags_status(uint32_t flags) {
    if (flags & (SPL_FLAG_TIMEOUT | SPL_FLAG_COPY_PENDING)) return SPL_ERR_TIMEOUT;
    if (flags & SPL_FLAG_BAD_RECORD) return SPL_ERR_BAD_PAYLOAD;
    if (flags & SPL_FLAG_NONFINITE) return SPL_ERR_NONFINITE;
    return SPL_OK;
}

int spl_last_cuda_error(void) { return g_last_cuda_error; }

// The codec a call names (NULL: the default one).  Returns false for a codec the library has
// no kernels for.
static bool resolve_codec(const spl_codec* c, spl::Codec* out) {
    if (c == nullptr) {
        *out = spl::Codec{SPL_CHUNK, SPL_TOPK, SPL_SCALE_MAX_ABS};
        return true;
    }
    if (c->chunk > 65536u || c->topk > 65536u || c->scale_rule > 1u) return false;
    *out = spl::Codec{static_cast<int>(c->chunk), static_cast<int>(c->topk),
                      static_cast<int>(c->scale_rule)};
    return spl::codec_record_bytes(*out) != 0;
}

static size_t chunks_of(size_t n, size_t L) { return n / L + (n % L != 0); }

static spl_status check_tensor(const void* delta, spl_dtype dt, const float* ef, size_t n,
                               size_t L) {
    if (n == 0) return SPL_OK;
    if (delta == nullptr || ef == nullptr) return SPL_ERR_INVALID_ARG;
    if (dt != SPL_F32 && dt != SPL_BF16) return SPL_ERR_INVALID_ARG;
    if (chunks_of(n, L) > kMaxChunks) return SPL_ERR_INVALID_ARG;
    if (!aligned(delta, 16) || !aligned(ef, 16)) return SPL_ERR_ALIGNMENT;
    const size_t esz = dt == SPL_F32 ? 4 : 2;
    if (overlap(delta, n * esz, ef, n * 4)) return SPL_ERR_INVALID_ARG;
    return SPL_OK;
}

static spl_status check_outputs(const spl_tensor* t, int num, spl_dtype dt, const uint8_t* payload,
                                const float* scales, const uint32_t* flags, size_t C, size_t rb) {
    if (C == 0) return SPL_OK;
    if (payload == nullptr || scales == nullptr) return SPL_ERR_INVALID_ARG;
    if (!aligned(payload, 16) || !aligned(scales, 4) || !aligned(flags, 4))
        return SPL_ERR_ALIGNMENT;
    const size_t esz = dt == SPL_F32 ? 4 : 2;
    if (overlap(payload, C * rb, scales, C * 4) || overlap(flags, 4, payload, C * rb) ||
        overlap(flags, 4, scales, C * 4))
        return SPL_ERR_INVALID_ARG;
    for (int i = 0; i < num; ++i) {
        const size_t n = t[i].n;
        if (overlap(payload, C * rb, t[i].delta, n * esz) ||
            overlap(payload, C * rb, t[i].ef, n * 4) ||
            overlap(scales, C * 4, t[i].delta, n * esz) || overlap(scales, C * 4, t[i].ef, n * 4) ||
            overlap(flags, 4, t[i].ef, n * 4) || overlap(flags, 4, t[i].delta, n * esz))
            return SPL_ERR_INVALID_ARG;
        for (int k = 0; k < i; ++k)
            if (overlap(t[k].ef, t[k].n * 4, t[i].ef, n * 4) ||
                overlap(t[k].ef, t[k].n * 4, t[i].delta, n * esz) ||
                overlap(t[i].ef, n * 4, t[k].delta, t[k].n * esz))
                return SPL_ERR_INVALID_ARG;
    }
    return SPL_OK;
}

static spl_status compress_impl(const spl::Codec& cd, const spl_tensor* tensors, int num_tensors,
                                spl_dtype delta_dtype, float beta, uint8_t* payload, float* scales,
                                uint32_t* d_flags, spl_stream_t stream) {
    if (tensors == nullptr || num_tensors < 1) return SPL_ERR_INVALID_ARG;
    if (delta_dtype != SPL_F32 && delta_dtype != SPL_BF16) return SPL_ERR_INVALID_ARG;
    if (!std::isfinite(beta)) return SPL_ERR_INVALID_ARG;
    const size_t L = static_cast<size_t>(cd.chunk);
    const size_t rb = static_cast<size_t>(spl::codec_record_bytes(cd));
    size_t C = 0;
    for (int i = 0; i < num_tensors; ++i) {
        const spl_status st =
            check_tensor(tensors[i].delta, delta_dtype, tensors[i].ef, tensors[i].n, L);
        if (st != SPL_OK) return st;
        C += chunks_of(tensors[i].n, L);
        if (C > kMaxChunks) return SPL_ERR_INVALID_ARG;
    }
    const spl_status st =
        check_outputs(tensors, num_tensors, delta_dtype, payload, scales, d_flags, C, rb);
    if (st != SPL_OK) return st;
    if (C == 0) return SPL_OK;
    // delta (and a device-resident error buffer) arrive by bulk copies (TMA) into shared
    // memory: device memory; an error buffer may instead be pinned host memory, then read and
    // written with plain accesses (one kind for the whole table)
    int ef_kind = -2;
    for (int i = 0; i < num_tensors; ++i) {
        if (tensors[i].n == 0) continue;
        if (memory_type(tensors[i].delta) != cudaMemoryTypeDevice) return SPL_ERR_INVALID_ARG;
        const int k = memory_type(tensors[i].ef);
        if (k != cudaMemoryTypeDevice && k != cudaMemoryTypeHost) return SPL_ERR_INVALID_ARG;
        if (ef_kind != -2 && k != ef_kind) return SPL_ERR_INVALID_ARG;
        ef_kind = k;
    }
    const bool ef_host = ef_kind == cudaMemoryTypeHost;
    if (ef_host && !spl::is_default_codec(cd)) return SPL_ERR_INVALID_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    size_t chunk0 = 0;
    for (int first = 0; first < num_tensors; first += spl::kMaxTensorsPerLaunch) {
        spl::CompressTable tab;
        std::memset(&tab, 0, sizeof tab);
        const int count = num_tensors - first < spl::kMaxTensorsPerLaunch
                              ? num_tensors - first : spl::kMaxTensorsPerLaunch;
        int64_t chunks = 0;
        for (int i = 0; i < count; ++i) {
            tab.delta[i] = tensors[first + i].delta;
            tab.ef[i] = tensors[first + i].ef;
            tab.n[i] = static_cast<int64_t>(tensors[first + i].n);
            tab.chunk_begin[i] = chunks;
            chunks += static_cast<int64_t>(chunks_of(tensors[first + i].n, L));
        }
        tab.chunk_begin[count] = chunks;
        tab.num = count;
        const spl_status ls = cuda_status(spl::launch_ef_compress(
            tab, cd, delta_dtype == SPL_BF16, ef_host, beta, payload + chunk0 * rb,
            scales + chunk0, d_flags, s));
        if (ls != SPL_OK) return ls;
        chunk0 += static_cast<size_t>(chunks);
    }
    return SPL_OK;
}

spl_status spl_ef_compress_multi(const spl_tensor* tensors, int num_tensors, spl_dtype delta_dtype,
                                 float beta, uint8_t* payload, float* scales, uint32_t* d_flags,
                                 spl_stream_t stream) {
    spl::Codec cd;
    resolve_codec(nullptr, &cd);
    return compress_impl(cd, tensors, num_tensors, delta_dtype, beta, payload, scales, d_flags,
                         stream);
}

spl_status spl_ef_compress_codec(const spl_codec* codec, const spl_tensor* tensors,
                                 int num_tensors, spl_dtype delta_dtype, float beta,
                                 uint8_t* payload, float* scales, uint32_t* d_flags,
                                 spl_stream_t stream) {
    spl::Codec cd;
    if (!resolve_codec(codec, &cd)) return SPL_ERR_INVALID_ARG;
    return compress_impl(cd, tensors, num_tensors, delta_dtype, beta, payload, scales, d_flags,
                         stream);
}

int64_t spl_codec_record_bytes(const spl_codec* codec) {
    spl::Codec cd;
    return resolve_codec(codec, &cd) ? spl::codec_record_bytes(cd) : -1;
}

size_t spl_codec_num_chunks(const spl_codec* codec, size_t n) {
    spl::Codec cd;
    return resolve_codec(codec, &cd) ? chunks_of(n, static_cast<size_t>(cd.chunk)) : 0;
}

spl_status spl_ef_compress(const void* delta, spl_dtype delta_dtype, float* ef, size_t n,
                           float beta, uint8_t* payload, float* scales, uint32_t* d_flags,
                           spl_stream_t stream) {
    const spl_tensor t = {delta, ef, n};
    if (n == 0) {
        if (delta_dtype != SPL_F32 && delta_dtype != SPL_BF16) return SPL_ERR_INVALID_ARG;
        return std::isfinite(beta) ? SPL_OK : SPL_ERR_INVALID_ARG;
    }
    return spl_ef_compress_multi(&t, 1, delta_dtype, beta, payload, scales, d_flags, stream);
}

static_assert(sizeof(spl_peer_stats) == sizeof(spl::PeerStats), "spl_peer_stats layout");

static spl_status decode_impl(const spl::Codec& cd, const uint8_t* const* payloads,
                              const float* const* scales, int P, size_t n, float* mean_out,
                              float* theta, float lr, bool validate, spl_peer_stats* d_stats,
                              uint32_t* d_flags, spl_stream_t stream) {
    if (P < 1 || P > SPL_MAX_PEERS) return SPL_ERR_INVALID_ARG;
    if (theta != nullptr && !std::isfinite(lr)) return SPL_ERR_INVALID_ARG;
    if (n == 0) return SPL_OK;
    if (payloads == nullptr || scales == nullptr || mean_out == nullptr) return SPL_ERR_INVALID_ARG;
    const size_t rb = static_cast<size_t>(spl::codec_record_bytes(cd));
    const size_t C = chunks_of(n, static_cast<size_t>(cd.chunk));
    if (C > kMaxChunks) return SPL_ERR_INVALID_ARG;
    if (!aligned(mean_out, 16) || !aligned(theta, 16) || !aligned(d_flags, 4))
        return SPL_ERR_ALIGNMENT;
    if (overlap(mean_out, n * 4, theta, n * 4)) return SPL_ERR_INVALID_ARG;
    if (overlap(d_flags, 4, mean_out, n * 4) || overlap(d_flags, 4, theta, n * 4))
        return SPL_ERR_INVALID_ARG;
    const size_t sb = static_cast<size_t>(P) * sizeof(spl_peer_stats);   // d_stats, if given
    spl::DecodeTable tab;
    std::memset(&tab, 0, sizeof tab);
    for (int p = 0; p < P; ++p) {
        if (payloads[p] == nullptr || scales[p] == nullptr) return SPL_ERR_INVALID_ARG;
        if (!aligned(payloads[p], 16) || !aligned(scales[p], 4)) return SPL_ERR_ALIGNMENT;
        if (overlap(payloads[p], C * rb, mean_out, n * 4) ||
            overlap(payloads[p], C * rb, theta, n * 4) ||
            overlap(scales[p], C * 4, mean_out, n * 4) || overlap(scales[p], C * 4, theta, n * 4) ||
            overlap(d_flags, 4, payloads[p], C * rb) || overlap(d_flags, 4, scales[p], C * 4) ||
            overlap(d_stats, sb, payloads[p], C * rb) || overlap(d_stats, sb, scales[p], C * 4))
            return SPL_ERR_INVALID_ARG;
        tab.payload[p] = payloads[p];
        tab.scale[p] = scales[p];
    }
    // theta arrives by bulk copies (TMA) into shared memory: device memory only (records and
    // scales are read with plain and 16-byte asynchronous loads, the outputs written with
    // plain stores; those take any memory the device can address)
    if (theta != nullptr && memory_type(theta) != cudaMemoryTypeDevice) return SPL_ERR_INVALID_ARG;
    return cuda_status(spl::launch_decode_aggregate(
        tab, cd, P, static_cast<int64_t>(n), mean_out, theta, lr, validate,
        reinterpret_cast<spl::PeerStats*>(d_stats), d_flags, reinterpret_cast<cudaStream_t>(stream)));
}

spl_status spl_decode_aggregate(const uint8_t* const* payloads, const float* const* scales, int P,
                                size_t n, float* mean_out, float* theta, float lr, int validate,
                                uint32_t* d_flags, spl_stream_t stream) {
    spl::Codec cd;
    resolve_codec(nullptr, &cd);
    return decode_impl(cd, payloads, scales, P, n, mean_out, theta, lr, validate != 0, nullptr,
                       d_flags, stream);
}

// Checks of a statistics array (P entries, 8-byte aligned, apart from the outputs).
static spl_status check_stats(const spl_peer_stats* d_stats, int P, size_t n,
                              const float* mean_out, const float* theta, const uint32_t* d_flags) {
    if (!aligned(d_stats, 8)) return SPL_ERR_ALIGNMENT;
    const size_t sb = static_cast<size_t>(P) * sizeof(spl_peer_stats);
    if (overlap(d_stats, sb, mean_out, n * 4) || overlap(d_stats, sb, theta, n * 4) ||
        overlap(d_stats, sb, d_flags, 4))
        return SPL_ERR_INVALID_ARG;
    return SPL_OK;
}

spl_status spl_decode_aggregate_codec(const spl_codec* codec, const uint8_t* const* payloads,
                                      const float* const* scales, int P, size_t n,
                                      float* mean_out, float* theta, float lr,
                                      spl_peer_stats* d_stats, uint32_t* d_flags,
                                      spl_stream_t stream) {
    spl::Codec cd;
    if (!resolve_codec(codec, &cd)) return SPL_ERR_INVALID_ARG;
    if (P < 1 || P > SPL_MAX_PEERS) return SPL_ERR_INVALID_ARG;
    if (d_stats != nullptr) {
        const spl_status st = check_stats(d_stats, P, n, mean_out, theta, d_flags);
        if (st != SPL_OK) return st;
    }
    return decode_impl(cd, payloads, scales, P, n, mean_out, theta, lr, true, d_stats, d_flags,
                       stream);
}

spl_status spl_decode_aggregate_stats(const uint8_t* const* payloads, const float* const* scales,
                                      int P, size_t n, float* mean_out, float* theta, float lr,
                                      spl_peer_stats* d_stats, uint32_t* d_flags,
                                      spl_stream_t stream) {
    if (P < 1 || P > SPL_MAX_PEERS || d_stats == nullptr) return SPL_ERR_INVALID_ARG;
    const spl_status st = check_stats(d_stats, P, n, mean_out, theta, d_flags);
    if (st != SPL_OK) return st;
    spl::Codec cd;
    resolve_codec(nullptr, &cd);
    return decode_impl(cd, payloads, scales, P, n, mean_out, theta, lr, true, d_stats, d_flags,
                       stream);
}

#if SPL_CHECKED
// Checked build: the debug arrays of every translation unit, merged (failed-check sites OR-ed,
// the first failure of the first unit that saw one, counts added).  Synchronises the device
// (symbol copies).
spl_status spl_debug_read(uint32_t* out, int reset) {
    if (out == nullptr) return SPL_ERR_INVALID_ARG;
    cudaError_t (*const readers[])(uint32_t*, bool) = {
        spl::debug_read_compress, spl::debug_read_compress_variants, spl::debug_read_decode,
        spl::debug_read_decode_variants, spl::debug_read_pack};
    for (int w = 0; w < spl::kDebugWords; ++w) out[w] = 0;
    for (auto rd : readers) {
        uint32_t d[spl::kDebugWords];
        const spl_status st = cuda_status(rd(d, reset != 0));
        if (st != SPL_OK) return st;
        out[spl::kDbgSites] |= d[spl::kDbgSites];
        if (out[spl::kDbgFirstSite] == 0 && d[spl::kDbgFirstSite] != 0) {
            out[spl::kDbgFirstSite] = d[spl::kDbgFirstSite];
            out[spl::kDbgFirstIndex] = d[spl::kDbgFirstIndex];
        }
        out[spl::kDbgFailures] += d[spl::kDbgFailures];
        for (int w = spl::kDbgChunks; w < spl::kDebugWords; ++w) out[w] += d[w];
    }
    return SPL_OK;
}
#endif

spl_status spl_pack(const uint16_t* idx, const uint8_t* codes, size_t num_chunks, uint8_t* payload,
                    spl_stream_t stream) {
    if (num_chunks == 0) return SPL_OK;
    if (idx == nullptr || codes == nullptr || payload == nullptr || num_chunks > kMaxChunks)
        return SPL_ERR_INVALID_ARG;
    if (!aligned(idx, 2) || !aligned(payload, 16)) return SPL_ERR_ALIGNMENT;
    if (overlap(payload, num_chunks * SPL_RECORD_BYTES, idx, num_chunks * SPL_TOPK * 2) ||
        overlap(payload, num_chunks * SPL_RECORD_BYTES, codes, num_chunks * SPL_TOPK))
        return SPL_ERR_INVALID_ARG;
    return cuda_status(spl::launch_pack(idx, codes, static_cast<int64_t>(num_chunks), payload,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

spl_status spl_unpack(const uint8_t* payload, size_t num_chunks, uint16_t* idx, uint8_t* codes,
                      spl_stream_t stream) {
    if (num_chunks == 0) return SPL_OK;
    if (idx == nullptr || codes == nullptr || payload == nullptr || num_chunks > kMaxChunks)
        return SPL_ERR_INVALID_ARG;
    if (!aligned(idx, 2) || !aligned(payload, 16)) return SPL_ERR_ALIGNMENT;
    if (overlap(payload, num_chunks * SPL_RECORD_BYTES, idx, num_chunks * SPL_TOPK * 2) ||
        overlap(payload, num_chunks * SPL_RECORD_BYTES, codes, num_chunks * SPL_TOPK) ||
        overlap(idx, num_chunks * SPL_TOPK * 2, codes, num_chunks * SPL_TOPK))
        return SPL_ERR_INVALID_ARG;
    return cuda_status(spl::launch_unpack(payload, static_cast<int64_t>(num_chunks), idx, codes,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

spl_status spl_calib_moves(spl_calib_pattern pattern, int persistent, const float* in0,
                           const float* in1, float* out0, float* out1, size_t n,
                           uint32_t* d_flags, spl_stream_t stream) {
    const bool sender = pattern == SPL_CALIB_SENDER_MOVES;
    if (!sender && pattern != SPL_CALIB_RECEIVER_MOVES) return SPL_ERR_INVALID_ARG;
    if (n % SPL_CHUNK != 0 || n / SPL_CHUNK > kMaxChunks) return SPL_ERR_INVALID_ARG;
    if (n == 0) return SPL_OK;
    const float* other = sender ? in1 : out1;   // the pattern's second array
    if (in0 == nullptr || out0 == nullptr || other == nullptr) return SPL_ERR_INVALID_ARG;
    if (!aligned(in0, 16) || !aligned(out0, 16) || !aligned(other, 16)) return SPL_ERR_ALIGNMENT;
    const size_t b = n * 4;
    if (overlap(out0, b, in0, b) || overlap(out0, b, other, b) ||
        (!sender && overlap(out1, b, in0, b)) || overlap(d_flags, 4, in0, b) ||
        overlap(d_flags, 4, out0, b) || overlap(d_flags, 4, other, b))
        return SPL_ERR_INVALID_ARG;
    if (memory_type(in0) != cudaMemoryTypeDevice || memory_type(out0) != cudaMemoryTypeDevice ||
        memory_type(other) != cudaMemoryTypeDevice)
        return SPL_ERR_INVALID_ARG;
    return cuda_status(spl::launch_calib_moves(sender, in0, sender ? in1 : nullptr, out0,
                                               sender ? nullptr : out1,
                                               static_cast<int64_t>(n / SPL_CHUNK),
                                               persistent != 0, d_flags,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
