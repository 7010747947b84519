/*
 * spl.h: C ABI of the SparseLoCo pseudo-gradient codec on one GPU.
 *
 * The codec is defined in "The Sparse Frontier: SparseLoCo and the Compression Math Behind
 * Permissionless Pre-Training" (blokz.dev), section "SparseLoCo: Three Compression Levers in
 * One Pass" (items 1-3 and the per-chunk size equation) and section "Why Extreme Sparsity
 * Doesn't Break Convergence" (error feedback; aggregation of the peers' sparse updates).
 * The pages name no interface; these calls follow the steps the pages list.
 *
 * Fixed format (both sides of the wire):
 *   - a pseudo-gradient of n values is cut into C = ceil(n / 4096) chunks of 4096 values; a
 *     tail chunk is padded with zeros (the pads are never read from or written to memory);
 *   - per chunk, the 64 entries of largest |a| are kept (ties go to the lower in-chunk index;
 *     a NaN ranks above every number, and all NaNs rank equal);
 *   - scale s = m / 1.5f (fp32, round to nearest), m = max |a| over the chunk;
 *     2-bit code = (sign << 1) | mag with sign = (v < 0) and mag = (|v| > s); the decoded
 *     value is +-0.5f*s (mag 0) or +-1.5f*s (mag 1);
 *   - the record of a chunk is 112 bytes: entry r (r = 0..63, indices ascending) is the
 *     14-bit field (code | idx << 2) at bits [14r, 14r + 14) of a 896-bit little-endian bit
 *     string, least significant bit first (equivalently 28 little-endian uint32 words);
 *   - the scales are a separate array of C fp32 values, so every record is 16-byte aligned.
 *
 * Conventions for every call:
 *   - pointers named d_* or documented as "device" are device memory owned by the caller;
 *     the library allocates nothing and keeps no per-call state;
 *   - work is enqueued on `stream` (NULL = the legacy default stream) and never waited for:
 *     results are valid once the stream has reached the call;
 *   - argument errors are found on the host before anything is enqueued and returned
 *     synchronously; SPL_ERR_CUDA means a launch failed (spl_last_cuda_error() gives the
 *     cudaError_t value on the calling thread);
 *   - conditions found on the device are OR-ed into *d_flags (if d_flags is not NULL), which
 *     the caller reads after synchronising: SPL_FLAG_NONFINITE, SPL_FLAG_BAD_RECORD, and
 *     SPL_FLAG_TIMEOUT (an asynchronous copy into shared memory did not complete within one
 *     second; the kernel stopped early and its outputs are incomplete), with
 *     SPL_FLAG_COPY_PENDING as well when a further bounded wait for that copy also ran out (a
 *     block then exited with the copy possibly still in flight into its shared memory, so the
 *     device's state is suspect and the context should be discarded); spl_flags_status()
 *     turns a flags word read back into a status.  No call returns a device-detected
 *     condition itself: calls never wait for the device, so they cannot know it;
 *   - device pointers to fp32/bf16 dense arrays and to records must be 16-byte aligned;
 *     scales and flags 4-byte aligned; idx 2-byte aligned.
 */
#ifndef SPL_H_
#define SPL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* spl_stream_t; /* a cudaStream_t */

typedef enum {
    SPL_OK = 0,
    SPL_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, non-finite beta/lr, overlap, bad dtype */
    SPL_ERR_ALIGNMENT = 2,   /* a pointer breaks the alignment rule above */
    SPL_ERR_CUDA = 3,        /* a CUDA call failed; see spl_last_cuda_error() */
    /* the next three are only returned by spl_flags_status(), from a flags word read back */
    SPL_ERR_NONFINITE = 4,   /* some accumulated value a was NaN or infinite */
    SPL_ERR_BAD_PAYLOAD = 5, /* some record was rejected by the receiver's validation */
    SPL_ERR_TIMEOUT = 6      /* a kernel stopped early on a bounded wait: outputs incomplete */
} spl_status;

typedef enum { SPL_F32 = 0, SPL_BF16 = 1 } spl_dtype;

enum {
    SPL_CHUNK = 4096,        /* values per chunk (item 1) */
    SPL_TOPK = 64,           /* values kept per chunk, largest |a| first (item 1) */
    SPL_RECORD_BYTES = 112,  /* 64 fields of 14 bits (per-chunk equation) */
    SPL_PAYLOAD_BYTES = SPL_RECORD_BYTES,  /* the same, by the name of the payload */
    SPL_MAX_PEERS = 256,     /* largest P accepted by spl_decode_aggregate */
    SPL_P_MAX = SPL_MAX_PEERS,             /* the same */
    SPL_MAX_TENSORS_PER_LAUNCH = 64 /* spl_ef_compress_multi splits larger tables */
};

enum {
    SPL_FLAG_NONFINITE = 1u,   /* sender: some a = beta * e + delta was not finite */
    SPL_FLAG_BAD_RECORD = 2u,  /* receiver: some record was rejected */
    SPL_FLAG_TIMEOUT = 4u,     /* a bounded wait for an asynchronous copy ran out */
    SPL_FLAG_COPY_PENDING = 8u /* ... and so did the wait for that copy after stopping */
};

/*
 * The status a flags word stands for, most severe first: SPL_ERR_TIMEOUT (SPL_FLAG_TIMEOUT or
 * SPL_FLAG_COPY_PENDING), SPL_ERR_BAD_PAYLOAD (SPL_FLAG_BAD_RECORD), SPL_ERR_NONFINITE
 * (SPL_FLAG_NONFINITE), else SPL_OK.  A host-side helper: `flags` is the value read back.
 */
spl_status spl_flags_status(uint32_t flags);

/* Number of 4096-value chunks of an n-value tensor: ceil(n / 4096). */
size_t spl_num_chunks(size_t n);

/* Static English text for a status code (never NULL). */
const char* spl_status_string(int status);

/* cudaError_t value of the last SPL_ERR_CUDA returned on the calling thread (0 if none). */
int spl_last_cuda_error(void);

/*
 * Sender, one round: error feedback, chunk top-64, 2-bit quantisation, packing and the
 * residual, fused in one pass over the tensor (items 1-3; "Error feedback accumulation").
 *
 *   a      = fmaf(beta, ef[i], delta[i])          (bf16 delta is widened exactly first)
 *   record = the 64 entries of largest |a| per chunk, as above
 *   ef[i]  = a - q[i] at the 64 kept positions (q = decoded value), a elsewhere
 *
 * delta:   device, n values of type delta_dtype (SPL_F32 or SPL_BF16), read only
 * ef:      n fp32 values, read and overwritten (the error-feedback buffer): device memory, or
 *          pinned host memory (cudaHostAlloc / cudaHostRegister) so that a buffer too large
 *          for HBM can stay in host memory; the kernel then reads and writes it over the
 *          host link with plain accesses, which bounds the call's throughput.  Pageable or
 *          managed memory is rejected (SPL_ERR_INVALID_ARG).
 * n:       number of values; n = 0 does nothing and accepts NULL pointers
 * beta:    error-feedback decay, finite
 * payload: device, spl_num_chunks(n) * 112 bytes, written
 * scales:  device, spl_num_chunks(n) fp32, written
 * d_flags: device uint32 or NULL; SPL_FLAG_NONFINITE is OR-ed in when some a is not finite
 *          (the records are still written, deterministically)
 * Outputs must not overlap the inputs or each other.  delta must be device memory
 * (SPL_ERR_INVALID_ARG otherwise); payload, scales and d_flags any memory the device can write.
 */
spl_status spl_ef_compress(const void* delta, spl_dtype delta_dtype, float* ef, size_t n,
                           float beta, uint8_t* payload, float* scales, uint32_t* d_flags,
                           spl_stream_t stream);

/* One tensor of a multi-tensor round: chunks never span two tensors. */
typedef struct {
    const void* delta; /* device, n values of the call's delta_dtype */
    float* ef;         /* device, n fp32 */
    size_t n;
} spl_tensor;

/*
 * spl_ef_compress over a table of tensors, each chunked on its own (its last chunk padded),
 * in one pass.  The records and scales of tensor i start at chunk sum_{j<i} ceil(n_j / 4096)
 * of payload / scales.  `tensors` is a HOST array of num_tensors entries (num_tensors >= 1);
 * entries with n = 0 are allowed.  Tables longer than SPL_MAX_TENSORS_PER_LAUNCH are
 * enqueued as several launches on the same stream.  The error buffers of one table are all
 * device memory or all pinned host memory.
 */
spl_status spl_ef_compress_multi(const spl_tensor* tensors, int num_tensors,
                                 spl_dtype delta_dtype, float beta, uint8_t* payload,
                                 float* scales, uint32_t* d_flags, spl_stream_t stream);

/*
 * Receiver: decode P peers' records of one n-value tensor and write their mean; optionally
 * apply the outer step theta <- theta - lr * mean in the same pass ("Sparse aggregation can
 * improve model quality"; the pseudo-gradient is pre- minus post-inner-loop weights, "Why
 * DiLoCo Alone Isn't Enough").
 *
 *   mean[i]  = (sum over peers p, in order p = 0..P-1, of q_p[i], fp32 from +0.0) / P
 *   theta[i] = fmaf(-lr, mean[i], theta[i])
 *
 * payloads: HOST array of P device pointers, each spl_num_chunks(n) * 112 bytes
 * scales:   HOST array of P device pointers, each spl_num_chunks(n) fp32
 * P:        1 .. SPL_MAX_PEERS
 * mean_out: device, n fp32, overwritten (not accumulated)
 * theta:    device, n fp32, updated in place, or NULL (then lr is ignored)
 * lr:       outer learning rate, finite when theta is given
 * validate: nonzero: every record is checked first, and one whose indices are not strictly
 *           ascending, or whose scale is NaN, infinite or negative, contributes nothing (the
 *           mean still divides by P) and sets SPL_FLAG_BAD_RECORD in *d_flags;
 *           0: the checks are skipped (for records the caller made or has already checked);
 *           a malformed record then gives an unspecified mean and theta, and still reads and
 *           writes nothing outside the arrays above (indices are 12 bits wide by construction)
 * d_flags:  device uint32 or NULL
 * Entries that decode past n (the pads of a tail chunk) are dropped.  mean_out and theta must
 * not overlap each other or any record or scale array, nor d_flags any array.  theta must be
 * device memory (SPL_ERR_INVALID_ARG otherwise); the other arrays any memory the device can
 * address.
 */
spl_status spl_decode_aggregate(const uint8_t* const* payloads, const float* const* scales,
                                int P, size_t n, float* mean_out, float* theta, float lr,
                                int validate, uint32_t* d_flags, spl_stream_t stream);

/*
 * Per-peer statistics of the records a receiver accepted, for screening updates that look
 * unlike the rest (The Sparse Frontier, "What the Blockchain Does (and Doesn't Do)": an
 * update built to game the screening is distributed differently from an honest one).
 * Counted over the 64 entries of every accepted record (a tail chunk's pads included).
 */
typedef struct {
    uint32_t rejected;  /* records rejected (indices not strictly ascending, or a bad scale) */
    uint32_t big;       /* entries with the magnitude bit set (|q| = 1.5 s) */
    uint32_t negative;  /* entries with the sign bit set */
    float max_scale;    /* largest scale among accepted records (0 if none) */
    double sumsq;       /* sum of q^2 over the entries (relative error ~1e-7: fp32 per record,
                           compensated sums; records summed in no fixed order) */
} spl_peer_stats;       /* 24 bytes */

/*
 * spl_decode_aggregate with validation on, and in the same pass the statistics above for each
 * peer (counting rejected records needs the checks, so this call always makes them).
 * d_stats: device array of P entries (8-byte aligned), ACCUMULATED into: zero it before the
 * first call (counts add up, max_scale takes the maximum, sumsq adds up across calls); it must
 * not overlap any other array of the call.
 */
spl_status spl_decode_aggregate_stats(const uint8_t* const* payloads, const float* const* scales,
                                      int P, size_t n, float* mean_out, float* theta, float lr,
                                      spl_peer_stats* d_stats, uint32_t* d_flags,
                                      spl_stream_t stream);

/*
 * Codec variants, for ablation.  The pages fix L = 4096 and k = 64 ("SparseLoCo: Three
 * Compression Levers in One Pass", item 1), give the index width as ceil(log2 L) (item 3) and
 * leave the scale rule open (item 2 names one scale per chunk, no formula).  A variant keeps the
 * record layout with fields of 2 + log2 L bits, k per record, in k x (2 + log2 L) / 8 bytes;
 * records follow one another with no padding (payload base 16-byte aligned; records of 52
 * or 56 bytes are then 4-byte aligned).  Scale rules:
 *   SPL_SCALE_MAX_ABS   s = max |a| / 1.5f (the default, above);
 *   SPL_SCALE_MEAN_ABS  s = (pairwise sum of the k chosen |a| in ascending index order) / k,
 *                       where the pairwise sum of x[0..m) is x[0] for m = 1 and otherwise the
 *                       sum of its first floor(m/2) entries plus the sum of the rest, each
 *                       summed the same way, in fp32 (round to nearest); codes, levels, the
 *                       residual and the decoder are those of the default rule.
 * Supported (L, k): (4096, 64) (the default), (4096, 32), (4096, 128), (2048, 32),
 * (8192, 128), each with either rule.  A NULL codec pointer means the default codec.
 */
typedef enum { SPL_SCALE_MAX_ABS = 0, SPL_SCALE_MEAN_ABS = 1 } spl_scale_rule;

typedef struct {
    uint32_t chunk;      /* L: values per chunk */
    uint32_t topk;       /* k: entries per record */
    uint32_t scale_rule; /* an spl_scale_rule */
} spl_codec;

/* Bytes of one record of the codec, or -1 when the library does not implement it. */
int64_t spl_codec_record_bytes(const spl_codec* codec);

/* ceil(n / L) for the codec's chunk length L (0 for a codec the library does not implement). */
size_t spl_codec_num_chunks(const spl_codec* codec, size_t n);

/*
 * spl_ef_compress_multi with the given codec: payload holds spl_codec_num_chunks(n_i) records
 * of spl_codec_record_bytes bytes per tensor, in table order.  Error buffers must be device
 * memory unless the codec is the default one.  SPL_ERR_INVALID_ARG for a codec the library
 * does not implement.
 */
spl_status spl_ef_compress_codec(const spl_codec* codec, const spl_tensor* tensors,
                                 int num_tensors, spl_dtype delta_dtype, float beta,
                                 uint8_t* payload, float* scales, uint32_t* d_flags,
                                 spl_stream_t stream);

/*
 * spl_decode_aggregate with validation on (d_stats NULL) or spl_decode_aggregate_stats
 * (d_stats given) for records of the given codec (only its L and k matter to the receiver): each payloads[p] holds
 * spl_codec_num_chunks(n) records of spl_codec_record_bytes bytes, 16-byte aligned at its
 * start; the statistics count over the k entries of each accepted record.
 */
spl_status spl_decode_aggregate_codec(const spl_codec* codec, const uint8_t* const* payloads,
                                      const float* const* scales, int P, size_t n,
                                      float* mean_out, float* theta, float lr,
                                      spl_peer_stats* d_stats, uint32_t* d_flags,
                                      spl_stream_t stream);

/*
 * Record layout helpers (per-chunk size equation): idx[C][64] and codes[C][64] to and from
 * payload[C][112].  Only the low 12 bits of an index and the low 2 bits of a code are used;
 * pack does not check ordering.  All pointers are device memory.
 */
spl_status spl_pack(const uint16_t* idx, const uint8_t* codes, size_t num_chunks,
                    uint8_t* payload, spl_stream_t stream);
spl_status spl_unpack(const uint8_t* payload, size_t num_chunks, uint16_t* idx,
                      uint8_t* codes, spl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPL_H_ */
