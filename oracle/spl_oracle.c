/*
 * SparseLoCo pseudo-gradient codec: the CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  This file exists so that the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg can check the CUDA library against a plain, slow,
 * obviously correct restatement of the method.  The product path never links, loads or
 * calls it, and it shares no code, header, table or constant generator with the CUDA
 * library: every constant below is restated here from the pages.
 *
 * Sources (page title, then the section):
 *   [SF]  "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
 *         Pre-Training" (blokz.dev):
 *           - "SparseLoCo: Three Compression Levers in One Pass", items 1-3 and the
 *             per-chunk size equation (64 x (2 + 12) bits = 896 bits = 112 bytes);
 *           - "Why Extreme Sparsity Doesn't Break Convergence", paragraphs "Error feedback
 *             accumulation" and "Sparse aggregation can improve model quality";
 *           - "Why DiLoCo Alone Isn't Enough" (the pseudo-gradient is the difference of the
 *             pre- and post-inner-loop weights).
 *   [CV]  "Covenant-72B: Decentralized Training is No Longer Just a Dream" (wispaper.ai),
 *         "Methodology", item 1 (top-k sparsification + 2-bit quantisation, error feedback).
 *
 * Where the pages leave a step open, the oracle takes these readings (the CUDA library takes
 * the same ones, written independently):
 *   - error feedback: a = fmaf(beta, e, delta), one rounding; beta is a caller argument;
 *   - top-k order: |a| descending, then in-chunk index ascending; a NaN ranks above every
 *     number and all NaNs rank equal; the 64 chosen indices are stored ascending;
 *   - scale: s = m / 1.5f with m = max |a| over the chunk (= |a| of the first-ranked entry);
 *   - levels +-0.5s, +-1.5s; magnitude bit = (|v| > s), so a value exactly at s takes the
 *     smaller level; sign bit = (v < 0), so -0.0 codes as positive; code = sign<<1 | mag;
 *   - decoded value: mag ? 1.5f*s : 0.5f*s, negated when the sign bit is set (one rounding);
 *   - residual: e = a - q (one rounding) at the 64 chosen positions, e = a elsewhere;
 *   - record layout: entry r is the 14-bit field (code | idx << 2) at bits [14r, 14r + 14)
 *     of a 896-bit little-endian bit string, least significant bit first;
 *   - a tail chunk is padded with zeros to 4096 entries; the pads take part in the
 *     selection (they lose every tie to a real entry, having larger indices) but are never
 *     stored back and are dropped on decode;
 *   - aggregation: plain mean over the P peers, summed in fp32 in peer order starting from
 *     +0.0, then divided by P (one rounding); a malformed record (indices not strictly
 *     ascending, or a scale that is NaN, infinite or negative) contributes nothing and sets
 *     flag bit 1;
 *   - outer step: theta = fmaf(-lr, mean, theta).
 *
 * Plain single-threaded C11.  Build with -O2 -ffp-contract=off and no fast-math: every
 * floating-point operation is one IEEE binary32 operation rounded to nearest-even, the
 * precision in which the codec's scale, residual and mean are defined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_CHUNK 4096         /* [SF] item 1: non-overlapping chunks of 4,096 parameters */
#define ORC_TOPK 64            /* [SF] item 1: top-64 values by absolute magnitude */
#define ORC_INDEX_BITS 12      /* [SF] item 3: ceil(log2(4096)) = 12 */
#define ORC_VALUE_BITS 2       /* [SF] item 2: four levels, two bits */
#define ORC_FIELD_BITS (ORC_VALUE_BITS + ORC_INDEX_BITS)
#define ORC_RECORD_BYTES ((ORC_TOPK * ORC_FIELD_BITS) / 8) /* 896 bits = 112 bytes */

#define ORC_FLAG_NONFINITE 1u
#define ORC_FLAG_BAD_RECORD 2u

int orc_chunk(void) { return ORC_CHUNK; }
int orc_topk(void) { return ORC_TOPK; }
int orc_record_bytes(void) { return ORC_RECORD_BYTES; }

int64_t orc_num_chunks(int64_t n) { return (n + ORC_CHUNK - 1) / ORC_CHUNK; }

/* ------------------------------------------------------------------------------------------
 * Top-k selection ([SF] item 1), written for any chunk length L and any k <= L so that tiny
 * cases can be checked against exhaustive enumeration.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    float mag;
    int is_nan;
    int idx;
} orc_item;

/* Total order: NaN first, then larger |a| first, then smaller index first. */
static int orc_cmp_rank(const void* pa, const void* pb) {
    const orc_item* a = (const orc_item*)pa;
    const orc_item* b = (const orc_item*)pb;
    if (a->is_nan != b->is_nan) return a->is_nan ? -1 : 1;
    if (!a->is_nan && a->mag != b->mag) return a->mag > b->mag ? -1 : 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

static int orc_cmp_int(const void* pa, const void* pb) {
    int a = *(const int*)pa, b = *(const int*)pb;
    return (a > b) - (a < b);
}

/* Writes the k chosen in-chunk indices of a[0..L) to out_idx in ascending order.
 * Returns the index of the first-ranked entry (the one whose magnitude is the chunk max). */
int orc_topk_select(const float* a, int L, int k, int* out_idx) {
    orc_item* items = (orc_item*)malloc(sizeof(orc_item) * (size_t)L);
    int top;
    int i;
    for (i = 0; i < L; ++i) {
        items[i].mag = fabsf(a[i]);
        items[i].is_nan = isnan(a[i]) ? 1 : 0;
        items[i].idx = i;
    }
    qsort(items, (size_t)L, sizeof(orc_item), orc_cmp_rank);
    top = items[0].idx;
    for (i = 0; i < k; ++i) out_idx[i] = items[i].idx;
    qsort(out_idx, (size_t)k, sizeof(int), orc_cmp_int);
    free(items);
    return top;
}

/* ------------------------------------------------------------------------------------------
 * 2-bit quantiser with a per-chunk scale ([SF] item 2).
 * ---------------------------------------------------------------------------------------- */
float orc_scale(float m) { return m / 1.5f; }

int orc_code(float v, float s) {
    int sign = v < 0.0f;
    int mag = fabsf(v) > s;
    return (sign << 1) | mag;
}

float orc_level(int code, float s) {
    float q = (code & 1) ? 1.5f * s : 0.5f * s;
    return (code & 2) ? -q : q;
}

/* ------------------------------------------------------------------------------------------
 * Record packing ([SF] per-chunk equation): 64 fields of 14 bits, written one bit at a time.
 * ---------------------------------------------------------------------------------------- */
void orc_pack_record(const uint16_t* idx, const uint8_t* code, uint8_t* out) {
    int r, b;
    memset(out, 0, ORC_RECORD_BYTES);
    for (r = 0; r < ORC_TOPK; ++r) {
        uint32_t field = (uint32_t)(code[r] & 3u) | ((uint32_t)(idx[r] & 0xFFFu) << ORC_VALUE_BITS);
        for (b = 0; b < ORC_FIELD_BITS; ++b) {
            int bit = r * ORC_FIELD_BITS + b;
            if ((field >> b) & 1u) out[bit >> 3] |= (uint8_t)(1u << (bit & 7));
        }
    }
}

void orc_unpack_record(const uint8_t* rec, uint16_t* idx, uint8_t* code) {
    int r, b;
    for (r = 0; r < ORC_TOPK; ++r) {
        uint32_t field = 0;
        for (b = 0; b < ORC_FIELD_BITS; ++b) {
            int bit = r * ORC_FIELD_BITS + b;
            if ((rec[bit >> 3] >> (bit & 7)) & 1u) field |= 1u << b;
        }
        code[r] = (uint8_t)(field & 3u);
        idx[r] = (uint16_t)(field >> ORC_VALUE_BITS);
    }
}

void orc_pack(const uint16_t* idx, const uint8_t* code, int64_t C, uint8_t* payload) {
    int64_t c;
    for (c = 0; c < C; ++c)
        orc_pack_record(idx + c * ORC_TOPK, code + c * ORC_TOPK, payload + c * ORC_RECORD_BYTES);
}

void orc_unpack(const uint8_t* payload, int64_t C, uint16_t* idx, uint8_t* code) {
    int64_t c;
    for (c = 0; c < C; ++c)
        orc_unpack_record(payload + c * ORC_RECORD_BYTES, idx + c * ORC_TOPK, code + c * ORC_TOPK);
}

/* ------------------------------------------------------------------------------------------
 * Sender: error feedback + chunk top-64 + 2-bit quantise + pack + residual, one chunk at a
 * time ([SF] items 1-3; "Error feedback accumulation").
 *
 * delta: n values, fp32 (delta_is_bf16 = 0) or bf16 bit patterns (delta_is_bf16 = 1);
 * ef: n fp32 values, read and overwritten; payload: C * 112 bytes; scales: C floats.
 * Returns flag bit 0 when any accumulated value a is not finite.
 * ---------------------------------------------------------------------------------------- */
static float orc_bf16_to_float(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

uint32_t orc_ef_compress(const void* delta, int delta_is_bf16, float* ef, int64_t n, float beta,
                         uint8_t* payload, float* scales) {
    int64_t C = orc_num_chunks(n);
    int64_t c;
    uint32_t flags = 0;
    float a[ORC_CHUNK];
    int sel[ORC_TOPK];
    uint16_t idx[ORC_TOPK];
    uint8_t code[ORC_TOPK];

    for (c = 0; c < C; ++c) {
        int64_t base = c * ORC_CHUNK;
        int j, r, top;
        float m, s;

        /* e <- beta * e + delta, on the zero-padded chunk */
        for (j = 0; j < ORC_CHUNK; ++j) {
            int64_t i = base + j;
            if (i < n) {
                float d = delta_is_bf16 ? orc_bf16_to_float(((const uint16_t*)delta)[i])
                                        : ((const float*)delta)[i];
                a[j] = fmaf(beta, ef[i], d);
                if (!isfinite(a[j])) flags |= ORC_FLAG_NONFINITE;
            } else {
                a[j] = 0.0f;
            }
        }

        top = orc_topk_select(a, ORC_CHUNK, ORC_TOPK, sel);
        m = fabsf(a[top]);
        s = orc_scale(m);

        for (r = 0; r < ORC_TOPK; ++r) {
            float v = a[sel[r]];
            code[r] = (uint8_t)orc_code(v, s);
            idx[r] = (uint16_t)sel[r];
            a[sel[r]] = v - orc_level(code[r], s); /* residual at a transmitted position */
        }

        for (j = 0; j < ORC_CHUNK; ++j)
            if (base + j < n) ef[base + j] = a[j];

        orc_pack_record(idx, code, payload + c * ORC_RECORD_BYTES);
        scales[c] = s;
    }
    return flags;
}

/* ------------------------------------------------------------------------------------------
 * Receiver: decode P peers' records and take their mean, optionally followed by the outer
 * step theta <- theta - lr * mean ([SF] item 3, "Sparse aggregation can improve model
 * quality"; [SF] "Why DiLoCo Alone Isn't Enough" for the pseudo-gradient's sign).
 *
 * payloads[p]: C * 112 bytes; scales[p]: C floats; mean_out: n floats (overwritten);
 * theta: n floats or NULL.  Returns flag bit 1 when some record was rejected.
 * ---------------------------------------------------------------------------------------- */
static int orc_record_ok(const uint16_t* idx, float s) {
    int r;
    if (isnan(s) || isinf(s) || s < 0.0f) return 0;
    for (r = 1; r < ORC_TOPK; ++r)
        if (!(idx[r - 1] < idx[r])) return 0;
    return 1;
}

uint32_t orc_decode_aggregate(const uint8_t* const* payloads, const float* const* scales, int P,
                              int64_t n, float* mean_out, float* theta, float lr) {
    int64_t C = orc_num_chunks(n);
    int64_t c;
    uint32_t flags = 0;
    float acc[ORC_CHUNK];
    uint16_t idx[ORC_TOPK];
    uint8_t code[ORC_TOPK];

    for (c = 0; c < C; ++c) {
        int64_t base = c * ORC_CHUNK;
        int p, r, j;
        for (j = 0; j < ORC_CHUNK; ++j) acc[j] = 0.0f;
        for (p = 0; p < P; ++p) {
            float s = scales[p][c];
            orc_unpack_record(payloads[p] + c * ORC_RECORD_BYTES, idx, code);
            if (!orc_record_ok(idx, s)) {
                flags |= ORC_FLAG_BAD_RECORD;
                continue;
            }
            for (r = 0; r < ORC_TOPK; ++r)
                if (base + idx[r] < n) acc[idx[r]] += orc_level(code[r], s);
        }
        for (j = 0; j < ORC_CHUNK; ++j) {
            int64_t i = base + j;
            if (i >= n) break;
            mean_out[i] = acc[j] / (float)P;
            if (theta) theta[i] = fmaf(-lr, mean_out[i], theta[i]);
        }
    }
    return flags;
}

/* ------------------------------------------------------------------------------------------
 * Receiver statistics per peer, for screening updates that look unlike the rest ([SF] "What
 * the Blockchain Does (and Doesn't Do)": a crafted sparse update looks different from a
 * naturally concentrated one).  Over the 64 entries of every accepted record of peer p:
 *   big[p]       entries with the magnitude bit set (|q| = 1.5 s)
 *   negative[p]  entries with the sign bit set
 *   max_scale[p] the largest scale among accepted records (0 if none)
 *   sumsq[p]     the sum of q^2 (fp64; q^2 is exact in fp64), records in chunk order
 * and rejected[p], the number of rejected records.  Arrays of P, overwritten.
 * ---------------------------------------------------------------------------------------- */
void orc_peer_stats(const uint8_t* const* payloads, const float* const* scales, int P, int64_t n,
                    uint32_t* rejected, uint32_t* big, uint32_t* negative, float* max_scale,
                    double* sumsq) {
    int64_t C = orc_num_chunks(n);
    int p;
    uint16_t idx[ORC_TOPK];
    uint8_t code[ORC_TOPK];
    for (p = 0; p < P; ++p) {
        int64_t c;
        rejected[p] = big[p] = negative[p] = 0;
        max_scale[p] = 0.0f;
        sumsq[p] = 0.0;
        for (c = 0; c < C; ++c) {
            float s = scales[p][c];
            int r;
            orc_unpack_record(payloads[p] + c * ORC_RECORD_BYTES, idx, code);
            if (!orc_record_ok(idx, s)) {
                rejected[p] += 1;
                continue;
            }
            if (s > max_scale[p]) max_scale[p] = s;
            for (r = 0; r < ORC_TOPK; ++r) {
                double q = (double)orc_level(code[r], s);
                big[p] += code[r] & 1u;
                negative[p] += (code[r] >> 1) & 1u;
                sumsq[p] += q * q;
            }
        }
    }
}
