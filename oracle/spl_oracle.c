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
 *           - "Why DiLoCo Alone Isn't Enough" (the pseudo-gradient is how far the inner
 *             optimisation moved the weights).
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
 * Codec variants, for ablation (the pages fix L = 4096 and k = 64 and give the index width as
 * ceil(log2 L); they leave the scale rule open):
 *   - chunk length L (a power of two) and k <= L: every field is 2 + ceil(log2 L) bits, a record
 *     is k such fields, packed as above, in ceil(k * (2 + log2 L) / 8) bytes; records follow one
 *     another with no padding between them;
 *   - scale rule 0 (the default): s = m / 1.5f as above;
 *     scale rule 1 (mean-abs): s = (pairwise sum of |a| over the k chosen entries, in ascending
 *     index order) / k, where the pairwise sum of x[0..n) is x[0] for n = 1 and otherwise the
 *     sum of the first floor(n/2) entries plus the sum of the rest, each summed the same way;
 *     the levels, the code rule, the residual and the decoder are those of rule 0.
 *
 * Plain single-threaded C11.  Build with -O2 -ffp-contract=off and no fast-math: every
 * floating-point operation is one IEEE binary32 operation rounded to nearest-even, the
 * precision in which the codec's scale, residual and mean are defined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_CHUNK 4096         /* [SF] item 1: the vector is cut into disjoint 4096-value chunks */
#define ORC_TOPK 64            /* [SF] item 1: the 64 largest |a| of each chunk are kept */
#define ORC_INDEX_BITS 12      /* [SF] item 3: ceil(log2(4096)) = 12 */
#define ORC_VALUE_BITS 2       /* [SF] item 2: four levels, two bits */
#define ORC_FIELD_BITS (ORC_VALUE_BITS + ORC_INDEX_BITS)
#define ORC_RECORD_BYTES ((ORC_TOPK * ORC_FIELD_BITS) / 8) /* 896 bits = 112 bytes */

#define ORC_FLAG_NONFINITE 1u
#define ORC_FLAG_BAD_RECORD 2u

#define ORC_SCALE_MAX 0        /* s = max |a| / 1.5 */
#define ORC_SCALE_MEAN_ABS 1   /* s = mean |a| over the chosen entries (variant) */

int orc_chunk(void) { return ORC_CHUNK; }
int orc_topk(void) { return ORC_TOPK; }
int orc_record_bytes(void) { return ORC_RECORD_BYTES; }

int64_t orc_num_chunks(int64_t n) { return (n + ORC_CHUNK - 1) / ORC_CHUNK; }

/* A codec: chunk length L, k entries per record, scale rule, and the derived widths. */
typedef struct {
    int L, k, rule;
    int idx_bits;      /* ceil(log2 L) ([SF] item 3) */
    int field_bits;    /* 2 + idx_bits */
    int record_bytes;  /* ceil(k * field_bits / 8) */
} orc_codec;

/* Fills cd; returns 0 when (L, k, rule) is not a codec: L a power of two in [2, 65536],
 * 1 <= k <= L, rule 0 or 1. */
static int orc_codec_init(orc_codec* cd, int L, int k, int rule) {
    int b = 0;
    if (L < 2 || L > 65536 || (L & (L - 1)) != 0) return 0;
    if (k < 1 || k > L || (rule != ORC_SCALE_MAX && rule != ORC_SCALE_MEAN_ABS)) return 0;
    while ((1 << b) < L) ++b;
    cd->L = L;
    cd->k = k;
    cd->rule = rule;
    cd->idx_bits = b;
    cd->field_bits = ORC_VALUE_BITS + b;
    cd->record_bytes = (k * cd->field_bits + 7) / 8;
    return 1;
}

/* Record bytes of codec (L, k), or -1 when it is not one. */
int orc_codec_record_bytes(int L, int k) {
    orc_codec cd;
    return orc_codec_init(&cd, L, k, ORC_SCALE_MAX) ? cd.record_bytes : -1;
}

int64_t orc_num_chunks_codec(int L, int64_t n) { return (n + L - 1) / L; }

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

/* Pairwise (recursive halving) sum of x[0..n), n >= 1, in fp32: the mean-abs scale's sum. */
float orc_pairwise_sum(const float* x, int n) {
    int h;
    if (n == 1) return x[0];
    h = n / 2;
    return orc_pairwise_sum(x, h) + orc_pairwise_sum(x + h, n - h);
}

/* ------------------------------------------------------------------------------------------
 * Record packing ([SF] per-chunk equation): k fields of 2 + idx_bits bits (64 fields of 14
 * bits for the default codec), written one bit at a time.
 * ---------------------------------------------------------------------------------------- */
static void orc_pack_record_cd(const orc_codec* cd, const uint16_t* idx, const uint8_t* code,
                               uint8_t* out) {
    int r, b;
    const uint32_t idx_mask = (1u << cd->idx_bits) - 1u;
    memset(out, 0, (size_t)cd->record_bytes);
    for (r = 0; r < cd->k; ++r) {
        uint32_t field = (uint32_t)(code[r] & 3u) | (((uint32_t)idx[r] & idx_mask) << ORC_VALUE_BITS);
        for (b = 0; b < cd->field_bits; ++b) {
            int bit = r * cd->field_bits + b;
            if ((field >> b) & 1u) out[bit >> 3] |= (uint8_t)(1u << (bit & 7));
        }
    }
}

static void orc_unpack_record_cd(const orc_codec* cd, const uint8_t* rec, uint16_t* idx,
                                 uint8_t* code) {
    int r, b;
    for (r = 0; r < cd->k; ++r) {
        uint32_t field = 0;
        for (b = 0; b < cd->field_bits; ++b) {
            int bit = r * cd->field_bits + b;
            if ((rec[bit >> 3] >> (bit & 7)) & 1u) field |= 1u << b;
        }
        code[r] = (uint8_t)(field & 3u);
        idx[r] = (uint16_t)(field >> ORC_VALUE_BITS);
    }
}

static orc_codec orc_default_codec(void) {
    orc_codec cd;
    orc_codec_init(&cd, ORC_CHUNK, ORC_TOPK, ORC_SCALE_MAX);
    return cd;
}

void orc_pack_record(const uint16_t* idx, const uint8_t* code, uint8_t* out) {
    orc_codec cd = orc_default_codec();
    orc_pack_record_cd(&cd, idx, code, out);
}

void orc_unpack_record(const uint8_t* rec, uint16_t* idx, uint8_t* code) {
    orc_codec cd = orc_default_codec();
    orc_unpack_record_cd(&cd, rec, idx, code);
}

/* idx[C][k], code[C][k] <-> payload[C][record_bytes] for codec (L, k).  Returns 0 when (L, k)
 * is not a codec (nothing written). */
int orc_pack_codec(int L, int k, const uint16_t* idx, const uint8_t* code, int64_t C,
                   uint8_t* payload) {
    orc_codec cd;
    int64_t c;
    if (!orc_codec_init(&cd, L, k, ORC_SCALE_MAX)) return 0;
    for (c = 0; c < C; ++c)
        orc_pack_record_cd(&cd, idx + c * k, code + c * k, payload + c * cd.record_bytes);
    return 1;
}

int orc_unpack_codec(int L, int k, const uint8_t* payload, int64_t C, uint16_t* idx,
                     uint8_t* code) {
    orc_codec cd;
    int64_t c;
    if (!orc_codec_init(&cd, L, k, ORC_SCALE_MAX)) return 0;
    for (c = 0; c < C; ++c)
        orc_unpack_record_cd(&cd, payload + c * cd.record_bytes, idx + c * k, code + c * k);
    return 1;
}

void orc_pack(const uint16_t* idx, const uint8_t* code, int64_t C, uint8_t* payload) {
    orc_pack_codec(ORC_CHUNK, ORC_TOPK, idx, code, C, payload);
}

void orc_unpack(const uint8_t* payload, int64_t C, uint16_t* idx, uint8_t* code) {
    orc_unpack_codec(ORC_CHUNK, ORC_TOPK, payload, C, idx, code);
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

static uint32_t orc_ef_compress_cd(const orc_codec* cd, const void* delta, int delta_is_bf16,
                                   float* ef, int64_t n, float beta, uint8_t* payload,
                                   float* scales) {
    const int L = cd->L, k = cd->k;
    int64_t C = orc_num_chunks_codec(L, n);
    int64_t c;
    uint32_t flags = 0;
    float* a = (float*)malloc(sizeof(float) * (size_t)L);
    float* mags = (float*)malloc(sizeof(float) * (size_t)k);
    int* sel = (int*)malloc(sizeof(int) * (size_t)k);
    uint16_t* idx = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)k);
    uint8_t* code = (uint8_t*)malloc((size_t)k);

    for (c = 0; c < C; ++c) {
        int64_t base = c * L;
        int j, r, top;
        float s;

        /* e <- beta * e + delta, on the zero-padded chunk */
        for (j = 0; j < L; ++j) {
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

        top = orc_topk_select(a, L, k, sel);
        if (cd->rule == ORC_SCALE_MAX) {
            s = orc_scale(fabsf(a[top]));
        } else {
            for (r = 0; r < k; ++r) mags[r] = fabsf(a[sel[r]]);
            s = orc_pairwise_sum(mags, k) / (float)k;
        }

        for (r = 0; r < k; ++r) {
            float v = a[sel[r]];
            code[r] = (uint8_t)orc_code(v, s);
            idx[r] = (uint16_t)sel[r];
            a[sel[r]] = v - orc_level(code[r], s); /* residual at a transmitted position */
        }

        for (j = 0; j < L; ++j)
            if (base + j < n) ef[base + j] = a[j];

        orc_pack_record_cd(cd, idx, code, payload + c * cd->record_bytes);
        scales[c] = s;
    }
    free(a);
    free(mags);
    free(sel);
    free(idx);
    free(code);
    return flags;
}

uint32_t orc_ef_compress(const void* delta, int delta_is_bf16, float* ef, int64_t n, float beta,
                         uint8_t* payload, float* scales) {
    orc_codec cd = orc_default_codec();
    return orc_ef_compress_cd(&cd, delta, delta_is_bf16, ef, n, beta, payload, scales);
}

/* The sender for codec (L, k, rule); payload holds ceil(n / L) records of
 * orc_codec_record_bytes(L, k) bytes.  Returns 0xffffffff when (L, k, rule) is not a codec. */
uint32_t orc_ef_compress_codec(int L, int k, int rule, const void* delta, int delta_is_bf16,
                               float* ef, int64_t n, float beta, uint8_t* payload,
                               float* scales) {
    orc_codec cd;
    if (!orc_codec_init(&cd, L, k, rule)) return 0xffffffffu;
    return orc_ef_compress_cd(&cd, delta, delta_is_bf16, ef, n, beta, payload, scales);
}

/* ------------------------------------------------------------------------------------------
 * Receiver: decode P peers' records and take their mean, optionally followed by the outer
 * step theta <- theta - lr * mean ([SF] item 3, "Sparse aggregation can improve model
 * quality"; [SF] "Why DiLoCo Alone Isn't Enough" for the pseudo-gradient's sign).
 *
 * payloads[p]: C * 112 bytes; scales[p]: C floats; mean_out: n floats (overwritten);
 * theta: n floats or NULL.  Returns flag bit 1 when some record was rejected.
 * ---------------------------------------------------------------------------------------- */
static int orc_record_ok(const uint16_t* idx, int k, float s) {
    int r;
    if (isnan(s) || isinf(s) || s < 0.0f) return 0;
    for (r = 1; r < k; ++r)
        if (!(idx[r - 1] < idx[r])) return 0;
    return 1;
}

static uint32_t orc_decode_aggregate_cd(const orc_codec* cd, const uint8_t* const* payloads,
                                        const float* const* scales, int P, int64_t n,
                                        float* mean_out, float* theta, float lr) {
    const int L = cd->L, k = cd->k;
    int64_t C = orc_num_chunks_codec(L, n);
    int64_t c;
    uint32_t flags = 0;
    float* acc = (float*)malloc(sizeof(float) * (size_t)L);
    uint16_t* idx = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)k);
    uint8_t* code = (uint8_t*)malloc((size_t)k);

    for (c = 0; c < C; ++c) {
        int64_t base = c * L;
        int p, r, j;
        for (j = 0; j < L; ++j) acc[j] = 0.0f;
        for (p = 0; p < P; ++p) {
            float s = scales[p][c];
            orc_unpack_record_cd(cd, payloads[p] + c * cd->record_bytes, idx, code);
            if (!orc_record_ok(idx, k, s)) {
                flags |= ORC_FLAG_BAD_RECORD;
                continue;
            }
            for (r = 0; r < k; ++r)
                if (base + idx[r] < n) acc[idx[r]] += orc_level(code[r], s);
        }
        for (j = 0; j < L; ++j) {
            int64_t i = base + j;
            if (i >= n) break;
            mean_out[i] = acc[j] / (float)P;
            if (theta) theta[i] = fmaf(-lr, mean_out[i], theta[i]);
        }
    }
    free(acc);
    free(idx);
    free(code);
    return flags;
}

uint32_t orc_decode_aggregate(const uint8_t* const* payloads, const float* const* scales, int P,
                              int64_t n, float* mean_out, float* theta, float lr) {
    orc_codec cd = orc_default_codec();
    return orc_decode_aggregate_cd(&cd, payloads, scales, P, n, mean_out, theta, lr);
}

/* The receiver for codec (L, k); 0xffffffff when (L, k) is not a codec. */
uint32_t orc_decode_aggregate_codec(int L, int k, const uint8_t* const* payloads,
                                    const float* const* scales, int P, int64_t n,
                                    float* mean_out, float* theta, float lr) {
    orc_codec cd;
    if (!orc_codec_init(&cd, L, k, ORC_SCALE_MAX)) return 0xffffffffu;
    return orc_decode_aggregate_cd(&cd, payloads, scales, P, n, mean_out, theta, lr);
}

/* ------------------------------------------------------------------------------------------
 * Receiver statistics per peer, for screening updates that look unlike the rest ([SF] "What
 * the Blockchain Does (and Doesn't Do)": an update built to game the screening is
 * distributed differently from an honest one).  Over the k entries of every accepted record
 * of peer p:
 *   big[p]       entries with the magnitude bit set (|q| = 1.5 s)
 *   negative[p]  entries with the sign bit set
 *   max_scale[p] the largest scale among accepted records (0 if none)
 *   sumsq[p]     the sum of q^2 (fp64; q^2 is exact in fp64), records in chunk order
 * and rejected[p], the number of rejected records.  Arrays of P, overwritten.
 * ---------------------------------------------------------------------------------------- */
static void orc_peer_stats_cd(const orc_codec* cd, const uint8_t* const* payloads,
                              const float* const* scales, int P, int64_t n, uint32_t* rejected,
                              uint32_t* big, uint32_t* negative, float* max_scale,
                              double* sumsq) {
    const int k = cd->k;
    int64_t C = orc_num_chunks_codec(cd->L, n);
    int p;
    uint16_t* idx = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)k);
    uint8_t* code = (uint8_t*)malloc((size_t)k);
    for (p = 0; p < P; ++p) {
        int64_t c;
        rejected[p] = big[p] = negative[p] = 0;
        max_scale[p] = 0.0f;
        sumsq[p] = 0.0;
        for (c = 0; c < C; ++c) {
            float s = scales[p][c];
            int r;
            orc_unpack_record_cd(cd, payloads[p] + c * cd->record_bytes, idx, code);
            if (!orc_record_ok(idx, k, s)) {
                rejected[p] += 1;
                continue;
            }
            if (s > max_scale[p]) max_scale[p] = s;
            for (r = 0; r < k; ++r) {
                double q = (double)orc_level(code[r], s);
                big[p] += code[r] & 1u;
                negative[p] += (code[r] >> 1) & 1u;
                sumsq[p] += q * q;
            }
        }
    }
    free(idx);
    free(code);
}

void orc_peer_stats(const uint8_t* const* payloads, const float* const* scales, int P, int64_t n,
                    uint32_t* rejected, uint32_t* big, uint32_t* negative, float* max_scale,
                    double* sumsq) {
    orc_codec cd = orc_default_codec();
    orc_peer_stats_cd(&cd, payloads, scales, P, n, rejected, big, negative, max_scale, sumsq);
}

/* Statistics for codec (L, k); returns 0 (nothing written) when (L, k) is not a codec. */
int orc_peer_stats_codec(int L, int k, const uint8_t* const* payloads, const float* const* scales,
                         int P, int64_t n, uint32_t* rejected, uint32_t* big, uint32_t* negative,
                         float* max_scale, double* sumsq) {
    orc_codec cd;
    if (!orc_codec_init(&cd, L, k, ORC_SCALE_MAX)) return 0;
    orc_peer_stats_cd(&cd, payloads, scales, P, n, rejected, big, negative, max_scale, sumsq);
    return 1;
}
