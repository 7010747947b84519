// Receiver kernel of the SparseLoCo codec: decode P peers' records, take their mean, and
// optionally apply the outer step theta <- theta - lr * mean, in one pass over HBM.
// Templated on the record geometry (chunk length L, k) and on the per-peer statistics; the
// translation units that include this header instantiate it (the default codec in
// decode_aggregate.cu, the variants in decode_aggregate_variants.cu).  The figures below are
// the default codec's.
//
// Method: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
// Pre-Training", "SparseLoCo: Three Compression Levers in One Pass" (item 3: the receiver
// rebuilds positions from the 12-bit indices) and "Why Extreme Sparsity Doesn't Break
// Convergence" ("Sparse aggregation can improve model quality": the peers' sparse updates
// are aggregated); "Why DiLoCo Alone Isn't Enough" for the pseudo-gradient's sign.
//
// Design (HBM-bound: P x 116 B read per chunk, 16 KB of mean written, 32 KB of theta read and
// written when the outer step is fused):
//   - one 256-thread CTA per chunk at a time; the grid runs in waves of the resident CTAs,
//     each CTA taking 32 chunks spaced a wave apart, so the chunks in flight stay close
//     together in memory; while a chunk is worked on, the next chunk's theta (one 16 KB bulk
//     copy, TMA) and its P records (one bulk copy each where the shape allows, else 16-byte
//     cp.async pieces spread over the threads) fly into a shared-memory stage, all completing
//     on one mbarrier; the next chunk's P scales travel as plain loads into registers (lane l
//     of warp w holds peer 8 l + w's); a mean of a few peers without theta or statistics
//     takes a lean shape instead (128 threads, four record stages, no theta stage, warp 0
//     free of copies);
//   - each warp unpacks whole records (one peer at a time): the 64 14-bit fields, a check that
//     the indices ascend strictly and the scale is finite and non-negative, and the decoded
//     value of every entry, stored as (position, value) pairs (+0.0 for a rejected record, an
//     exact identity in the adds; with statistics, the warp also counts the record's magnitude
//     and sign bits and keeps them beside its scale);
//   - then one warp adds the peers into a 16 KB shared accumulator in order p = 0..P-1, two
//     entries per lane (distinct positions within a valid record, so a lane reads both sums
//     before writing either back: one shared-memory round trip per peer), so every position
//     is summed in fp32 in peer order from +0.0, as a plain sequential loop over peers would,
//     with no atomics and no branch per peer; a single warp keeps every lane busy and the instruction
//     count minimal, while the other resident CTAs keep the SM fed (with statistics, threads
//     of warps 1-2 meanwhile fold one record each into per-CTA per-peer totals, flushed with
//     atomics at the end);
//   - the dense pass divides by P (correctly rounded, with a precomputed reciprocal; one
//     multiply when P is a power of two, whose reciprocal is exact), stores the mean and the
//     updated theta with plain 16-byte stores and clears the accumulator.  Peers
//     are unpacked in groups of up to 64 (32 for k = 128 at L = 8192; at L = 4096 the k = 128
//     entries are the raw 2-byte fields and a per-peer scale), so shared memory stays bounded
//     for any P.
#pragma once

#include <cfloat>

#include "spl_device.cuh"
#include "spl_kernels.h"

namespace spl {
namespace {

// Per-codec sizes of the receiver (default: 256 threads, 512 positions and 4 vectors per
// thread of each warp, groups of 64 peers, two entries per lane, seven 16-byte pieces per
// record, one prefetch stage: chunk c + G's copies fly while chunk c is worked on).  L = 2048
// takes 128 threads (8 CTAs per SM hide its per-chunk fixed costs at the usual peer counts:
// 0.67 -> 0.56 ms at 24 peers, 2^28 values; 200 peers, where shared memory allows fewer CTAs,
// run 11 % slower), L = 8192 takes 512, so a warp still holds 512 positions.
// kLean (L = 4096, k <= 64, a few peers, no theta, no statistics): 128 threads, so 8 CTAs share
// an SM, and four prefetch stages (chunks c + G .. c + 4G), cheap without a theta stage: the
// 8-peer mean of 2^27 values goes from 63 % to 73 % of the measured copy bandwidth.
template <class Geo, bool kLean = false, bool kStats = false>
struct RecvShape {
    static constexpr int kChunk = Geo::kChunk;
    static constexpr int kTopK = Geo::kTopK;
    static_assert(!kLean || (kChunk == 4096 && kTopK <= 64), "lean receiver shape");
    static constexpr int kThreads = kLean ? 128 : (kChunk == 8192 ? 512 : (kChunk == 2048 ? 128 : 256));
    static constexpr bool kIsLean = kLean;
    static constexpr int kStages = kLean ? 4 : 1;           // prefetch stages (<= 4 mbarriers)
    static constexpr int kWarps = kThreads / 32;
    static constexpr int kSlice = kChunk / kWarps;          // positions per warp
    static constexpr int kVec = kSlice / 128;               // vectors of 4 per thread
    // entries: (position, value) pairs of 8 bytes; for k = 128 at 256 threads the raw 2-byte
    // fields, decoded by the adding warp with the peer's scale, so that 64 peers' entries fit
    // 16 KB and one pass takes them all (2.85 -> 2.71 ms for the 24-peer decode; the k <= 64
    // decode measured 1.3 % slower that way, L = 8192 at 512 threads 3.5 %)
    static constexpr bool kFieldEntries = kTopK > 64 && kThreads == 256;
    static constexpr int kEntryBytes = kFieldEntries ? 2 : 8;
    // peers unpacked per pass, a multiple of the warp count (peer p is unpacked by warp p mod
    // W): 32 for 8-byte entries of k = 128, so the entries stay at 32 KB
    static constexpr int kGroup = kTopK <= 64 || kFieldEntries ? 64 : 32;
    static constexpr int kPerLane = kTopK / 32;             // entries per lane of a record
    static constexpr int kPieceBytes = Geo::kVecRecords ? 16 : 4;
    static constexpr int kPieces = Geo::kRecordBytes / kPieceBytes;   // copies per record
    // records of a multiple of 16 bytes as one bulk copy each, from the last warp (measured
    // per shape: the 24-peer decode with theta 2.137 -> 2.086 ms, L = 8192 2.44 -> 2.33 ms;
    // the lean shape (3 %), k = 128 at 256 threads (3 %) and statistics (0.4 %) measured
    // slower that way and keep 16-byte cp.async pieces spread over the threads)
    static constexpr bool kBulkRecords =
        Geo::kVecRecords && !kLean && !kStats && (kTopK <= 64 || kThreads == 512);
    static constexpr int kMinBlocks = kThreads == 256 && kChunk > 4096 ? 2 : 1024 / kThreads;
    // scales a lane carries: peer (32 W) i + W lane + w in slot i, for up to 256 peers
    static constexpr int kScalesPerLane = (kMaxPeers + 32 * kWarps - 1) / (32 * kWarps);
    static_assert(kScalesPerLane <= 2, "scale slots per lane");
};

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Largest P the lean shape takes (its record stages and entries then still let 7-8 CTAs share
// an SM).
constexpr int kLeanMaxPeers = 16;

// Dynamic shared memory for P peers (offsets 16-byte aligned), G = min(P, group):
//   bar[4] | theta stage [S][4096] f32 (with theta only) | record stage [S][P][112] (+16) |
//   acc [4096] f32 | entries [G][k] (position, value), or for k > 64 raw fields [G][k] u16
//   and the peers' scales [G] f32 | validity [G] u32 (read with statistics only) |
//   with statistics only: (scale, magnitude | sign << 8 bit counts) [G] | per-peer totals of
//   this CTA: sum of squares and its Kahan compensation [2][P] f32 | rejected, big, negative
//   [3][P] u32 | max scale [P] f32
template <class Geo, class S>
struct Layout {
    size_t bar, theta, rec, acc, ent, scl, ok, sgrp, st_sq, st_cnt, st_max, total;
    __host__ __device__ Layout(int P, bool stats, bool with_theta) {
        const size_t G = static_cast<size_t>(P < S::kGroup ? P : S::kGroup);
        bar = 0;
        theta = 32;
        rec = theta + (with_theta ? S::kStages * S::kChunk * 4 : 0);
        acc = rec + align16(S::kStages * static_cast<size_t>(P) * Geo::kRecordBytes) + 16;
        ent = acc + S::kChunk * 4;
        scl = ent + align16(G * S::kTopK * S::kEntryBytes);
        ok = scl + (S::kFieldEntries ? align16(G * 4) : 0);
        sgrp = ok + align16(G * 4);
        st_sq = sgrp + align16(G * 8);
        st_cnt = st_sq + align16(static_cast<size_t>(P) * 8);
        st_max = st_cnt + align16(3 * static_cast<size_t>(P) * 4);
        total = stats ? st_max + align16(static_cast<size_t>(P) * 4) : sgrp;
    }
};

// All threads: start chunk c's copies into one stage.  Where the shape takes records as bulk
// copies (kBulkRecords), the last warp starts one per record and theta's, and its first lane
// arrives with all their bytes (one arrival per phase).  Otherwise thread 0 arrives with the
// expected theta bytes (a full chunk when the outer step is fused) and starts its bulk copy; the
// record pieces (7 x 16 B per peer; 4-byte pieces for a variant whose records are not 16-byte
// aligned) are spread over the threads, each of which arrives once its own copies have
// landed.  In the lean shape piece i comes from thread 32 + i (from warp 0 only past
// kThreads - 32 pieces), so that warp 0 goes straight on to the ordered adds: 8-peer mean of
// 2^27 values 0.0985 -> 0.0959 ms; the wide shape with theta measured 0.6 % slower that way.
// Arrivals per phase: min(pieces, threads) + 1.
template <class Geo, class S>
__device__ __forceinline__ void prefetch(const DecodeTable& tab, int P, int64_t c, int64_t C,
                                         bool full, const float* theta, uint64_t* bar,
                                         uint8_t* st_rec, float* st_theta, int tid) {
    constexpr int kThreads = S::kThreads;
    constexpr int kChunk = S::kChunk;
    constexpr int kRecordBytes = Geo::kRecordBytes;
    constexpr int kPieces = S::kPieces;
    constexpr int kPieceBytes = S::kPieceBytes;
    if constexpr (S::kBulkRecords) {
        // one bulk copy per record, from the last warp, with theta's; one arrival with all
        // the bytes
        if (tid >= kThreads - 32) {
            const int lane = tid - (kThreads - 32);
            fence_async_smem();
            if (lane == 0) {
                const bool th = theta != nullptr && full;
                mbar_expect_tx(bar, static_cast<uint32_t>(P * kRecordBytes) + (th ? kChunk * 4u : 0u));
                if (th) bulk_load(st_theta, theta + c * kChunk, kChunk * 4, bar);
            }
            __syncwarp();
            for (int p = lane; p < P; p += 32)
                if (SPL_CHECK(c < C && p < P, kSiteRecCopy, c))
                    bulk_load(st_rec + p * kRecordBytes, tab.payload[p] + c * kRecordBytes,
                              kRecordBytes, bar);
        }
        return;
    }
    if (tid == 0) {
        if (theta != nullptr && full) {
            fence_async_smem();
            mbar_expect_tx(bar, kChunk * 4);
            bulk_load(st_theta, theta + c * kChunk, kChunk * 4, bar);
        } else {
            mbar_arrive(bar);
        }
    }
    const int pieces = P * kPieces;
    const int t = !S::kIsLean ? tid : (tid >= 32 ? tid - 32 : tid + kThreads - 32);   // first piece
    if (t < pieces) {
        for (int i = t; i < pieces; i += kThreads) {
            const int p = i / kPieces;
            const int w = i - p * kPieces;
            if (!SPL_CHECK(c < C && p < P, kSiteRecCopy, c)) continue;
            if constexpr (kPieceBytes == 16)
                cp_async16(st_rec + i * 16, tab.payload[p] + c * kRecordBytes + w * 16);
            else
                cp_async4(st_rec + i * 4, tab.payload[p] + c * kRecordBytes + w * 4);
        }
        cp_async_arrive(bar);
    }
}

template <class Geo, bool kLean, bool kStats, bool kPow2>
__global__ void __launch_bounds__(RecvShape<Geo, kLean, kStats>::kThreads, RecvShape<Geo, kLean, kStats>::kMinBlocks)
k_decode_aggregate(const DecodeTable tab, int P, float rp, int64_t n, float* __restrict__ mean,
                   float* __restrict__ theta_arg, float neg_lr, bool validate,
                   PeerStats* __restrict__ stats, uint32_t* __restrict__ flags, int ctas,
                   int per_cta) {
    using S = RecvShape<Geo, kLean, kStats>;
    constexpr int kStages = S::kStages;
    // the lean shape is launched without theta: knowing so here drops its code and registers
    float* __restrict__ const theta = kLean ? nullptr : theta_arg;
    constexpr int kThreads = S::kThreads;
    constexpr int kWarps = S::kWarps;
    constexpr int kChunk = S::kChunk;
    constexpr int kTopK = S::kTopK;
    constexpr int kSlice = S::kSlice;
    constexpr int kVec = S::kVec;
    constexpr int kGroup = S::kGroup;
    constexpr int kPerLane = S::kPerLane;
    constexpr int kRecordBytes = Geo::kRecordBytes;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const Layout<Geo, S> L(P, kStats, theta != nullptr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + L.bar);
    float* st_theta = reinterpret_cast<float*>(smem_raw + L.theta);
    uint8_t* st_rec = smem_raw + L.rec;
    float* acc = reinterpret_cast<float*>(smem_raw + L.acc);
    uint2* ent = reinterpret_cast<uint2*>(smem_raw + L.ent);
    uint16_t* ent16 = reinterpret_cast<uint16_t*>(smem_raw + L.ent);   // k > 64: raw fields
    float* scl = reinterpret_cast<float*>(smem_raw + L.scl);         // k > 64: 0 if rejected
    uint32_t* okp = reinterpret_cast<uint32_t*>(smem_raw + L.ok);
    uint2* sgrp = reinterpret_cast<uint2*>(smem_raw + L.sgrp);
    float* st_sum = reinterpret_cast<float*>(smem_raw + L.st_sq);        // [P]
    float* st_comp = st_sum + P;                                           // [P]
    uint32_t* st_cnt = reinterpret_cast<uint32_t*>(smem_raw + L.st_cnt);   // [3][P]
    float* st_max = reinterpret_cast<float*>(smem_raw + L.st_max);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t C = (n + kChunk - 1) / kChunk;
    const int64_t G = ctas;   // between one CTA's chunks
    const ChunkSpan span = cta_chunks(C, ctas, per_cta, blockIdx.x);
    const int64_t end = span.end;
    if (span.first >= end) return;
    const float pf = static_cast<float>(P);
    const int slice0 = kSlice * warp;    // this warp's positions: slice0 + 128 v + 4 lane + u
    constexpr int kSpl = S::kScalesPerLane;
    int my_peer[kSpl];                            // the peers whose scales this lane carries
#pragma unroll
    for (int i = 0; i < kSpl; ++i) my_peer[i] = 32 * kWarps * i + kWarps * lane + warp;

#pragma unroll
    for (int v = 0; v < kVec; ++v)
        *reinterpret_cast<float4*>(&acc[slice0 + 128 * v + 4 * lane]) = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (kStats) {
        for (int p = tid; p < P; p += kThreads) {
            st_sum[p] = st_comp[p] = 0.0f;
            st_cnt[p] = st_cnt[P + p] = st_cnt[2 * P + p] = 0u;
            st_max[p] = 0.0f;
        }
    }
    if (tid == 0) {
        const uint32_t arrivals =
            S::kBulkRecords ? 1u : static_cast<uint32_t>(min(P * S::kPieces, kThreads) + 1);
        for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], arrivals);
    }
    __syncthreads();
    for (int st = 0; st < kStages; ++st) {
        const int64_t c = span.first + st * G;
        if (c < end)
            prefetch<Geo, S>(tab, P, c, C, (c + 1) * kChunk <= n, theta, &bars[st],
                     st_rec + st * P * kRecordBytes, st_theta + st * kChunk, tid);
    }
    float sc_cur[kSpl];
#pragma unroll
    for (int i = 0; i < kSpl; ++i)
        sc_cur[i] = my_peer[i] < P ? __ldcs(tab.scale[my_peer[i]] + span.first) : 0.0f;

    bool bad = false;
    bool aborted = false;
    int it = 0;
    int64_t c = span.first;
    for (; c < end; c += G, ++it) {
        const int st = it % kStages;
        const uint32_t parity = static_cast<uint32_t>(it / kStages) & 1u;
        const uint8_t* rec = st_rec + st * P * kRecordBytes;
        const int64_t base = c * kChunk;
        const bool full = base + kChunk <= n;
        const int valid = full ? kChunk : static_cast<int>(n - base);

        const bool timed_out = !mbar_wait(&bars[st], parity);
        float4 th[kVec];
        if (theta != nullptr && full) {
#pragma unroll
            for (int v = 0; v < kVec; ++v)
                th[v] = *reinterpret_cast<const float4*>(
                    &st_theta[st * kChunk + slice0 + 128 * v + 4 * lane]);
        }
        float sc_next[kSpl];
#pragma unroll
        for (int i = 0; i < kSpl; ++i) sc_next[i] = 0.0f;

        for (int g0 = 0; g0 < P; g0 += kGroup) {
            const int gn = P - g0 < kGroup ? P - g0 : kGroup;
            // ---- unpack: one warp per peer --------------------------------------------
            for (int g = warp; g < gn; g += kWarps) {
                const int p = g0 + g;
                const uint32_t* words = reinterpret_cast<const uint32_t*>(rec + p * kRecordBytes);
                // entry lane + 32 m of the record, m = 0 .. k/32 - 1 (its two words lie inside
                // the stage and the 16 bytes after it)
                uint32_t f[kPerLane], ix[kPerLane];
#pragma unroll
                for (int m = 0; m < kPerLane; ++m) {
                    f[m] = SPL_CHECK(p < P && g < kGroup, kSiteRecStage, p)
                               ? record_field_fs<Geo::kFieldBits>(words, lane + 32 * m) : 0u;
                    ix[m] = f[m] >> 2;
                }
                const int slot = p / (32 * kWarps);   // the same for the whole warp
                const float sv = (kSpl == 1 || slot == 0) ? sc_cur[0] : sc_cur[kSpl - 1];
                const float s = __shfl_sync(0xffffffffu, sv, (p / kWarps) % 32);
                bool ok = true;
                if (validate) {   // uniform: a launch argument
                    // indices strictly ascending: each entry below the next one
                    bool asc = true;
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) {
                        uint32_t next = __shfl_down_sync(0xffffffffu, ix[m], 1);
                        if (m + 1 < kPerLane) {
                            const uint32_t first = __shfl_sync(0xffffffffu, ix[m + 1 < kPerLane ? m + 1 : m], 0);
                            if (lane == 31) next = first;
                            asc = asc && ix[m] < next;
                        } else {
                            asc = asc && (lane == 31 || ix[m] < next);
                        }
                    }
                    ok = __all_sync(0xffffffffu, asc) && s >= 0.0f && s <= FLT_MAX;
                }
                if constexpr (kStats) {
                    // the record's magnitude bits (low byte) and sign bits (<< 8), summed over
                    // the warp in one reduction outside the branch on ok (ballots inside it cost
                    // the unpack a fifth more instructions)
                    uint32_t bits = 0;
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) bits += (f[m] & 1u) + ((f[m] & 2u) << 7);
                    bits = __reduce_add_sync(0xffffffffu, bits);
                    if (ok && lane == 0) sgrp[g] = make_uint2(__float_as_uint(s), bits);
                }
                // a rejected record adds +0.0 at its own (in-chunk) positions: the accumulator
                // starts at +0.0 and a correctly rounded sum is -0.0 only for (-0) + (-0), so it
                // never holds -0.0, and x + (+0.0) is x for every value it can hold (a NaN
                // there is already the canonical one); the adds need no per-peer branch
                if constexpr (S::kFieldEntries) {   // the fields, and the scale they decode with
                    uint16_t* eg = ent16 + g * kTopK;
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) eg[lane + 32 * m] = static_cast<uint16_t>(f[m]);
                    if (lane == 0) scl[g] = ok ? s : 0.0f;   // +-0.0 values: as above
                } else {
                    uint2* eg = ent + g * kTopK;
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m)
                        eg[lane + 32 * m] = make_uint2(
                            ix[m], ok ? __float_as_uint(level_value(f[m] & 3u, s)) : 0u);
                }
                bad = bad || !ok;
                if (kStats && lane == 0) okp[g] = ok ? 1u : 0u;
            }
            const bool last = g0 + kGroup >= P;
            if (last) {
                if (__syncthreads_or(timed_out)) {
                    aborted = true;
                    break;
                }
                // the stage has been read: start chunk c + S G's copies, and c + G's scales
                const int64_t c2 = c + kStages * G;
                if (c2 < end)
                    prefetch<Geo, S>(tab, P, c2, C, (c2 + 1) * kChunk <= n, theta, &bars[st],
                             st_rec + st * P * kRecordBytes, st_theta + st * kChunk, tid);
#pragma unroll
                for (int i = 0; i < kSpl; ++i)
                    if (my_peer[i] < P && c + G < end) sc_next[i] = __ldcs(tab.scale[my_peer[i]] + c + G);
            } else {
                __syncthreads();
            }
            // ---- the other warps, meanwhile: per-peer statistics, one record per thread ----
            // (a group holds at most 64 peers; peer p is always thread 32 + p mod 64)
            if (kStats && tid >= 32 && tid - 32 < gn &&
                SPL_CHECK(g0 + tid - 32 < P, kSiteStats, g0 + tid - 32)) {
                const int g = tid - 32;
                const int p = g0 + g;
                if (okp[g] == 0u) {
                    st_cnt[p] += 1u;
                } else {
                    const uint2 sg = sgrp[g];
                    const float s = __uint_as_float(sg.x);
                    const uint32_t nbig = sg.y & 0xffu;
                    const uint32_t nneg = sg.y >> 8;
                    const float lo = level_value(0u, s);
                    const float hi = level_value(1u, s);
                    // every entry decodes to +-RN(0.5 s) or +-RN(1.5 s): the record's sum of
                    // squares from the two counts, in fp32 (fp64 is scarce on this GPU), added
                    // to the CTA's total with Kahan compensation
                    const float t = __fmaf_rn(__fmul_rn(hi, hi), static_cast<float>(nbig),
                                              __fmul_rn(__fmul_rn(lo, lo),
                                                        static_cast<float>(kTopK - nbig)));
                    const float y = __fsub_rn(t, st_comp[p]);
                    const float z = __fadd_rn(st_sum[p], y);
                    st_comp[p] = __fsub_rn(__fsub_rn(z, st_sum[p]), y);
                    st_sum[p] = z;
                    st_cnt[P + p] += nbig;
                    st_cnt[2 * P + p] += nneg;
                    st_max[p] = fmaxf(st_max[p], s);
                }
            }
            // ---- one warp: add the peers in order, k/32 entries per lane ------------------
            if (S::kFieldEntries && warp == 0) {
                uint32_t fn[kPerLane];
#pragma unroll
                for (int m = 0; m < kPerLane; ++m) fn[m] = ent16[lane + 32 * m];
                float sn = scl[0];
                for (int g = 0; g < gn; ++g) {
                    uint32_t fe[kPerLane];
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) fe[m] = fn[m];
                    const float s = sn;
                    const int gnext = g + 1 < gn ? g + 1 : g;
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) fn[m] = ent16[gnext * kTopK + lane + 32 * m];
                    sn = scl[gnext];
                    // level_value, with the peer's two magnitudes formed once
                    const uint32_t lo = __float_as_uint(__fmul_rn(0.5f, s));
                    const uint32_t hi = __float_as_uint(__fmul_rn(1.5f, s));
                    // an accepted record's positions are distinct and a rejected one adds
                    // +0.0, so a lane's k/32 sums may be read before any of them is written
                    // back: one shared-memory round trip per peer instead of k/32
                    float a[kPerLane];
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) {
                        const uint32_t pos = fe[m] >> 2;
                        a[m] = SPL_CHECK(pos < static_cast<uint32_t>(kChunk), kSiteAcc, pos) ? acc[pos] : 0.0f;
                    }
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) {
                        const uint32_t pos = fe[m] >> 2;
                        const float v = __uint_as_float(((fe[m] & 1u) ? hi : lo) ^ ((fe[m] & 2u) << 30));
                        if (SPL_CHECK(pos < static_cast<uint32_t>(kChunk), kSiteAcc, pos))
                            acc[pos] = __fadd_rn(a[m], v);
                    }
                    __syncwarp();
                }
            } else if (warp == 0) {
                uint2 en[kPerLane];
#pragma unroll
                for (int m = 0; m < kPerLane; ++m) en[m] = ent[lane + 32 * m];
                for (int g = 0; g < gn; ++g) {
                    uint2 e[kPerLane];
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) e[m] = en[m];
                    // the next peer's entries (after the last peer: its own again, unused)
                    const int gnext = g + 1 < gn ? g + 1 : g;
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m) en[m] = ent[gnext * kTopK + lane + 32 * m];
                    // the lane's sums are all read before any is written back (see above)
                    float a[kPerLane];
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m)
                        a[m] = SPL_CHECK(e[m].x < static_cast<uint32_t>(kChunk), kSiteAcc, e[m].x)
                                   ? acc[e[m].x] : 0.0f;
#pragma unroll
                    for (int m = 0; m < kPerLane; ++m)
                        if (SPL_CHECK(e[m].x < static_cast<uint32_t>(kChunk), kSiteAcc, e[m].x))
                            acc[e[m].x] = __fadd_rn(a[m], __uint_as_float(e[m].y));
                    __syncwarp();
                }
            }
            __syncthreads();   // the accumulator is complete; entries are rewritten next pass
        }
        if (aborted) break;
#pragma unroll
        for (int i = 0; i < kSpl; ++i) sc_cur[i] = sc_next[i];

        // ---- dense pass: mean, outer step --------------------------------------------------
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            const int j0 = slice0 + 128 * v + 4 * lane;
            float4 m4 = *reinterpret_cast<const float4*>(&acc[j0]);
            *reinterpret_cast<float4*>(&acc[j0]) = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (kPow2) {   // 1/P = 2^-k exactly: the rounded product is the rounded quotient
                m4.x = __fmul_rn(m4.x, rp);
                m4.y = __fmul_rn(m4.y, rp);
                m4.z = __fmul_rn(m4.z, rp);
                m4.w = __fmul_rn(m4.w, rp);
            } else {
                m4.x = div_rn(m4.x, pf, rp);
                m4.y = div_rn(m4.y, pf, rp);
                m4.z = div_rn(m4.z, pf, rp);
                m4.w = div_rn(m4.w, pf, rp);
            }
            if (!SPL_CHECK(j0 + 3 < kChunk, kSiteMean, j0)) continue;
            if (full) {
                // plain stores: with the chunks in wave order they beat streaming (evict-first)
                // ones, 2.031 against 2.050 ms for the 24-peer receive step at 2^30 values, and
                // 0.0956 against 0.0962 ms for the 8-peer mean of 2^27 values
                *reinterpret_cast<float4*>(mean + base + j0) = m4;
                if (theta != nullptr) {
                    float4 t4 = th[v];
                    t4.x = __fmaf_rn(neg_lr, m4.x, t4.x);
                    t4.y = __fmaf_rn(neg_lr, m4.y, t4.y);
                    t4.z = __fmaf_rn(neg_lr, m4.z, t4.z);
                    t4.w = __fmaf_rn(neg_lr, m4.w, t4.w);
                    *reinterpret_cast<float4*>(theta + base + j0) = t4;
                }
            } else {
                const float m[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = j0 + u;
                    if (j < valid && SPL_CHECK(base + j < n, kSiteMean, j)) {
                        mean[base + j] = m[u];
                        if (theta != nullptr)
                            theta[base + j] = __fmaf_rn(neg_lr, m[u], theta[base + j]);
                    }
                }
            }
        }
    }
    bool copy_pending = false;
    if (aborted && tid == 0) {
        // copies still in flight may land late: wait for them (bounded) before the CTA's
        // shared memory is released: the stage that timed out and any armed after it (if a
        // wait runs out again, the block exits with a copy possibly in flight: reported)
        for (int k = 0; k < kStages; ++k) {
            const int it2 = it + k;
            if (c + k * G < end &&
                !mbar_wait(&bars[it2 % kStages], static_cast<uint32_t>(it2 / kStages) & 1u))
                copy_pending = true;
        }
    }
    if constexpr (kStats) {
        __syncthreads();
        for (int p = tid; p < P; p += kThreads) {
            PeerStats* o = stats + p;
            if (st_cnt[p]) atomicAdd(&o->rejected, st_cnt[p]);
            if (st_cnt[P + p]) atomicAdd(&o->big, st_cnt[P + p]);
            if (st_cnt[2 * P + p]) atomicAdd(&o->negative, st_cnt[2 * P + p]);
            if (st_max[p] > 0.0f)   // non-negative floats order like their bit patterns
                atomicMax(reinterpret_cast<unsigned int*>(&o->max_scale), __float_as_uint(st_max[p]));
            if (st_sum[p] != 0.0f)
                atomicAdd(&o->sumsq, static_cast<double>(st_sum[p]) - static_cast<double>(st_comp[p]));
        }
    }
    if (flags != nullptr) {
        if (bad && lane == 0) atomicOr(flags, kFlagBadRecord);
        if (aborted && tid == 0) atomicOr(flags, kFlagTimeout | (copy_pending ? kFlagCopyPending : 0u));
    }
}

template <class Geo, bool kLean, bool kStats, bool kPow2>
cudaError_t launch_kernel(const DecodeTable& tab, int P, int64_t n, int64_t C, float* mean,
                          float* theta, float lr, bool validate, PeerStats* stats, uint32_t* flags,
                          cudaStream_t stream) {
    using S = RecvShape<Geo, kLean, kStats>;
    const size_t smem = Layout<Geo, S>(P, kStats, theta != nullptr).total;
    const void* kern = reinterpret_cast<const void*>(&k_decode_aggregate<Geo, kLean, kStats, kPow2>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    constexpr int kThreads = S::kThreads;
    const int resident = persistent_grid(kern, kThreads, smem);
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    const int grid = wave_grid(C, resident, kRecvChunksPerCta);
    const float rp = 1.0f / static_cast<float>(P);   // correctly rounded on the host
    k_decode_aggregate<Geo, kLean, kStats, kPow2><<<grid, kThreads, smem, stream>>>(
        tab, P, rp, n, mean, theta, -lr, validate || kStats, stats, flags, resident,
        kRecvChunksPerCta);
    return cudaGetLastError();
}

// For P a power of two the mean is one multiply by 1/P = 2^-k (exact), else the corrected
// reciprocal division; the choice is made per launch, so each kernel has one straight path.
template <class Geo, bool kStats>
cudaError_t launch_decode(const DecodeTable& tab, int P, int64_t n, float* mean, float* theta,
                          float lr, bool validate, PeerStats* stats, uint32_t* flags,
                          cudaStream_t stream) {
    const int64_t C = (n + Geo::kChunk - 1) / Geo::kChunk;
    if (C == 0) return cudaSuccess;
    // the lean shape where it applies: a mean of at most 16 peers with no outer step and no
    // statistics, for the chunk lengths and k it is built for
    constexpr bool kLeanOk = !kStats && Geo::kChunk == 4096 && Geo::kTopK <= 64;
    const bool pow2 = (P & (P - 1)) == 0;
    if constexpr (kLeanOk) {
        if (theta == nullptr && P <= kLeanMaxPeers)
            return pow2 ? launch_kernel<Geo, true, kStats, true>(tab, P, n, C, mean, theta, lr,
                                                                 validate, stats, flags, stream)
                        : launch_kernel<Geo, true, kStats, false>(tab, P, n, C, mean, theta, lr,
                                                                  validate, stats, flags, stream);
    }
    return pow2 ? launch_kernel<Geo, false, kStats, true>(tab, P, n, C, mean, theta, lr, validate,
                                                          stats, flags, stream)
                : launch_kernel<Geo, false, kStats, false>(tab, P, n, C, mean, theta, lr, validate,
                                                           stats, flags, stream);
}

// Launch for one record geometry, with or without statistics (which need validation on).
template <class Geo>
cudaError_t launch_geometry(const DecodeTable& tab, int P, int64_t n, float* mean, float* theta,
                            float lr, bool validate, PeerStats* stats, uint32_t* flags,
                            cudaStream_t stream) {
    return stats != nullptr
               ? launch_decode<Geo, true>(tab, P, n, mean, theta, lr, true, stats, flags, stream)
               : launch_decode<Geo, false>(tab, P, n, mean, theta, lr, validate, stats, flags,
                                           stream);
}

}  // namespace
}  // namespace spl
