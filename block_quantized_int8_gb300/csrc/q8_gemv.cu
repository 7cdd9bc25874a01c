// q8_gemv.cu -- Q8_0 W8A16 matrix-vector product (M = 1) over one or several
// matrices in one persistent launch.
//
// y[n] = sum_k s[n][k/32] * q[n][k] * x[k].  "Frigg" README, "The machine"
// (at batch 1 every decode matmul is this GEMV shape and it is bound by
// memory bandwidth) and Finding 3 (a decode step of many small matrices is
// launch-bound first: hence one launch for the whole list).
//
// Design (warp-specialised, bulk-copy fed):
//  * A "stage" is RT consecutive weight rows with their full K.  Rows of the
//    row-major codes q[N][K] and scales s[N][K/32] are contiguous, so a stage
//    is ONE bulk async copy of RT*K code bytes plus one of RT*K/16 scale bytes.
//  * Each CTA owns a contiguous range of the stages of all matrices, cut so
//    every CTA gets the same work (bytes, weighted up for split rows).
//  * Lane 0 of warp 0 also produces: it keeps kStages copies in flight
//    (cp.async.bulk -> shared memory, completion on a "full" mbarrier) and
//    refills a slot once every warp has released it ("empty" mbarrier).  A
//    CTA is 8 warps, so two CTAs fit on an SM without capping registers
//    (a ninth warp would put five warps on one SM sub-partition).
//  * All 8 warps consume; each copies its share of a stage into registers and
//    releases the slot before doing any arithmetic.  A row is split into
//    P = pow2(ceil(K/1536)) K-slices and a stage holds the most rows that fit
//    48 KB in groups of 16/P, so a stage is a whole number (>= 2) of row pairs
//    for every warp: the units (row, slice) warp + 8j, j = 0, 1, ...  Each warp always owns the same slice (w % P), so its part of x
//    stays in registers as fp32 (at most 48 values per lane), reloaded only
//    when the matrix changes.  Lanes read 16-byte chunks of the row from
//    shared memory (consecutive lanes, consecutive chunks: no bank
//    conflicts), turn codes into floats exactly (2^23 + byte trick) and use
//    packed fma.rn.f32x2 for the dot product; each half block's sum is scaled
//    by its binary16 scale in fp32; a warp shuffle tree sums the lanes.
//  * With P > 1 the slices of a row are added in slice order by whichever warp
//    finishes the row last (shared-memory counter; nobody waits), so results
//    are deterministic and independent of how matrices are batched.
// Every wait is bounded (Q8_DEV_TIMEOUT on expiry); no barrier spans warps
// that might have given up.
#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kStages = 2;
constexpr int kSliceK = 1536;                  // widest K slice of one warp
constexpr int kCodeBytes = 32 * kSliceK;       // RT * K <= 48 KB per stage
constexpr int kRedRows = 32;                   // rows per stage when P > 1 (at most 24)
constexpr int kMaxPairs = 4;                   // row pairs per warp per stage: RT * P <= 64
constexpr int kScaleBytes = kCodeBytes / 16 + 16;  // RT * K / 16, plus up to 14 bytes of alignment offset
constexpr int kStageBytes = kCodeBytes + kScaleBytes;
constexpr int kMaxK = 8 * kSliceK;             // P <= 8
constexpr int kMaxGrid = 512;
// Work of a stage for the partition, relative to its bytes: a matrix whose
// rows are split over warps (P > 1) costs more per byte (narrower slices,
// cross-warp combine).  1.2 measured best on the decode layer set
// (K = 1536 and K = 4096 matrices in one launch: +3 % over byte balance).
constexpr double kSplitCost = 1.2;
constexpr int kJMax = 3;                       // 16-code chunks per lane per slice (1536 k)
// Share of a CTA's balanced stage range that it owns outright; the rest of
// every range goes to a pool that CTAs draw from one stage at a time once
// their own part is done (CTAs start up to a few microseconds apart and SMs
// stream at different rates, so equal static shares finish unevenly).
constexpr double kStaticShare = 0.95;

struct GDesc {
    const int8_t *q;
    const uint16_t *s;
    const uint16_t *x;
    float *y;
    int32_t N;
    int32_t K;
    int32_t nb;          // K / 32
    int32_t P;           // slices per row (power of two <= 8)
    int32_t lp;          // log2(P)
    int32_t RT;          // rows per stage: a multiple of 16 / P, RT * K <= 48 KB
    int32_t bps;         // blocks per slice
    int32_t stage_begin; // first global stage index of this matrix
    int32_t stages;      // ceil(N / RT)
};

struct GParams {
    GDesc d[Q8_MAX_BATCH];
    uint32_t *status;
    uint32_t *sched;        // pool counter, zero between launches (null: no pool)
    int32_t count;
    int32_t total_stages;
    int32_t grid;
    int32_t pool_total;     // stages in the pool
    int32_t chained;        // launched as a programmatic dependent: weights may be read early
    int32_t early_signal;   // the grid fills every CTA slot: signal dependents at start
    int32_t cta_begin[kMaxGrid + 1];  // CTA c's balanced range [cta_begin[c], cta_begin[c+1])
    int32_t cta_split[kMaxGrid];      // it owns [cta_begin[c], cta_split[c]); the rest is pooled
    int32_t pool_off[kMaxGrid + 1];   // pool index of the first pooled stage of CTA c's range
    uint32_t zero;                    // 0 (a value the compiler cannot see: see warp_loaded_zero)
};

struct Smem {
    alignas(128) uint8_t stage[kStages][kStageBytes];
    float red[2 * kStages][kRedRows][8];   // per-stage slice sums (P > 1), ring of 2*kStages
    uint32_t cnt[2 * kStages][kRedRows];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t named[kStages];               // the producer has written sidx of the slot
    int32_t sidx[kStages];                 // stage in a slot drawn from the pool; -1: no more
};

__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    return (static_cast<unsigned long long>(__float_as_uint(b)) << 32) | __float_as_uint(a);
}
__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long add_f32x2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Four codes of word w times four activations (two packed pairs) added to acc.
// Codes become exact floats: 0x4B000000 | (c ^ 0x80) is 2^23 + 128 + c.
__device__ __forceinline__ unsigned long long dot4(uint32_t w, unsigned long long x01, unsigned long long x23,
                                                   unsigned long long acc) {
    const uint32_t u = w ^ 0x80808080u;
    const unsigned long long m01 = (static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7651)) << 32) |
                                   __byte_perm(u, 0x4B000000u, 0x7650);
    const unsigned long long m23 = (static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7653)) << 32) |
                                   __byte_perm(u, 0x4B000000u, 0x7652);
    const unsigned long long nb2 = 0xCB000080CB000080ull;  // (-(2^23 + 128), -(2^23 + 128))
    acc = fma_f32x2(add_f32x2(m01, nb2), x01, acc);
    acc = fma_f32x2(add_f32x2(m23, nb2), x23, acc);
    return acc;
}


// One lane's share of a stage for rows A and B: NJ chunks of 16 codes and
// their half-block scales, pulled from shared memory into registers so the
// slot can be handed back to the producer before any arithmetic.
template <int NJ>
struct RowPair {
    uint4 wA[NJ], wB[NJ];
    uint32_t h[NJ];  // binary16 scale bits: row A low half, row B high half
};

// FULL: both rows exist and every lane has NJ chunks (the common case), so
// the loads need no predicates and no zero fill.
template <int NJ, bool FULL>
__device__ __forceinline__ void load_rows(RowPair<NJ> &rp, const uint8_t *cA, const uint8_t *cB,
                                          const uint16_t *sA, const uint16_t *sB, bool vA, bool vB, int lane,
                                          int chunks_slice) {
    if constexpr (FULL) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int c = lane + 32 * j;
            rp.wA[j] = *reinterpret_cast<const uint4 *>(cA + 16 * c);
            rp.wB[j] = *reinterpret_cast<const uint4 *>(cB + 16 * c);
            rp.h[j] = static_cast<uint32_t>(sA[c >> 1]) | (static_cast<uint32_t>(sB[c >> 1]) << 16);
        }
    } else {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int c = lane + 32 * j;
            rp.wA[j] = make_uint4(0u, 0u, 0u, 0u);
            rp.wB[j] = rp.wA[j];
            rp.h[j] = 0u;
            if (c < chunks_slice && vA) {
                rp.wA[j] = *reinterpret_cast<const uint4 *>(cA + 16 * c);
                rp.h[j] = sA[c >> 1];
            }
            if (c < chunks_slice && vB) {
                rp.wB[j] = *reinterpret_cast<const uint4 *>(cB + 16 * c);
                rp.h[j] |= static_cast<uint32_t>(sB[c >> 1]) << 16;
            }
        }
    }
}

// Dot products of the lane's chunks with its x chunks, each half block's sum
// scaled by its binary16 scale.  NJ is a compile-time constant so both rows'
// chunks form one straight-line block the scheduler can interleave; two packed
// accumulators per chunk keep the fma.rn.f32x2 dependency chains short.
template <int NJ, int KJ>
__device__ __forceinline__ void dot_rows(const RowPair<NJ> &rp, const unsigned long long (&xr)[KJ][8],
                                         float &accA, float &accB) {
    static_assert(NJ <= KJ, "x chunk out of range");
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        unsigned long long a0 = dot4(rp.wA[j].x, xr[j][0], xr[j][1], 0ull);
        unsigned long long a1 = dot4(rp.wA[j].y, xr[j][2], xr[j][3], 0ull);
        unsigned long long b0 = dot4(rp.wB[j].x, xr[j][0], xr[j][1], 0ull);
        unsigned long long b1 = dot4(rp.wB[j].y, xr[j][2], xr[j][3], 0ull);
        a0 = dot4(rp.wA[j].z, xr[j][4], xr[j][5], a0);
        a1 = dot4(rp.wA[j].w, xr[j][6], xr[j][7], a1);
        b0 = dot4(rp.wB[j].z, xr[j][4], xr[j][5], b0);
        b1 = dot4(rp.wB[j].w, xr[j][6], xr[j][7], b1);
        const unsigned long long a = add_f32x2(a0, a1);
        const unsigned long long b = add_f32x2(b0, b1);
        accA = fmaf(f16_bits_to_f32(rp.h[j] & 0xFFFFu), __uint_as_float(static_cast<uint32_t>(a)) +
                                                           __uint_as_float(static_cast<uint32_t>(a >> 32)), accA);
        accB = fmaf(f16_bits_to_f32(rp.h[j] >> 16), __uint_as_float(static_cast<uint32_t>(b)) +
                                                       __uint_as_float(static_cast<uint32_t>(b >> 32)), accB);
    }
}

// Load a row pair of the stage into registers and compute; release the slot
// if this is the warp's last pair of the stage (empty_bar != nullptr).
template <int NJ, int KJ, bool FULL>
__device__ __forceinline__ void stage_rows(const uint8_t *cA, const uint8_t *cB, const uint16_t *sA,
                                           const uint16_t *sB, bool vA, bool vB, int lane, int chunks_slice,
                                           const unsigned long long (&xr)[KJ][8], uint64_t *empty_bar,
                                           uint32_t zero, float &accA, float &accB) {
    RowPair<NJ> rp;
    load_rows<NJ, FULL>(rp, cA, cB, sA, sB, vA, vB, lane, chunks_slice);
    dot_rows<NJ, KJ>(rp, xr, accA, accB);
    if (empty_bar) {
        // the slot goes back to the bulk-copy producer once every lane's
        // loads above have returned, not when they were issued: the release
        // depends on the two sums, which every loaded word feeds (see
        // warp_loaded_zero)
        const uint32_t dep = warp_loaded_zero(__float_as_uint(accA) | __float_as_uint(accB), zero);
        if (lane == 0) {
            asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(empty_bar) + dep)
                         : "memory");
        }
    }
}

// This warp's share of one stage.  Its (row, slice) units are warp + 8j, all
// of slice `slice`, taken as row pairs (warp + 16t, warp + 16t + 8): rows
// (warp >> lp) + t * (16 >> lp) and that plus (8 >> lp), t < nsteps <= kMaxPairs.
// Only a ragged last stage (U < RT * P valid units) leaves a pair with one
// row.  The slot is released once the warp's last pair of the stage is summed.  The
// lanes' partial sums of all (up to 8) rows are reduced together at the end:
// a transposed butterfly halves the values a lane carries at each of the
// first three exchanges, so lane l ends with row value (l >> 2) & 7 and the
// stage costs 9 shuffles and one dependent chain, not one per pair.
template <int NJ, int KJ>
__device__ __forceinline__ void stage_pairs(Smem &sm, int slot, int rs, const uint8_t *cA, const uint16_t *sA,
                                            int K, int nb, int lp, int U, int nsteps, int warp, int lane, int slice,
                                            bool full_slice, int chunks_slice, float *yrow, int wrow,
                                            const unsigned long long (&xr)[KJ][8], uint32_t zero) {
    const int pstride = 16 >> lp;  // rows from one pair of the warp to the next
    const int boff = 8 >> lp;      // row B - row A
    float acc[2 * kMaxPairs];
#pragma unroll
    for (int t = 0; t < kMaxPairs; ++t) {
        acc[2 * t] = 0.f;
        acc[2 * t + 1] = 0.f;
        if (t < nsteps) {
            const bool vB = warp + 16 * t + 8 < U;
            const uint8_t *ca = cA + t * pstride * K;
            const uint16_t *sa = sA + t * pstride * nb;
            uint64_t *rel = (t == nsteps - 1) ? &sm.empty[slot] : nullptr;
            if (vB && full_slice)
                stage_rows<NJ, KJ, true>(ca, ca + boff * K, sa, sa + boff * nb, true, vB, lane, chunks_slice, xr,
                                         rel, zero, acc[2 * t], acc[2 * t + 1]);
            else
                stage_rows<NJ, KJ, false>(ca, ca + boff * K, sa, sa + boff * nb, true, vB, lane, chunks_slice, xr,
                                          rel, zero, acc[2 * t], acc[2 * t + 1]);
        }
    }
    // transposed butterfly: keep the half of the values selected by the lane
    // bit, add the partner's copy of that half
    float h4[4], h2[2];
    const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const float keep = b4 ? acc[v + 4] : acc[v];
        const float give = b4 ? acc[v] : acc[v + 4];
        h4[v] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
    }
#pragma unroll
    for (int v = 0; v < 2; ++v) {
        const float keep = b3 ? h4[v + 2] : h4[v];
        const float give = b3 ? h4[v] : h4[v + 2];
        h2[v] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
    }
    float r;
    {
        const float keep = b2 ? h2[1] : h2[0];
        const float give = b2 ? h2[0] : h2[1];
        r = keep + __shfl_xor_sync(0xffffffffu, give, 4);
    }
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    // lane 4v holds value v: pair v >> 1, row A (v even) or B (v odd)
    const int v = lane >> 2;
    const int t = v >> 1;
    const bool isB = (v & 1) != 0;
    if ((lane & 3) == 0 && t < nsteps && (!isB || warp + 16 * t + 8 < U)) {
        const int row = wrow + t * pstride + (isB ? boff : 0);
        if (lp == 0) {
            yrow[row] = r;
        } else {
            const int P = 1 << lp;
            sm.red[rs][row][slice] = r;
            __threadfence_block();
            const uint32_t prev = atomicAdd(&sm.cnt[rs][row], 1u);
            if (prev == static_cast<uint32_t>(P - 1)) {
                __threadfence_block();
                float tot = sm.red[rs][row][0];
                for (int sl = 1; sl < P; ++sl) tot += sm.red[rs][row][sl];
                yrow[row] = tot;
                sm.cnt[rs][row] = 0u;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Descriptor of a stage (binary search: pool stages come from anywhere).
__device__ __forceinline__ int find_gdesc(const GParams &p, int stage) {
    int lo = 0, hi = p.count;  // d[lo].stage_begin <= stage < d[hi].stage_begin
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.d[mid].stage_begin <= stage) lo = mid; else hi = mid;
    }
    return lo;
}

// Stage of pool index j: the pooled part of CTA c's range holds pool indices
// [pool_off[c], pool_off[c+1]).
__device__ __forceinline__ int pool_stage(const GParams &p, int j) {
    int lo = 0, hi = p.grid;  // pool_off[lo] <= j < pool_off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.pool_off[mid] <= j) lo = mid; else hi = mid;
    }
    return p.cta_split[lo] + (j - p.pool_off[lo]);
}

// The work of one CTA: its own stages [begin, split), then stages drawn from
// the pool until it is empty; KJ is the number of 16-code chunks per lane in
// a warp's K slice (3: slices up to 1536 wide).  Ring position k uses slot
// k % kStages and mbarrier phase (k / kStages) & 1.
template <int KJ>
__device__ __forceinline__ void cta_work(const GParams &p, Smem &sm, int begin, int split, int warp, int lane) {
    // Lane 0 of warp 0 is also the producer.  Before warp 0 consumes position
    // k it tops the ring up: positions up to k + kStages - 1 are issued as soon
    // as their slot is free (non-blocking check); position k itself is issued
    // even if that means waiting for the slowest warp to release its slot, so
    // no consumer can wait on a copy that nobody will start.  Positions past
    // the CTA's own stages take pool indices from the counter, drawn one
    // position ahead so that the atomic's latency hides behind a stage; the
    // stage goes to sidx[slot] (announced on named[slot] at once, so that the
    // consumers can load x for it while the copy is in flight), and once the
    // pool is empty an end marker (-1) takes its place.  Every CTA draws exactly
    // one index past the pool, so the CTA that draws the grid's last one
    // leaves the counter zero for the next launch.
    const int nown = split - begin;
    int pi = 0;                         // positions issued so far (producer lane only)
    int pd = nown > 0 ? find_gdesc(p, begin) : 0;  // descriptor of the stage being issued
    bool prod_ok = true;                // false once timed out or past the end marker
    uint32_t ahead = 0xFFFFFFFFu;       // pool index drawn for the next pool position
    auto draw = [&]() { ahead = p.sched ? atomicAdd(p.sched, 1u) : 0xFFFFFFFFu; };
    auto produce = [&](int upto) {
        while (prod_ok && pi <= upto) {
            const int slot = pi % kStages;
            if (pi >= kStages) {
                const uint32_t par = ((pi / kStages) - 1) & 1;
                const bool must = pi <= upto - (kStages - 1);
                if (must) {
                    if (!mbar_wait_bounded(&sm.empty[slot], par)) {
                        prod_ok = false;
                        if (p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
                        return;
                    }
                } else if (!mbar_test_wait(&sm.empty[slot], par)) {
                    return;
                }
            }
            int i;
            if (pi < nown) {
                i = begin + pi;
                while (i >= p.d[pd].stage_begin + p.d[pd].stages) ++pd;
            } else {
                const uint32_t j = ahead;
                if (j >= static_cast<uint32_t>(p.pool_total)) {
                    if (p.sched && j == static_cast<uint32_t>(p.pool_total + p.grid - 1)) atomicExch(p.sched, 0u);
                    sm.sidx[slot] = -1;
                    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];"
                                 :: "r"(smem_addr(&sm.named[slot])) : "memory");
                    prod_ok = false;
                    // nothing left to issue: a chained launch after this one
                    // may start once every CTA is this far
                    if (!p.early_signal) pdl_launch_dependents();
                    return;
                }
                i = pool_stage(p, static_cast<int>(j));
                pd = find_gdesc(p, i);
                sm.sidx[slot] = i;
                asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];"
                             :: "r"(smem_addr(&sm.named[slot])) : "memory");
            }
            const GDesc &D = p.d[pd];
            const int r0 = (i - D.stage_begin) * D.RT;
            const int rows = min(D.RT, D.N - r0);
            const uint32_t cbytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.K);
            // scales: bulk copies need 16-byte aligned source AND destination, so
            // the stage keeps them at the same address offset mod 16 as in global
            // memory; the unaligned head and tail (< 16 bytes each) go by plain
            // copies, published by the arrive below
            const uint32_t sbytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.nb) * 2u;
            const int64_t sstart = static_cast<int64_t>(r0) * D.nb * 2;
            const uint32_t a = static_cast<uint32_t>(sstart & 15);
            const uint8_t *gs = reinterpret_cast<const uint8_t *>(D.s) + sstart;
            uint8_t *dst = sm.stage[slot];
            uint8_t *sdst = dst + kCodeBytes + a;
            const uint32_t head = min(sbytes, a ? 16u - a : 0u);
            const uint32_t body = (sbytes - head) & ~15u;
            for (uint32_t b = 0; b < head; b += 2)
                *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
            for (uint32_t b = head + body; b < sbytes; b += 2)
                *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
            mbar_arrive_expect_tx(&sm.full[slot], cbytes + body);
            bulk_g2s(dst, D.q + static_cast<int64_t>(r0) * D.K, cbytes, &sm.full[slot]);
            if (body) bulk_g2s(sdst + head, gs + head, body, &sm.full[slot]);
            if (pi >= nown - 1) draw();
            ++pi;
        }
    };

    // ---------------------------------------------------------------- consumers
    int d = nown > 0 ? find_gdesc(p, begin) : 0;
    unsigned long long xr[KJ][8];  // this lane's x chunks as packed fp32 pairs
    int slice = 0, nj = 0, k0 = 0, chunks_slice = 0;
    // x in the registers: activation row and geometry (K, P) it was loaded for
    const uint16_t *cur_x = nullptr;
    int cur_K = 0, cur_P = 0;
    // (re)load this warp's slice of x into registers as fp32 pairs, unless
    // they already hold it (matrices of one launch often share their x)
    auto load_x = [&](const GDesc &D) {
        if (D.x == cur_x && D.K == cur_K && D.P == cur_P) return;
        cur_x = D.x;
        cur_K = D.K;
        cur_P = D.P;
        slice = warp & (D.P - 1);
        const int kb0 = slice * D.bps;
        const int kb1 = min(D.nb, kb0 + D.bps);
        chunks_slice = (kb1 - kb0) * 2;  // 16-code chunks in the slice
        k0 = kb0 * 32;
        nj = (chunks_slice + 31) / 32;
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
            const int c = lane + 32 * j;
            uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
            if (c < chunks_slice) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(D.x + k0 + 16 * c);
                a = __ldg(xp);
                b = __ldg(xp + 1);
            }
            const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) xr[j][e] = f2_pack(bf16lo_f32(v[e]), bf16hi_f32(v[e]));
        }
    };
    // Chained launch: the first own stages that need no draw (weights only) are
    // issued before the previous kernel in the stream has completed; x, y and
    // the counter are touched only after the wait below.
    if (p.chained && warp == 0 && lane == 0) produce(min(kStages, nown - 1) - 1);
    pdl_wait_prior();
    if (warp == 0 && lane == 0 && nown == 0) draw();
    for (int k = 0;; ++k) {
        if (warp == 0 && lane == 0) produce(k + kStages - 1);
        __syncwarp();
        const int slot = k % kStages;
        int i;
        if (k < nown) {
            // own stage: x for it loads while its copy is in flight
            i = begin + k;
            while (i >= p.d[d].stage_begin + p.d[d].stages) ++d;
            load_x(p.d[d]);
            if (!mbar_wait_bounded(&sm.full[slot], (k / kStages) & 1)) {
                if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
                drain_after_timeout();
                return;
            }
        } else {
            // pool stage: its index is published (named) when it is issued,
            // so x for it loads while its copy is in flight
            const int kp = k - nown;  // pool positions before this one
            if (!mbar_wait_bounded(&sm.named[slot], (kp / kStages) & 1)) {
                if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
                drain_after_timeout();
                return;
            }
            i = *reinterpret_cast<volatile const int32_t *>(&sm.sidx[slot]);
            if (i < 0) return;
            d = find_gdesc(p, i);
            load_x(p.d[d]);
            if (!mbar_wait_bounded(&sm.full[slot], (k / kStages) & 1)) {
                if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
                drain_after_timeout();
                return;
            }
        }
        const GDesc &D = p.d[d];
        const uint8_t *codes = sm.stage[slot];
        const int r0 = (i - D.stage_begin) * D.RT;
        const uint16_t *scales = reinterpret_cast<const uint16_t *>(
            sm.stage[slot] + kCodeBytes + ((static_cast<int64_t>(r0) * D.nb * 2) & 15));
        const int rows = min(D.RT, D.N - r0);
        const int U = rows << D.lp;                       // valid (row, slice) units
        const int nsteps = (max(0, (U - warp + 7) >> 3) + 1) >> 1;  // this warp's row pairs
        if (nsteps == 0) {
            __syncwarp();
            if (lane == 0) {
                asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(&sm.empty[slot])) : "memory");
            }
            continue;
        }
        const int wrow = warp >> D.lp;
        const uint8_t *cA = codes + wrow * D.K + k0;
        const uint16_t *sA = scales + wrow * D.nb + (k0 >> 5);
        const int rs = k % (2 * kStages);
        const bool full_slice = chunks_slice == 32 * nj;
        float *yrow = D.y + r0;
        switch (nj) {
            case 1: stage_pairs<1, KJ>(sm, slot, rs, cA, sA, D.K, D.nb, D.lp, U, nsteps, warp, lane, slice, full_slice, chunks_slice, yrow, wrow, xr, p.zero); break;
            case 2: stage_pairs<2, KJ>(sm, slot, rs, cA, sA, D.K, D.nb, D.lp, U, nsteps, warp, lane, slice, full_slice, chunks_slice, yrow, wrow, xr, p.zero); break;
            default: stage_pairs<3, KJ>(sm, slot, rs, cA, sA, D.K, D.nb, D.lp, U, nsteps, warp, lane, slice, full_slice, chunks_slice, yrow, wrow, xr, p.zero); break;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const __grid_constant__ GParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int begin = p.cta_begin[blockIdx.x];
    const int split = p.cta_split[blockIdx.x];

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kConsumerWarps);
            mbar_init(&sm.named[i], 1);
        }
        fence_mbar_init();
    }
    for (int i = tid; i < 2 * kStages * kRedRows; i += kThreads) (&sm.cnt[0][0])[i] = 0u;
    __syncthreads();
    // A grid that fills every CTA slot lets a chained launch after it start
    // at once: its CTAs can only take the slots ours free as they exit.  A
    // smaller grid signals late (else chained calls would start one after
    // another and crowd the GPU with waiting CTAs).
    if (p.early_signal && tid == 0) pdl_launch_dependents();
    cta_work<kJMax>(p, sm, begin, split, warp, lane);
}

int g_configured_dev = -1;
int g_occ = 0;

}  // namespace

bool gemv_k_supported(int64_t K) { return K <= kMaxK; }

q8_status launch_gemv(const q8_linear_desc *descs, int count, uint32_t *sched, uint32_t *dev_status,
                      cudaStream_t stream, bool chained) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (g_configured_dev != di->device) {
        if (cudaFuncSetAttribute(gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(Smem))) != cudaSuccess)
            return Q8_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, gemv_kernel, kThreads, sizeof(Smem)) != cudaSuccess)
            return Q8_ERR_CUDA;
        g_occ = std::max(o, 1);
        g_configured_dev = di->device;
    }
    static thread_local GParams p;  // large: keep it off the stack
    double total_bytes = 0.0;
    int stages = 0;
    for (int i = 0; i < count; ++i) {
        GDesc &D = p.d[i];
        const int K = static_cast<int>(descs[i].K);
        int P = 1;
        while (P * kSliceK < K) P *= 2;
        D.q = descs[i].q;
        D.s = descs[i].s;
        D.x = descs[i].x;
        D.y = descs[i].y;
        D.N = static_cast<int32_t>(descs[i].N);
        D.K = K;
        D.nb = K / 32;
        D.P = P;
        D.lp = __builtin_ctz(static_cast<unsigned>(P));
        // the most rows that fit kCodeBytes in whole groups of 16 / P rows, so
        // every stage is whole row pairs for all 8 warps (RT * P = 16 * pairs);
        // K <= P * kSliceK guarantees at least two pairs; at most kMaxPairs
        D.RT = std::min((kCodeBytes / K) / (16 / P) * (16 / P), 16 * kMaxPairs / P);
        D.bps = (D.nb + P - 1) / P;
        D.stage_begin = stages;
        D.stages = (D.N + D.RT - 1) / D.RT;
        stages += D.stages;
        total_bytes += static_cast<double>(D.N) * K * 1.0625 * (D.P > 1 ? kSplitCost : 1.0);
    }
    p.status = dev_status;
    p.zero = 0u;
    p.count = count;
    p.total_stages = stages;
    if (stages == 0) return Q8_OK;
    const int grid = std::min(std::min(stages, di->sm_count * g_occ), kMaxGrid);
    // cut the stage list into `grid` ranges of (nearly) equal work
    int c = 0;
    double acc = 0.0;
    p.cta_begin[0] = 0;
    for (int i = 0; i < count && c < grid - 1; ++i) {
        const GDesc &D = p.d[i];
        const double full = static_cast<double>(D.RT) * D.K * 1.0625 * (D.P > 1 ? kSplitCost : 1.0);
        for (int st = 0; st < D.stages && c < grid - 1; ++st) {
            const int rows = std::min(D.RT, D.N - st * D.RT);
            acc += full * rows / D.RT;
            while (c < grid - 1 && acc >= total_bytes * (c + 1) / grid) p.cta_begin[++c] = D.stage_begin + st + 1;
        }
    }
    while (c < grid) p.cta_begin[++c] = stages;
    // each CTA keeps the first kStaticShare of its range; the rest is pooled
    p.sched = sched;
    p.grid = grid;
    p.pool_off[0] = 0;
    for (int b = 0; b < grid; ++b) {
        const int len = p.cta_begin[b + 1] - p.cta_begin[b];
        const int own = sched ? static_cast<int>(len * kStaticShare) : len;
        p.cta_split[b] = p.cta_begin[b] + own;
        p.pool_off[b + 1] = p.pool_off[b] + (len - own);
    }
    p.pool_total = p.pool_off[grid];
    p.chained = chained ? 1 : 0;
    p.early_signal = grid >= di->sm_count * g_occ ? 1 : 0;
    if (launch_kernel(gemv_kernel, dim3(grid), dim3(kThreads), sizeof(Smem), stream, chained, p) != cudaSuccess)
        return Q8_ERR_CUDA;
    return Q8_OK;
}

}  // namespace q8
