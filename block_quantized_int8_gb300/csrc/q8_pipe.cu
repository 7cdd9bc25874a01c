// q8_pipe.cu -- Q8_0 W8A16 matmul for 1 <= M <= 8 activation rows over one or
// several matrices in one persistent launch (K <= 4096).
//
// Y[m][n] = sum_k s[n][k/32] * q[n][k] * x[m][k]; "Frigg" README, Finding 8
// (a batched W8A16 kernel reads each weight once for the whole batch of rows)
// and Finding 3 (one launch for the many small matrices of a decode step).
//
// Design (bulk-copy fed, tensor cores through warp mma):
//  * A stage is RT consecutive weight rows with their full K, about 48 KB.
//    Each row goes by one cp.async.bulk into a
//    shared-memory row padded to K + 32 bytes (the padding puts the rows that
//    one mma reads at the same k on distinct banks), and the RT*K/16 scale
//    bytes with one more copy.  The ring has S = 2 or 3 slots (as many as the
//    launch's largest stage allows with two CTAs per SM).  There is no
//    producer warp: thread 0 issues the first S stages and then the warp that
//    releases a slot last (a shared-memory counter) issues the stage S later
//    into it, so a slot is refilled the moment it is free.  CTAs own
//    byte-balanced contiguous stage ranges (as in q8_gemv.cu).
//  * Rows come in groups of 8 and K in P slices (P a power of two <= 8).  A
//    full-tile stage has 16/P groups and slices of at most 384: each warp
//    owns one slice (w % P) of two groups, one whole m16n8k16 tile.  A
//    half-tile stage has 8/P groups and slices of at most 512: each warp owns
//    one slice of one group, half a tile (the upper rows of the mma operand
//    are zero and never converted).  Full tiles are used whenever their
//    slices fit (K <= 3072: e.g. K = 1536, 32 rows, two slots); otherwise
//    half tiles (K = 4096: 8 rows, three slots).  A warp's x slice stays in registers in
//    the mma B-fragment layout (at most 16 blocks), reloaded only when the
//    matrix changes.
//  * Per 32-code block two mma.sync.m16n8k16 (binary16 in, fp32 out) with
//    the weights as the 16-row A operand (lane (g, t) holds bytes [8t, 8t+8)
//    of its rows) and x^T as B (columns = activation rows, zero past M).
//    Codes become binary16 exactly (|q| <= 127) in three operations per pair;
//    x is converted once per matrix: bf16 has 8 significant bits, so a value
//    that is zero or of magnitude in [2^-17, 65504] is exact in binary16.  A
//    block holding any other x value (tiny, huge, inf, nan) takes an exact
//    bf16 path instead (codes -> bf16 by a sign split, x from global memory).
//    Each block's fp32 result is scaled by its binary16 scale.  The warps
//    compute straight from shared memory.
//  * The P partial tiles of a stage are added in slice order by whichever of
//    the P warps finishes last (shared-memory counter, nobody waits), so the
//    results are deterministic and independent of batching.  A warp releases
//    its slot after its partial is published (the last one after reading all
//    partials), which also protects the partial buffers, one per slot.
// Every wait is bounded (Q8_DEV_TIMEOUT on expiry).
#include <algorithm>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPad = 32;               // bytes after each shared-memory row
constexpr int kSliceK = 384;           // widest slice of a full-tile stage
constexpr int kHalfSliceK = 512;       // widest slice of a half-tile stage
constexpr int kPipeMaxK = 4096;
constexpr int kMaxSlots = 3;
constexpr int kMaxGrid = 1024;
// Work of a stage for the partition, relative to its bytes: half-tile
// stages cost more per byte (measured 3.7 vs 4.9 TB/s on K = 4096 and
// K = 1536 batches).
constexpr double kHalfCost = 1.3;
constexpr int kSmemBudget = 115712;    // dynamic shared memory per CTA, two CTAs per SM
constexpr int kCtlBytes = 256;         // counters and mbarriers

struct PDesc {
    const int8_t *q;
    const uint16_t *s;
    const uint16_t *x;
    float *y;
    int64_t ldx;
    int64_t ldy;
    int32_t N;
    int32_t K;
    int32_t nb;
    int32_t RT;          // rows per stage (a multiple of 8)
    int32_t RS;          // shared-memory row stride, K + kPad
    int32_t P;           // K slices (power of two <= 8)
    int32_t lp;          // log2(P)
    int32_t half;        // 1: one 8-row group per stage, half tiles
    int32_t bps;         // blocks per slice
    int32_t scale_off;   // offset of the scales in a slot: RT * RS
    int32_t stage_begin;
    int32_t stages;
};

struct PParams {
    PDesc d[Q8_MAX_BATCH];
    uint32_t *status;
    int32_t count;
    int32_t M;
    int32_t S;           // slots in the ring
    int32_t slot_bytes;
    int32_t red_off;     // partial tiles: S entries of red_entry bytes
    int32_t red_entry;   // 8 warps x 32 lanes x (float4 full tiles, float2 half tiles)
    int32_t ctl_off;     // counters [kMaxSlots][8], release counts [kMaxSlots], then full[kMaxSlots]
    int32_t early_signal;  // the grid fills every CTA slot: signal dependents at start
    int32_t cta_begin[kMaxGrid + 1];
};

__device__ __forceinline__ int find_pdesc(const PParams &p, int stage) {
    int d = 0;
    while (d + 1 < p.count && stage >= p.d[d + 1].stage_begin) ++d;
    return d;
}

// One warp's share of a stage: BPW blocks of its slice for row ra (lower half
// of the mma tile) and, if TWO, row rb (upper half), straight from shared
// memory.  FULL: both rows exist and the slice has BPW blocks, so nothing is
// predicated.  acc[0..1]: row ra, activation rows 2t, 2t+1; acc[2..3]: rb.
// x is binary16 (xr); blocks that binary16 cannot hold are zero there and
// done by slow_blocks.
template <int BPW, bool TWO, bool FULL, int KJ>
__device__ __forceinline__ void tile_mma(const uint8_t *ca, const uint8_t *cb, const uint16_t *sa,
                                         const uint16_t *sb, bool va, bool vb, int nblk, int t,
                                         const uint4 (&xr)[KJ], float (&acc)[4]) {
    static_assert(BPW <= KJ, "x fragment out of range");
#pragma unroll
    for (int j = 0; j < BPW; ++j) {
        if (!FULL && j >= nblk) break;
        uint2 wa = make_uint2(0u, 0u), wb = wa;
        uint32_t ha = 0u, hb = 0u;
        if (FULL || va) {
            wa = *reinterpret_cast<const uint2 *>(ca + 32 * j + 8 * t);
            ha = sa[j];
        }
        if constexpr (TWO) {
            if (FULL || vb) {
                wb = *reinterpret_cast<const uint2 *>(cb + 32 * j + 8 * t);
                hb = sb[j];
            }
        }
        uint32_t a01, a23, a45, a67, b01 = 0u, b23 = 0u, b45 = 0u, b67 = 0u;
        codes4_to_f16x2(wa.x, a01, a23);
        codes4_to_f16x2(wa.y, a45, a67);
        if constexpr (TWO) {
            codes4_to_f16x2(wb.x, b01, b23);
            codes4_to_f16x2(wb.y, b45, b67);
        }
        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
        mma_f16_16816(d0, d1, d2, d3, a01, b01, a23, b23, xr[j].x, xr[j].y);
        mma_f16_16816(d0, d1, d2, d3, a45, b45, a67, b67, xr[j].z, xr[j].w);
        const float s_a = f16_bits_to_f32(ha);
        acc[0] = fmaf(s_a, d0, acc[0]);
        acc[1] = fmaf(s_a, d1, acc[1]);
        if constexpr (TWO) {
            const float s_b = f16_bits_to_f32(hb);
            acc[2] = fmaf(s_b, d2, acc[2]);
            acc[3] = fmaf(s_b, d3, acc[3]);
        }
    }
}

// The blocks of a warp's slice whose x binary16 cannot hold (bits of
// `slow`): exact bf16 products with x from global memory (xg, null past M).
// Rare for activations, so kept out of line.
__device__ __noinline__ float4 slow_blocks(const uint8_t *ca, const uint8_t *cb, const uint16_t *sa,
                                           const uint16_t *sb, bool va, bool vb, int t, uint32_t slow,
                                           const uint16_t *xg, float4 acc) {
    while (slow) {
        const int j = __ffs(slow) - 1;
        slow &= slow - 1u;
        uint2 wa = make_uint2(0u, 0u), wb = wa;
        uint32_t ha = 0u, hb = 0u;
        if (va) {
            wa = *reinterpret_cast<const uint2 *>(ca + 32 * j + 8 * t);
            ha = sa[j];
        }
        if (vb) {
            wb = *reinterpret_cast<const uint2 *>(cb + 32 * j + 8 * t);
            hb = sb[j];
        }
        uint4 xb = make_uint4(0u, 0u, 0u, 0u);
        if (xg) xb = __ldg(reinterpret_cast<const uint4 *>(xg + 32 * j));
        uint32_t a01, a23, a45, a67, b01, b23, b45, b67;
        codes4_to_bf16x2(wa.x, a01, a23);
        codes4_to_bf16x2(wa.y, a45, a67);
        codes4_to_bf16x2(wb.x, b01, b23);
        codes4_to_bf16x2(wb.y, b45, b67);
        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
        mma_bf16_16816(d0, d1, d2, d3, a01, b01, a23, b23, xb.x, xb.y);
        mma_bf16_16816(d0, d1, d2, d3, a45, b45, a67, b67, xb.z, xb.w);
        const float s_a = f16_bits_to_f32(ha), s_b = f16_bits_to_f32(hb);
        acc.x = fmaf(s_a, d0, acc.x);
        acc.y = fmaf(s_a, d1, acc.y);
        acc.z = fmaf(s_b, d2, acc.z);
        acc.w = fmaf(s_b, d3, acc.w);
    }
    return acc;
}

// x slice of activation row g (xg, null past M) as binary16 for the mma B
// operand.  bf16 has 8 significant bits, so binary16 holds a bf16 value
// exactly when it is zero or its magnitude lies in [2^-17, 65504] (below
// 2^-14 as a subnormal that is still a multiple of 2^-24).  A block with any
// other value (tiny, huge, inf, nan) is left zero and flagged in `slow` for
// the exact bf16 path.
template <int KJ>
__device__ __forceinline__ void prep_x(const uint16_t *xg, int nblk, uint4 (&xr)[KJ], uint32_t &slow) {
    slow = 0u;
    // all loads first (independent, so they overlap), then the conversions
#pragma unroll
    for (int j = 0; j < KJ; ++j)
        xr[j] = (xg && j < nblk) ? __ldg(reinterpret_cast<const uint4 *>(xg + 32 * j)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < KJ; ++j) {
        uint32_t h[4] = {0u, 0u, 0u, 0u};
        bool inexact = false;
        {
            const uint4 v = xr[j];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                h[q] = f32x2_to_f16x2(bf16lo_f32(w4[q]), bf16hi_f32(w4[q]));
                inexact |= !bf16_fits_f16(w4[q] & 0xFFFFu) || !bf16_fits_f16(w4[q] >> 16);
            }
        }
        xr[j] = make_uint4(h[0], h[1], h[2], h[3]);
        if (__any_sync(0xffffffffu, inexact)) {
            slow |= 1u << j;
            xr[j] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// KJ: x blocks a warp keeps in registers (12: full tiles only; 16: any).
template <int KJ>
__global__ void __launch_bounds__(kThreads, 2) pipe_kernel(const __grid_constant__ PParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int begin = p.cta_begin[blockIdx.x];
    const int end = p.cta_begin[blockIdx.x + 1];
    const int M = p.M;
    const int S = p.S;
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem_raw + p.ctl_off);     // [S][8 tiles]
    uint32_t *rel = cnt + kMaxSlots * 8;                                     // [S] release counts
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw + p.ctl_off + kMaxSlots * 9 * 4 + 4);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
        for (int i = 0; i < kMaxSlots * 9; ++i) cnt[i] = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    // a grid that fills every CTA slot signals a chained launch after it at
    // once (its CTAs can only take the slots ours free); a smaller one late
    if (p.early_signal && tid == 0) pdl_launch_dependents();
    if (end <= begin) return;

    // ---- refills ------------------------------------------------------------------
    // Thread 0 issues the first S stages; afterwards the warp that releases a
    // slot last issues the stage S later into it at once, so a free slot never
    // waits for a particular warp to come round.
    const int nstages = end - begin;
    auto issue = [&](int pi, int pd) {
        const int slot = pi % S;
        const int i = begin + pi;
        while (i >= p.d[pd].stage_begin + p.d[pd].stages) ++pd;
        const PDesc &D = p.d[pd];
        const int r0 = (i - D.stage_begin) * D.RT;
        const int rows = min(D.RT, D.N - r0);
        uint8_t *dst = smem_raw + static_cast<size_t>(slot) * p.slot_bytes;
        // scales: same offset mod 16 as in global memory; the unaligned head
        // and tail go by plain copies, published by the arrive below
        const uint32_t sbytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.nb) * 2u;
        const int64_t sstart = static_cast<int64_t>(r0) * D.nb * 2;
        const uint32_t a = static_cast<uint32_t>(sstart & 15);
        const uint8_t *gs = reinterpret_cast<const uint8_t *>(D.s) + sstart;
        uint8_t *sdst = dst + D.scale_off + a;
        const uint32_t head = min(sbytes, a ? 16u - a : 0u);
        const uint32_t body = (sbytes - head) & ~15u;
        for (uint32_t b = 0; b < head; b += 2)
            *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
        for (uint32_t b = head + body; b < sbytes; b += 2)
            *reinterpret_cast<uint16_t *>(sdst + b) = *reinterpret_cast<const uint16_t *>(gs + b);
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(rows) * static_cast<uint32_t>(D.K) + body);
        const int8_t *src = D.q + static_cast<int64_t>(r0) * D.K;
        for (int r = 0; r < rows; ++r)
            bulk_g2s(dst + r * D.RS, src + static_cast<int64_t>(r) * D.K, static_cast<uint32_t>(D.K), &full[slot]);
        if (body) bulk_g2s(sdst + head, gs + head, body, &full[slot]);
    };
    if (tid == 0) {
        const int d0 = find_pdesc(p, begin);
        for (int pi = 0; pi < min(S, nstages); ++pi) issue(pi, d0);
    }
    // the first stages are weights only; x and y only after the kernels
    // before this one (when launched as their dependent) have completed
    pdl_wait_prior();

    // ---- consumers --------------------------------------------------------------
    int d = find_pdesc(p, begin);
    int cur_d = -1;
    uint4 xr[KJ];          // x slice of activation row g, binary16
    int kb0 = 0, nblk = 0;
    uint32_t slow = 0u;    // blocks that take the exact bf16 path
    for (int i = begin, k = 0; i < end; ++i, ++k) {
        // every stage of this CTA is issued: a chained launch after this one
        // may start once all CTAs are this far
        if (!p.early_signal && k == max(0, nstages - S) && tid == 0) pdl_launch_dependents();
        while (i >= p.d[d].stage_begin + p.d[d].stages) ++d;
        const PDesc &D = p.d[d];
        const int lp = D.lp;
        const int P = 1 << lp;
        if (d != cur_d) {
            // this warp's x fragments: x[m = g][block kb0 + j][8t .. 8t+8), zero
            // past M; kept when the next matrix reads the same x slice
            const int nkb0 = (warp & (P - 1)) * D.bps;
            const int nnblk = max(0, min(D.nb - nkb0, D.bps));
            const bool same = cur_d >= 0 && D.x == p.d[cur_d].x && D.ldx == p.d[cur_d].ldx && nkb0 == kb0 &&
                              nnblk == nblk;
            cur_d = d;
            kb0 = nkb0;
            nblk = nnblk;
            if (!same) prep_x<KJ>(g < M ? D.x + g * D.ldx + kb0 * 32 + 8 * t : nullptr, nblk, xr, slow);
        }
        const int slot = k % S;
        if (!mbar_wait_bounded(&full[slot], (k / S) & 1)) {
            if (lane == 0 && p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
            drain_after_timeout();
            return;
        }
        const uint8_t *codes = smem_raw + static_cast<size_t>(slot) * p.slot_bytes;
        const int r0 = (i - D.stage_begin) * D.RT;
        const int rows = min(D.RT, D.N - r0);
        const uint16_t *scales = reinterpret_cast<const uint16_t *>(
            codes + D.scale_off + ((static_cast<int64_t>(r0) * D.nb * 2) & 15));
        // this warp's rows: row g of group ga (lower half of the tile) and, for
        // full tiles, row g of group ga + 8/P (upper half)
        const int ga = warp >> lp;
        const int ra = 8 * ga + g;
        const int rb = ra + (64 >> lp);
        const bool two = D.half == 0;
        const bool va = ra < rows;
        const bool vb = two && rb < rows;
        const uint8_t *ca = codes + ra * D.RS + kb0 * 32;
        const uint8_t *cb = codes + rb * D.RS + kb0 * 32;
        const uint16_t *sa = scales + ra * D.nb + kb0;
        const uint16_t *sb = scales + rb * D.nb + kb0;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const bool full_tile = rows == D.RT && nblk == D.bps;
        if (two) {
            if (full_tile && nblk == 12)
                tile_mma<12, true, true, KJ>(ca, cb, sa, sb, va, vb, nblk, t, xr, acc);
            else if (full_tile && nblk == 8)
                tile_mma<8, true, true, KJ>(ca, cb, sa, sb, va, vb, nblk, t, xr, acc);
            else if (full_tile && nblk == 4)
                tile_mma<4, true, true, KJ>(ca, cb, sa, sb, va, vb, nblk, t, xr, acc);
            else
                tile_mma<12, true, false, KJ>(ca, cb, sa, sb, va, vb, nblk, t, xr, acc);
        } else if constexpr (KJ >= 16) {
            if (full_tile && nblk == 16)
                tile_mma<16, false, true, KJ>(ca, cb, sa, sb, va, vb, nblk, t, xr, acc);
            else if (full_tile && nblk == 8)
                tile_mma<8, false, true, KJ>(ca, cb, sa, sb, va, vb, nblk, t, xr, acc);
            else
                tile_mma<16, false, false, KJ>(ca, cb, sa, sb, va, vb, nblk, t, xr, acc);
        }
        if (slow != 0u) {
            const float4 r = slow_blocks(ca, cb, sa, sb, va, vb, t, slow,
                                         g < M ? D.x + g * D.ldx + kb0 * 32 + 8 * t : nullptr,
                                         make_float4(acc[0], acc[1], acc[2], acc[3]));
            acc[0] = r.x;
            acc[1] = r.y;
            acc[2] = r.z;
            acc[3] = r.w;
        }
        // publish this warp's partial tile; the last of the tile's P warps adds
        // them in slice order and writes y
        const int tile = warp >> lp;
        uint8_t *rs = smem_raw + p.red_off + slot * p.red_entry;
        if (two)
            reinterpret_cast<float4 *>(rs)[warp * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        else
            reinterpret_cast<float2 *>(rs)[warp * 32 + lane] = make_float2(acc[0], acc[1]);
        __threadfence_block();
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) prev = atomicAdd(&cnt[slot * 8 + tile], 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == static_cast<uint32_t>(P - 1)) {
            __threadfence_block();
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sl = 0; sl < P; ++sl) {
                const int src = ((tile << lp) + sl) * 32 + lane;
                if (two) {
                    const float4 u = reinterpret_cast<const float4 *>(rs)[src];
                    if (sl == 0) {
                        v = u;
                    } else {
                        v.x += u.x;
                        v.y += u.y;
                        v.z += u.z;
                        v.w += u.w;
                    }
                } else {
                    const float2 u = reinterpret_cast<const float2 *>(rs)[src];
                    if (sl == 0) {
                        v.x = u.x;
                        v.y = u.y;
                    } else {
                        v.x += u.x;
                        v.y += u.y;
                    }
                }
            }
            const int m0 = 2 * t;
            if (va) {
                if (m0 < M) D.y[m0 * D.ldy + r0 + ra] = v.x;
                if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + r0 + ra] = v.y;
            }
            if (vb) {
                if (m0 < M) D.y[m0 * D.ldy + r0 + rb] = v.z;
                if (m0 + 1 < M) D.y[(m0 + 1) * D.ldy + r0 + rb] = v.w;
            }
            if (lane == 0) cnt[slot * 8 + tile] = 0u;
        }
        // release the slot: this warp's reads of the slot and of the partial
        // buffer are ordered (fence, counter, fence) before the refill that
        // the last of the 8 warps issues
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const uint32_t done = atomicAdd(&rel[slot], 1u);
            if (done == kWarps - 1) {
                __threadfence_block();
                rel[slot] = 0u;
                fence_proxy_async_smem();
                if (k + S < nstages) issue(k + S, d);
            }
        }
        __syncwarp();
    }
}

int g_configured_dev = -1;
int g_occ = 0;

template <int KJ>
bool configure_kernel(int &occ) {
    if (cudaFuncSetAttribute(pipe_kernel<KJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget) != cudaSuccess)
        return false;
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, pipe_kernel<KJ>, kThreads, kSmemBudget) != cudaSuccess)
        return false;
    occ = std::min(occ, std::max(o, 1));
    return true;
}

struct Shape {
    int P, lp, half, RT, RS, bps, scale_off, stage_bytes;
};

// Partial-tile buffer per slot: 8 warps x 32 lanes x float4 (full tiles) or
// float2 (half tiles).
constexpr int red_entry_bytes(bool any_full) { return kWarps * 32 * (any_full ? 16 : 8); }

Shape make_shape(int K, int half, int P) {
    Shape h{};
    const int nb = K / 32;
    h.P = P;
    h.lp = __builtin_ctz(static_cast<unsigned>(P));
    h.half = half;
    h.RT = (half ? 64 : 128) / P;
    h.RS = K + kPad;
    h.bps = (nb + P - 1) / P;
    h.scale_off = h.RT * h.RS;
    h.stage_bytes = h.scale_off + h.RT * nb * 2 + 16;
    return h;
}

// Slots of a ring of stages of `stage_bytes` (0 if fewer than 2 fit).
int slots_for(int stage_bytes, bool any_full) {
    const int slot = (stage_bytes + 127) / 128 * 128;
    for (int S = kMaxSlots; S >= 2; --S)
        if (S * slot + S * red_entry_bytes(any_full) + kCtlBytes <= kSmemBudget) return S;
    return 0;
}

// The stage shape of a matrix: full tiles (slices of at most 384, 128/P
// rows) or half tiles (slices of at most 512, 64/P rows), P the fewest slices
// that respect the slice width and fit two slots; full tiles if they fit,
// else (between half-tile shapes) the most bytes in flight.
// The shape depends on K alone, so a matrix is summed in the same order
// whatever else shares its launch (batched == separate calls, bit for bit).
Shape shape_of(int K) {
    Shape best{};
    long best_score = -1;
    for (int half = 0; half <= 1; ++half) {
        const int width = half ? kHalfSliceK : kSliceK;
        int P = 1;
        while (P * width < K && P < 8) P *= 2;
        if (P * width < K) continue;
        Shape h = make_shape(K, half, P);
        while (slots_for(h.stage_bytes, !half) == 0 && P < 8) {
            P *= 2;
            h = make_shape(K, half, P);
        }
        const int S = slots_for(h.stage_bytes, !half);
        if (S == 0) continue;
        // full tiles (12 x blocks per warp, two rows per lane) win whenever
        // they fit: measured faster than half tiles with more slots
        const long score = static_cast<long>(S) * h.stage_bytes + (half ? 0L : (1L << 40));
        if (score > best_score) {
            best = h;
            best_score = score;
        }
    }
    return best;  // RT == 0 if no shape fits
}

// Ring layout of a launch: slot size, slot count, offsets.  Returns false if
// some matrix has no shape or two slots do not fit.
bool layout_for(const q8_linear_desc *descs, int count, int &S, int &slot_bytes, int &red_off, int &ctl_off,
                int &red_entry) {
    int mx = 0;
    bool any_full = false;
    for (int i = 0; i < count; ++i) {
        const Shape h = shape_of(static_cast<int>(descs[i].K));
        if (h.RT == 0) return false;
        mx = std::max(mx, h.stage_bytes);
        any_full = any_full || !h.half;
    }
    S = slots_for(mx, any_full);
    if (S < 2) return false;
    slot_bytes = (mx + 127) / 128 * 128;
    red_entry = red_entry_bytes(any_full);
    red_off = S * slot_bytes;
    ctl_off = red_off + S * red_entry;
    return true;
}

}  // namespace

bool pipe_k_supported(int64_t K) { return K <= kPipeMaxK && shape_of(static_cast<int>(K)).RT != 0; }

namespace {

q8_status launch_set(const q8_linear_desc *descs, int count, int M, uint32_t *dev_status, cudaStream_t stream,
                     bool chained) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    if (g_configured_dev != di->device) {
        int o = 1 << 30;
        if (!configure_kernel<12>(o) || !configure_kernel<16>(o)) return Q8_ERR_CUDA;
        g_occ = o;
        g_configured_dev = di->device;
    }
    static thread_local PParams p;
    if (!layout_for(descs, count, p.S, p.slot_bytes, p.red_off, p.ctl_off, p.red_entry)) return Q8_ERR_UNSUPPORTED;
    double total_bytes = 0.0;
    int stages = 0;
    bool wide_x = false;  // some matrix needs more than 12 x blocks per warp
    for (int i = 0; i < count; ++i) {
        PDesc &D = p.d[i];
        const int K = static_cast<int>(descs[i].K);
        const Shape h = shape_of(K);
        D.q = descs[i].q;
        D.s = descs[i].s;
        D.x = descs[i].x;
        D.y = descs[i].y;
        D.ldx = descs[i].ldx;
        D.ldy = descs[i].ldy;
        D.N = static_cast<int32_t>(descs[i].N);
        D.K = K;
        D.nb = K / 32;
        D.RT = h.RT;
        D.RS = h.RS;
        D.P = h.P;
        D.lp = h.lp;
        D.half = h.half;
        D.bps = h.bps;
        D.scale_off = h.scale_off;
        wide_x = wide_x || h.half || h.bps > 12;
        D.stage_begin = stages;
        D.stages = (D.N + D.RT - 1) / D.RT;
        stages += D.stages;
        total_bytes += static_cast<double>(D.N) * K * 1.0625 * (D.half ? kHalfCost : 1.0);
    }
    p.status = dev_status;
    p.count = count;
    p.M = M;
    if (stages == 0) return Q8_OK;
    const int grid = std::min(std::min(stages, di->sm_count * g_occ), kMaxGrid);
    // cut the stage list into `grid` ranges of (nearly) equal work
    int c = 0;
    double acc = 0.0;
    p.cta_begin[0] = 0;
    for (int i = 0; i < count && c < grid - 1; ++i) {
        const PDesc &D = p.d[i];
        const double full = static_cast<double>(D.RT) * D.K * 1.0625 * (D.half ? kHalfCost : 1.0);
        for (int st = 0; st < D.stages && c < grid - 1; ++st) {
            const int rows = std::min(D.RT, D.N - st * D.RT);
            acc += full * rows / D.RT;
            while (c < grid - 1 && acc >= total_bytes * (c + 1) / grid) p.cta_begin[++c] = D.stage_begin + st + 1;
        }
    }
    while (c < grid) p.cta_begin[++c] = stages;
    const size_t smem = static_cast<size_t>(p.ctl_off) + kCtlBytes;
    p.early_signal = grid >= di->sm_count * g_occ ? 1 : 0;
    const cudaError_t e = wide_x ? launch_kernel(pipe_kernel<16>, dim3(grid), dim3(kThreads), smem, stream, chained, p)
                                 : launch_kernel(pipe_kernel<12>, dim3(grid), dim3(kThreads), smem, stream, chained, p);
    return e == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}

}  // namespace

q8_status launch_pipe(const q8_linear_desc *descs, int count, int M, uint32_t *dev_status, cudaStream_t stream,
                      bool chained) {
    if (M < 1 || M > 8) return Q8_ERR_UNSUPPORTED;
    for (int i = 0; i < count; ++i)
        if (!pipe_k_supported(descs[i].K)) return Q8_ERR_UNSUPPORTED;
    // every mix of K <= 4096 fits one ring (the largest half-tile stage
    // with a full tile's reduction entries still leaves two slots), so the
    // launch never depends on which matrices share it
    return launch_set(descs, count, M, dev_status, stream, chained);
}

}  // namespace q8
