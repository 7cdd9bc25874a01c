// q8_skinny.cu -- Q8_0 W8A16 matmul for 1 <= M <= 32 decode rows.
//
// Y[m][n] = sum_k s[n][k/32] * q[n][k] * x[m][k]; "Frigg" README, Finding 8
// (W8A16 decode: every weight is read from HBM exactly once per call, whatever
// M is; split-K goes through a partial-sum buffer, not float atomics, so that
// replays are bit-identical).
//
// One persistent kernel serves q8_gemv, q8_gemm_skinny and q8_linear_batch:
// the host flattens every matrix into work items (matrix, 128-row tile,
// K split) and the grid (SMs x resident CTAs) walks that static list.
//
// Per work item, a CTA of 8 warps
//   1. has the activation slice x[0..M)[k0..k1) copied into shared memory by
//      bulk async copies (cp.async.bulk, one per row, completion on an
//      mbarrier; double-buffered so the next item's slice lands while this
//      one computes);
//   2. streams its 128 weight rows: each warp owns 16 rows, lane (g = lane/4,
//      t = lane%4) reads bytes [8t, 8t+8) of every 32-code block of rows g and
//      g+8 (one 32-byte sector per row per block across the 4 lanes) with
//      non-allocating 8-byte loads, several blocks in flight;
//   3. dequantises in registers and multiplies:
//        SIMT: codes -> fp32 exactly, one FMA per weight per activation row,
//              block sum times the block scale, fp32 accumulators;
//        MMA : codes -> bf16 exactly (integers |q| <= 127), one warp
//              mma.sync m16n8k16 (bf16 in, fp32 out) per half block with the
//              weights as the 16-row A operand and x^T as B (n = M rows,
//              padded to 8), then the block scale is applied to the fp32
//              result; products q*x are exact, only fp32 summation rounds;
//   4. writes y, or -- when K is split -- its fp32 partial sums plus an
//      atomic ticket; the CTA that draws the last ticket adds the partials in
//      split order 0..S-1 (fixed, hence deterministic) and resets the ticket.
// No wait in this kernel can block forever: the copy waits give up after a
// time limit and report Q8_DEV_TIMEOUT; the split-K ticket never waits.
#include <algorithm>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "q8_dev.cuh"
#include "q8_internal.h"

namespace q8 {

namespace {

constexpr int kU = 4;  // blocks per unrolled step (loads in flight per thread: 2*kU)

struct DescDev {
    const int8_t *q;
    const uint16_t *s;
    const uint16_t *x;
    float *y;
    float *part;        // [S][M][N] fp32 partials, or null if S == 1
    const int8_t *xq;   // W8A8: x quantized to Q8_0, codes [M][K] ...
    const uint16_t *xs; // ... and binary16 scales [M][K / 32]
    uint32_t *tickets;  // [tiles], or null if S == 1
    int64_t K;
    int64_t ldx;
    int64_t ldy;
    int32_t N;
    int32_t nb;         // blocks per row (K / 32)
    int32_t S;
    int32_t bps;        // blocks per split
    int32_t tiles;
    int32_t item_begin;
};

struct BatchParams {
    DescDev d[Q8_MAX_BATCH];
    uint32_t *status;
    int32_t count;
    int32_t M;
    int32_t total_items;
};

template <int MT, int VAR>
struct Cfg {
    static constexpr int KSB = MT <= 8 ? 64 : (MT <= 16 ? 32 : 16);  // == ksb_for_m
    // bytes per staged x row: KSB blocks of 32 bf16 (W8A8: of 32 codes)
    static constexpr int XROW = KSB * (VAR == Q8_VARIANT_W8A8 ? 32 : 64) + 16;
    static constexpr int XROWS = MT;                                     // rows per buffer
    static constexpr int XBUF = XROWS * XROW;
    static constexpr int SMEM = 128 + 2 * XBUF;
    static constexpr int MINB = (VAR == Q8_VARIANT_SIMT && MT >= 16) ? 1 : 2;
};

__device__ __forceinline__ int find_desc(const BatchParams &p, int item) {
    int d = 0;
    while (d + 1 < p.count && item >= p.d[d + 1].item_begin) ++d;
    return d;
}

template <int MT, int VAR>
__device__ __forceinline__ void issue_x(const BatchParams &p, int item, uint8_t *xb, uint64_t *bar) {
    const int d = find_desc(p, item);
    const DescDev &D = p.d[d];
    const int local = item - D.item_begin;
    const int split = local % D.S;
    const int kb0 = split * D.bps;
    const int nblk = min(D.bps, D.nb - kb0);
    if constexpr (VAR == Q8_VARIANT_W8A8) {
        // the codes of x's blocks (16-byte aligned: K and kb0 * 32 are multiples of 32)
        const uint32_t bytes = static_cast<uint32_t>(nblk) * 32u;
        mbar_arrive_expect_tx(bar, bytes * static_cast<uint32_t>(p.M));
        for (int m = 0; m < p.M; ++m)
            bulk_g2s(xb + m * Cfg<MT, VAR>::XROW, D.xq + m * D.K + static_cast<int64_t>(kb0) * 32, bytes, bar);
    } else {
        const uint32_t bytes = static_cast<uint32_t>(nblk) * 64u;
        mbar_arrive_expect_tx(bar, bytes * static_cast<uint32_t>(p.M));
        for (int m = 0; m < p.M; ++m)
            bulk_g2s(xb + m * Cfg<MT, VAR>::XROW, D.x + m * D.ldx + static_cast<int64_t>(kb0) * 32, bytes, bar);
    }
}

// Per-thread results of one item: rows g and g+8 of the warp's 16 rows.
//   MMA, W8A8: acc[j][0..1] = row g,   m = 8j + 2t + {0,1}
//         acc[j][2..3] = row g+8, m = 8j + 2t + {0,1}
//   SIMT: after the lane reduction, accg[m] / acch[m] for every m (all four
//         t-lanes hold the sums; lane t stores m with m % 4 == t).

template <int MT, int VAR>
__device__ __forceinline__ void compute_item(const BatchParams &p, int item, const uint8_t *xb,
                                             int &s_last_flag) {
    constexpr int NT = (MT + 7) / 8;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int M = p.M;

    const int d = find_desc(p, item);
    const DescDev &D = p.d[d];
    const int local = item - D.item_begin;
    const int tile = local / D.S;
    const int split = local % D.S;
    const int kb0 = split * D.bps;
    const int nblk = min(D.bps, D.nb - kb0);
    const int N = D.N;
    const int64_t K = D.K;

    const int n0 = tile * kTileRows + warp * 16;
    const int ng = n0 + g;
    const int nh = n0 + g + 8;
    const int rg = min(ng, N - 1);  // clamp: rows past N read row N-1, results are dropped
    const int rh = min(nh, N - 1);
    const int8_t *qg = D.q + static_cast<int64_t>(rg) * K + static_cast<int64_t>(kb0) * 32 + 8 * t;
    const int8_t *qh = D.q + static_cast<int64_t>(rh) * K + static_cast<int64_t>(kb0) * 32 + 8 * t;
    const uint16_t *sg = D.s + static_cast<int64_t>(rg) * D.nb + kb0;
    const uint16_t *sh = D.s + static_cast<int64_t>(rh) * D.nb + kb0;

    float acc[NT][4];
    float accg[MT], acch[MT];
    if constexpr (VAR != Q8_VARIANT_SIMT) {
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) accg[m] = acch[m] = 0.f;
    }

    for (int b = 0; b < nblk; b += kU) {
        uint2 cg[kU], ch[kU];
        uint32_t sgr[kU], shr[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (b + u < nblk) {
                cg[u] = ldg_stream_u2(qg + (b + u) * 32);
                ch[u] = ldg_stream_u2(qh + (b + u) * 32);
                sgr[u] = ldg_stream_u16(sg + b + u);
                shr[u] = ldg_stream_u16(sh + b + u);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (b + u < nblk) {
                const float sgv = f16_bits_to_f32(sgr[u]);
                const float shv = f16_bits_to_f32(shr[u]);
                if constexpr (VAR == Q8_VARIANT_W8A8) {
                    // one int8 MMA per block and 8 activation rows: each
                    // lane's 8 code bytes stand for the same k slots
                    // {4t..4t+3, 16+4t..16+4t+3} of weights and x (the dot
                    // product is the same for any common order of k); the
                    // exact int32 dot times s_w * s_x (exact in fp32)
                    const uint8_t *xrow = xb + (b + u) * 32 + 8 * t;
                    const int kb = kb0 + b + u;
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        uint2 xa = make_uint2(0u, 0u);
                        if (8 * j + g < M)
                            xa = *reinterpret_cast<const uint2 *>(xrow + (8 * j + g) * Cfg<MT, VAR>::XROW);
                        int d0, d1, d2, d3;
                        mma_s8_16832(d0, d1, d2, d3, cg[u].x, ch[u].x, cg[u].y, ch[u].y, xa.x, xa.y);
                        const int m0 = 8 * j + 2 * t;
                        const float x0 = m0 < M ? f16_bits_to_f32(__ldg(D.xs + static_cast<int64_t>(m0) * D.nb + kb)) : 0.f;
                        const float x1 =
                            m0 + 1 < M ? f16_bits_to_f32(__ldg(D.xs + static_cast<int64_t>(m0 + 1) * D.nb + kb)) : 0.f;
                        acc[j][0] = fmaf(sgv * x0, static_cast<float>(d0), acc[j][0]);
                        acc[j][1] = fmaf(sgv * x1, static_cast<float>(d1), acc[j][1]);
                        acc[j][2] = fmaf(shv * x0, static_cast<float>(d2), acc[j][2]);
                        acc[j][3] = fmaf(shv * x1, static_cast<float>(d3), acc[j][3]);
                    }
                } else if constexpr (VAR == Q8_VARIANT_MMA) {
                    const uint8_t *xrow = xb + (b + u) * 64 + 16 * t;
                    uint32_t g01, g23, g45, g67, h01, h23, h45, h67;
                    codes4_to_bf16x2(cg[u].x, g01, g23);
                    codes4_to_bf16x2(cg[u].y, g45, g67);
                    codes4_to_bf16x2(ch[u].x, h01, h23);
                    codes4_to_bf16x2(ch[u].y, h45, h67);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                        if (8 * j + g < M)
                            xv = *reinterpret_cast<const uint4 *>(xrow + (8 * j + g) * Cfg<MT, VAR>::XROW);
                        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
                        // block positions 8t+{0..3} (first k16 step) and 8t+{4..7}
                        mma_bf16_16816(d0, d1, d2, d3, g01, h01, g23, h23, xv.x, xv.y);
                        mma_bf16_16816(d0, d1, d2, d3, g45, h45, g67, h67, xv.z, xv.w);
                        acc[j][0] = fmaf(sgv, d0, acc[j][0]);
                        acc[j][1] = fmaf(sgv, d1, acc[j][1]);
                        acc[j][2] = fmaf(shv, d2, acc[j][2]);
                        acc[j][3] = fmaf(shv, d3, acc[j][3]);
                    }
                } else {
                    const uint8_t *xrow = xb + (b + u) * 64 + 16 * t;
                    float cgf[8], chf[8];
                    codes4_to_f32(cg[u].x, cgf[0], cgf[1], cgf[2], cgf[3]);
                    codes4_to_f32(cg[u].y, cgf[4], cgf[5], cgf[6], cgf[7]);
                    codes4_to_f32(ch[u].x, chf[0], chf[1], chf[2], chf[3]);
                    codes4_to_f32(ch[u].y, chf[4], chf[5], chf[6], chf[7]);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < M) {
                            const uint4 xv = *reinterpret_cast<const uint4 *>(xrow + m * Cfg<MT, VAR>::XROW);
                            const float x0 = bf16lo_f32(xv.x), x1 = bf16hi_f32(xv.x);
                            const float x2 = bf16lo_f32(xv.y), x3 = bf16hi_f32(xv.y);
                            const float x4 = bf16lo_f32(xv.z), x5 = bf16hi_f32(xv.z);
                            const float x6 = bf16lo_f32(xv.w), x7 = bf16hi_f32(xv.w);
                            float pg = cgf[0] * x0;
                            float ph = chf[0] * x0;
                            pg = fmaf(cgf[1], x1, pg); ph = fmaf(chf[1], x1, ph);
                            pg = fmaf(cgf[2], x2, pg); ph = fmaf(chf[2], x2, ph);
                            pg = fmaf(cgf[3], x3, pg); ph = fmaf(chf[3], x3, ph);
                            pg = fmaf(cgf[4], x4, pg); ph = fmaf(chf[4], x4, ph);
                            pg = fmaf(cgf[5], x5, pg); ph = fmaf(chf[5], x5, ph);
                            pg = fmaf(cgf[6], x6, pg); ph = fmaf(chf[6], x6, ph);
                            pg = fmaf(cgf[7], x7, pg); ph = fmaf(chf[7], x7, ph);
                            accg[m] = fmaf(sgv, pg, accg[m]);
                            acch[m] = fmaf(shv, ph, acch[m]);
                        }
                    }
                }
            }
        }
    }

    if constexpr (VAR == Q8_VARIANT_SIMT) {
        // sum the four t-lanes of each row (fixed butterfly order)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            accg[m] += __shfl_xor_sync(0xffffffffu, accg[m], 1);
            acch[m] += __shfl_xor_sync(0xffffffffu, acch[m], 1);
            accg[m] += __shfl_xor_sync(0xffffffffu, accg[m], 2);
            acch[m] += __shfl_xor_sync(0xffffffffu, acch[m], 2);
        }
    }

    // ---- epilogue ------------------------------------------------------------
    float *out;
    int64_t ld;
    if (D.S == 1) {
        out = D.y;
        ld = D.ldy;
    } else {
        out = D.part + static_cast<int64_t>(split) * M * N;
        ld = N;
    }
    if constexpr (VAR != Q8_VARIANT_SIMT) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int m0 = 8 * j + 2 * t;
            if (ng < N) {
                if (m0 < M) out[m0 * ld + ng] = acc[j][0];
                if (m0 + 1 < M) out[(m0 + 1) * ld + ng] = acc[j][1];
            }
            if (nh < N) {
                if (m0 < M) out[m0 * ld + nh] = acc[j][2];
                if (m0 + 1 < M) out[(m0 + 1) * ld + nh] = acc[j][3];
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M && (m & 3) == t) {
                if (ng < N) out[m * ld + ng] = accg[m];
                if (nh < N) out[m * ld + nh] = acch[m];
            }
        }
    }

    if (D.S > 1) {
        // publish this split, draw a ticket; the last split of the tile reduces
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const uint32_t prev = atomicAdd(D.tickets + tile, 1u);
            s_last_flag = (prev == static_cast<uint32_t>(D.S - 1)) ? 1 : 0;
        }
        __syncthreads();
        if (s_last_flag) {
            __threadfence();
            const int r0 = tile * kTileRows;
            for (int e = tid; e < M * kTileRows; e += kSkinnyThreads) {
                const int m = e / kTileRows;
                const int n = r0 + (e - m * kTileRows);
                if (n < N) {
                    const float *pp = D.part + static_cast<int64_t>(m) * N + n;
                    float v = __ldcg(pp);
                    for (int sp = 1; sp < D.S; ++sp) v += __ldcg(pp + static_cast<int64_t>(sp) * M * N);
                    D.y[m * D.ldy + n] = v;
                }
            }
            if (tid == 0) D.tickets[tile] = 0u;  // ready for the next call / replay
        }
    }
}

template <int MT, int VAR>
__global__ void __launch_bounds__(kSkinnyThreads, Cfg<MT, VAR>::MINB)
skinny_kernel(const __grid_constant__ BatchParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *xbase = smem + 128;
    __shared__ int s_last;
    const int tid = threadIdx.x;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // chained launches: wait for the previous kernel before reading x or the
    // workspace (a chained launch after this one starts when this one ends)
    pdl_wait_prior();

    int item = blockIdx.x;
    if (item >= p.total_items) return;
    if (tid == 0) issue_x<MT, VAR>(p, item, xbase, &bars[0]);

    int it = 0;
    int timed_out = 0;
    for (; item < p.total_items; ++it, item += gridDim.x) {
        const int buf = it & 1;
        int bad = mbar_wait_bounded(&bars[buf], (it >> 1) & 1) ? 0 : 1;
        bad = __syncthreads_or(bad);  // also: everyone is done with buffer buf^1
        if (bad) {
            timed_out = 1;
            break;
        }
        const int next = item + gridDim.x;
        if (tid == 0 && next < p.total_items)
            issue_x<MT, VAR>(p, next, xbase + (buf ^ 1) * Cfg<MT, VAR>::XBUF, &bars[buf ^ 1]);
        compute_item<MT, VAR>(p, item, xbase + buf * Cfg<MT, VAR>::XBUF, s_last);
    }
    if (timed_out && tid == 0) {
        if (p.status) atomicOr(p.status, Q8_DEV_TIMEOUT);
        // let the copy we gave up on land before the CTA's shared memory goes away
        (void)mbar_wait_bounded(&bars[it & 1], (it >> 1) & 1);
    }
}

template <int MT, int VAR>
q8_status run(const BatchParams &p, const DeviceInfo *di, cudaStream_t stream, bool chained) {
    using C = Cfg<MT, VAR>;
    static int configured_dev = -1;
    static int occ = 0;
    if (configured_dev != di->device) {
        if (cudaFuncSetAttribute(skinny_kernel<MT, VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return Q8_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, skinny_kernel<MT, VAR>, kSkinnyThreads, C::SMEM) != cudaSuccess)
            return Q8_ERR_CUDA;
        occ = std::max(o, 1);
        configured_dev = di->device;
    }
    const int grid = std::min(p.total_items, di->sm_count * occ);
    return launch_kernel(skinny_kernel<MT, VAR>, dim3(grid), dim3(kSkinnyThreads), C::SMEM, stream, chained, p) ==
                   cudaSuccess
               ? Q8_OK
               : Q8_ERR_CUDA;
}

}  // namespace

// Split heuristic: a function of (N, K, M) only, so a matrix gets the same
// split -- hence the same bits -- alone or inside a batch.
static void plan_one(int64_t N, int64_t K, int M, SplitPlan &pl, bool invariant) {
    constexpr int kTargetItems = 512;
    const int nb = static_cast<int>(K / 32);
    pl.tiles = static_cast<int32_t>((N + kTileRows - 1) / kTileRows);
    if (invariant) {
        // the split from K alone (the fewest ranges whose x slices fit the
        // staging of every M): the sum order does not depend on M
        const int S0 = (nb + ksb_for_m(Q8_SKINNY_MAX_M) - 1) / ksb_for_m(Q8_SKINNY_MAX_M);
        pl.bps = (nb + S0 - 1) / S0;
        pl.S = (nb + pl.bps - 1) / pl.bps;
        return;
    }
    const int s_min = (nb + ksb_for_m(M) - 1) / ksb_for_m(M);
    const int s_want = (kTargetItems + pl.tiles - 1) / pl.tiles;
    const int s_cap_blocks = std::max(1, nb / 8);                                   // >= 8 blocks per split
    const int s_cap_traffic = std::max(1, static_cast<int>(K / (30 * static_cast<int64_t>(M))));  // partials <= ~1/4 of weight bytes
    int S = std::max(s_min, std::min(s_want, std::min(s_cap_blocks, s_cap_traffic)));
    S = std::min(S, nb);
    int bps = (nb + S - 1) / S;
    S = (nb + bps - 1) / bps;
    pl.S = S;
    pl.bps = bps;
}

size_t plan_skinny(const q8_linear_desc *descs, int count, int M, SplitPlan *plans, bool invariant) {
    size_t off = 0;
    for (int i = 0; i < count; ++i) {
        plan_one(descs[i].N, descs[i].K, M, plans[i], invariant);
        plans[i].part_off = plans[i].ticket_off = 0;
        if (plans[i].S > 1) {
            plans[i].ticket_off = off;
            off += (static_cast<size_t>(plans[i].tiles) * 4 + 255) / 256 * 256;
            plans[i].part_off = off;
            off += (static_cast<size_t>(plans[i].S) * M * descs[i].N * 4 + 255) / 256 * 256;
        }
    }
    return off;
}

namespace {

enum Route { kRouteGemv, kRoutePipe, kRouteTile, kRouteGeneral, kRoutes };

// The kernel that serves one matrix, from its own K, M and the variant only,
// so a matrix gets the same kernel -- hence the same bits -- whatever else
// shares its call.  M = 1: the CUDA-core bulk-copy GEMV (AUTO, SIMT);
// M = 2..8: the TMA-fed chunked tile kernel for K % 256 == 0 except
// K = 1536, the warp-MMA bulk-copy pipeline for K = 1536 and for the other
// K it takes (also M = 1 with MMA), the tile kernel with a partial last
// chunk beyond; M = 9..32: the tile kernel (any K >= 256); everything else:
// the general kernel below.  The batch-invariant variant takes the tile kernel's
// bf16 arithmetic for K % 256 == 0 and the general kernel's warp-MMA
// arithmetic with a split of K that depends on K alone otherwise (for
// both, each output row's sums depend on that row only, never on M); W8A8
// takes the tiles' int8 block dots for K % 256 == 0 and the general
// kernel's for other K.  (Measured on 64-matrix batches at M = 2..8: the tiles are
// 10-35 % faster at K = 512..1280 and 4096; at K = 1536, the pipeline's
// best stage shape, the two are within 4 % and a lone matrix takes 8.7 us
// on the pipeline against 10.7 us on the tiles.)
Route route_of(int64_t K, int M, int variant) {
    if (variant == Q8_VARIANT_BATCH_INVARIANT || variant == Q8_VARIANT_W8A8)
        return tile_k_whole_chunks(K) ? kRouteTile : kRouteGeneral;
    if (M == 1 && variant != Q8_VARIANT_MMA && gemv_k_supported(K)) return kRouteGemv;
    if (variant == Q8_VARIANT_SIMT) return kRouteGeneral;
    if (M <= 8 && pipe_k_supported(K) && (K == 1536 || !tile_k_whole_chunks(K))) return kRoutePipe;
    if (M >= 2 && tile_k_supported(K)) return kRouteTile;
    if (M <= 8 && pipe_k_supported(K)) return kRoutePipe;
    return kRouteGeneral;
}

}  // namespace

namespace {

size_t up256b(int64_t b) { return static_cast<size_t>((b + 255) / 256 * 256); }

// W8A8 on the general kernel: each distinct x (pointer, row stride, K) is
// widened to binary32 [M][K] and quantized to Q8_0 by the A1 quantizer:
// codes [M][K] and binary16 scales [M][K / 32], each 256-byte rounded.
size_t w8a8_x_bytes(int64_t K, int M) {
    return up256b(static_cast<int64_t>(M) * K * 4) + up256b(static_cast<int64_t>(M) * K) +
           up256b(static_cast<int64_t>(M) * (K / 32) * 2);
}
// index of the first matrix with the same x as matrix i
int first_same_x(const q8_linear_desc *d, int i) {
    for (int j = 0; j < i; ++j)
        if (d[j].x == d[i].x && d[j].ldx == d[i].ldx && d[j].K == d[i].K) return j;
    return i;
}

// bf16 x [M][ldx] -> binary32 [M][K]
__global__ void widen_rows_kernel(const uint16_t *__restrict__ x, int64_t ldx, int M, int64_t K,
                                  float *__restrict__ xf) {
    const int64_t total = static_cast<int64_t>(M) * K;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / K;
        xf[i] = __uint_as_float(static_cast<uint32_t>(x[m * ldx + (i - m * K)]) << 16);
    }
}

}  // namespace

// The W8A8 workspace: the tile kernel's for K % 256 == 0, then the general
// kernel's quantized x and its split-K partials for the other matrices.
size_t w8a8_workspace(const q8_linear_desc *all, int all_count, int M, size_t *gen_x_off, size_t *gen_plan_off) {
    q8_linear_desc tiles[Q8_MAX_BATCH], gen[Q8_MAX_BATCH];
    int nt = 0, ng = 0;
    for (int i = 0; i < all_count; ++i) {
        if (tile_k_whole_chunks(all[i].K)) tiles[nt++] = all[i];
        else gen[ng++] = all[i];
    }
    size_t off = nt > 0 ? tile_workspace(tiles, nt, M, nullptr, nullptr, true) : 0;
    if (gen_x_off) *gen_x_off = off;
    for (int i = 0; i < ng; ++i)
        if (first_same_x(gen, i) == i) off += w8a8_x_bytes(gen[i].K, M);
    if (gen_plan_off) *gen_plan_off = off;
    SplitPlan plans[Q8_MAX_BATCH];
    return off + (ng > 0 ? plan_skinny(gen, ng, M, plans, false) : 0);
}

size_t skinny_workspace(const q8_linear_desc *descs, int count, int M, SplitPlan *plans, size_t *sched_off,
                        size_t *tile_off) {
    size_t need = count > 0 ? plan_skinny(descs, count, M, plans, false) : 0;
    *sched_off = SIZE_MAX;
    bool gemv = false;
    q8_linear_desc tiles[Q8_MAX_BATCH];
    int ntiles = 0;
    for (int i = 0; i < count; ++i) {
        const Route r = route_of(descs[i].K, M, Q8_VARIANT_AUTO);
        gemv = gemv || r == kRouteGemv;
        if (r == kRouteTile && ntiles < Q8_MAX_BATCH) tiles[ntiles++] = descs[i];
    }
    const size_t tile_bytes = ntiles > 0 ? tile_workspace(tiles, ntiles, M) : 0;
    if (gemv) {
        *sched_off = (need + 255) / 256 * 256;
        need = *sched_off + 256;
    }
    if (tile_off) *tile_off = SIZE_MAX;
    if (tile_bytes > 0) {
        const size_t off = (need + 255) / 256 * 256;
        if (tile_off) *tile_off = off;
        need = off + tile_bytes;
    }
    return need;
}

namespace {

// The words the kernels count with (split-K tickets, the GEMV's pool
// counter) are left zero by every launch, but where they sit depends on the
// call's shapes: another call's partial sums or x copies can cover them.  So
// the library keeps, per workspace address, the byte ranges that calls
// enqueued on it may have left nonzero (their partial sums and x copies); a
// call clears those of its counter ranges that meet one (one memset each,
// in its stream), and an address seen for the first time is taken as all
// nonzero.  Calls that write no such data (the GEMV) or repeat the same
// shapes clear nothing.
struct Range {
    size_t off, len;
};
std::mutex g_ws_mu;
std::unordered_map<const void *, std::vector<Range>> g_ws_dirty;
constexpr size_t kMaxTrackedWorkspaces = 1 << 16;
constexpr size_t kMaxDirtyRanges = 64;

bool meets(const std::vector<Range> &set, const Range &r) {
    for (const Range &d : set)
        if (d.off < r.off + r.len && r.off < d.off + d.len) return true;
    return false;
}

// set minus r (pieces of at most two ranges per member)
void subtract(std::vector<Range> &set, const Range &r) {
    std::vector<Range> out;
    for (const Range &d : set) {
        if (d.off + d.len <= r.off || r.off + r.len <= d.off) {
            out.push_back(d);
            continue;
        }
        if (d.off < r.off) out.push_back({d.off, r.off - d.off});
        if (d.off + d.len > r.off + r.len) out.push_back({r.off + r.len, d.off + d.len - (r.off + r.len)});
    }
    set.swap(out);
}

q8_status clear_met_counters(void *ws, const std::vector<Range> &counters, const std::vector<Range> &data,
                             cudaStream_t stream) {
    if (ws == nullptr) return Q8_OK;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    auto it = g_ws_dirty.find(ws);
    if (it == g_ws_dirty.end()) {
        // (a forgotten address is taken as unknown again: cleared on its next use)
        if (g_ws_dirty.size() >= kMaxTrackedWorkspaces) g_ws_dirty.clear();
        it = g_ws_dirty.emplace(ws, std::vector<Range>{{0, SIZE_MAX / 2}}).first;
    }
    std::vector<Range> &dirty = it->second;
    for (const Range &r : counters) {
        if (!meets(dirty, r)) continue;
        if (cudaMemsetAsync(static_cast<uint8_t *>(ws) + r.off, 0, r.len, stream) != cudaSuccess) return Q8_ERR_CUDA;
        subtract(dirty, r);
    }
    for (const Range &r : data) {
        subtract(dirty, r);
        dirty.push_back(r);
    }
    // a long history collapses into one range over all of it (more clearing, never less)
    if (dirty.size() > kMaxDirtyRanges) {
        size_t lo = SIZE_MAX, hi = 0;
        for (const Range &d : dirty) {
            lo = std::min(lo, d.off);
            hi = std::max(hi, d.off + d.len);
        }
        dirty.assign(1, Range{lo, hi - lo});
    }
    return Q8_OK;
}

}  // namespace

q8_status launch_skinny(const q8_linear_desc *all, int all_count, int M, int variant,
                        void *ws, size_t ws_bytes, uint32_t *dev_status, cudaStream_t stream, bool chained) {
    const DeviceInfo *di = device_info();
    if (!di) return Q8_ERR_CUDA;
    static thread_local q8_linear_desc part[kRoutes][Q8_MAX_BATCH];
    int n[kRoutes] = {0, 0, 0, 0};
    for (int i = 0; i < all_count; ++i) {
        const Route r = route_of(all[i].K, M, variant);
        part[r][n[r]++] = all[i];
    }
    // the documented workspace (the plan of every matrix, whatever kernel
    // serves it, and the GEMV's pool counter) is checked before anything is
    // enqueued; the general kernel uses the front of it
    SplitPlan plans[Q8_MAX_BATCH];
    size_t sched_off = SIZE_MAX, tile_off = SIZE_MAX;
    // the batch-invariant arithmetic needs the general kernel's partial sums
    // for its matrices (K % 256 != 0) only; W8A8 (tiles only) needs the tile
    // kernel's, from the start of the workspace
    size_t need = 0, w8_x_off = 0, w8_plan_off = 0;
    if (variant == Q8_VARIANT_W8A8) {
        need = w8a8_workspace(all, all_count, M, &w8_x_off, &w8_plan_off);
        tile_off = 0;
    } else if (variant == Q8_VARIANT_BATCH_INVARIANT) {
        need = n[kRouteGeneral] > 0 ? plan_skinny(part[kRouteGeneral], n[kRouteGeneral], M, plans, true) : 0;
    } else {
        need = skinny_workspace(all, all_count, M, plans, &sched_off, &tile_off);
    }
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return Q8_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(ws) & 255u)) return Q8_ERR_ALIGN;
    const q8_linear_desc *descs = part[kRouteGeneral];
    const int count = n[kRouteGeneral];
    if (count > 0) plan_skinny(descs, count, M, plans, variant == Q8_VARIANT_BATCH_INVARIANT);
    // every item's x slice fits the staging buffer of this M (the plans keep
    // to it; checked before anything is enqueued)
    for (int i = 0; i < count; ++i)
        if (plans[i].bps > ksb_for_m(M)) return Q8_ERR_UNSUPPORTED;
    {
        // this call's counter words (cleared first where an earlier call on
        // this workspace may have left data) and the data it writes
        std::vector<Range> counters, data;
        if (sched_off != SIZE_MAX) counters.push_back({sched_off, 256});
        if (n[kRouteTile] > 0 && tile_off != SIZE_MAX && variant != Q8_VARIANT_BATCH_INVARIANT) {
            size_t toff = 0, tbytes = 0;
            const size_t total =
                tile_workspace(part[kRouteTile], n[kRouteTile], M, &toff, &tbytes, variant == Q8_VARIANT_W8A8);
            if (tbytes > 0) counters.push_back({tile_off + toff, tbytes});
            if (toff > 0) data.push_back({tile_off, toff});  // x copies and flags
            if (total > toff + tbytes) data.push_back({tile_off + toff + tbytes, total - toff - tbytes});
        }
        const size_t gbase = variant == Q8_VARIANT_W8A8 ? w8_plan_off : 0;
        if (variant == Q8_VARIANT_W8A8 && w8_plan_off > w8_x_off) data.push_back({w8_x_off, w8_plan_off - w8_x_off});
        for (int i = 0; i < count; ++i) {
            if (plans[i].S <= 1) continue;
            counters.push_back({gbase + plans[i].ticket_off, plans[i].part_off - plans[i].ticket_off});
            data.push_back({gbase + plans[i].part_off,
                            static_cast<size_t>(plans[i].S) * M * static_cast<size_t>(descs[i].N) * 4});
        }
        const q8_status st = clear_met_counters(ws, counters, data, stream);
        if (st != Q8_OK) return st;
    }
    if (n[kRouteGemv] > 0) {
        uint32_t *sched = sched_off == SIZE_MAX
                              ? nullptr
                              : reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + sched_off);
        const q8_status st = launch_gemv(part[kRouteGemv], n[kRouteGemv], sched, dev_status, stream, chained);
        if (st != Q8_OK) return st;
    }
    if (n[kRoutePipe] > 0) {
        const q8_status st = launch_pipe(part[kRoutePipe], n[kRoutePipe], M, dev_status, stream, chained);
        if (st != Q8_OK) return st;
    }
    if (n[kRouteTile] > 0) {
        uint8_t *xws = tile_off == SIZE_MAX ? nullptr : static_cast<uint8_t *>(ws) + tile_off;
        const int mode = variant == Q8_VARIANT_BATCH_INVARIANT ? 1 : (variant == Q8_VARIANT_W8A8 ? 2 : 0);
        const q8_status st = launch_tile(part[kRouteTile], n[kRouteTile], M, xws, dev_status, stream, chained, mode);
        if (st != Q8_OK) return st;
    }
    if (count == 0) return Q8_OK;

    // W8A8: quantize each distinct x of the general kernel's matrices
    // (binary32 copy, then the A1 quantizer) ahead of the kernel, in order
    const int8_t *w8_q[Q8_MAX_BATCH] = {};
    const uint16_t *w8_s[Q8_MAX_BATCH] = {};
    if (variant == Q8_VARIANT_W8A8) {
        size_t off = w8_x_off;
        for (int i = 0; i < count; ++i) {
            const int j = first_same_x(descs, i);
            if (j < i) {
                w8_q[i] = w8_q[j];
                w8_s[i] = w8_s[j];
                continue;
            }
            const int64_t K = descs[i].K;
            uint8_t *base = static_cast<uint8_t *>(ws) + off;
            float *xf = reinterpret_cast<float *>(base);
            int8_t *xq = reinterpret_cast<int8_t *>(base + up256b(static_cast<int64_t>(M) * K * 4));
            uint16_t *xs = reinterpret_cast<uint16_t *>(base + up256b(static_cast<int64_t>(M) * K * 4) +
                                                        up256b(static_cast<int64_t>(M) * K));
            off += w8a8_x_bytes(K, M);
            const int64_t total = static_cast<int64_t>(M) * K;
            const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 4096));
            widen_rows_kernel<<<blocks, 256, 0, stream>>>(descs[i].x, descs[i].ldx, M, K, xf);
            if (cudaGetLastError() != cudaSuccess) return Q8_ERR_CUDA;
            const q8_status st = launch_quantize(xf, M, K, xq, xs, dev_status, stream);
            if (st != Q8_OK) return st;
            w8_q[i] = xq;
            w8_s[i] = xs;
        }
    }
    uint8_t *plan_base = static_cast<uint8_t *>(ws) + (variant == Q8_VARIANT_W8A8 ? w8_plan_off : 0);

    BatchParams p;
    int items = 0;
    for (int i = 0; i < count; ++i) {
        DescDev &D = p.d[i];
        D.xq = w8_q[i];
        D.xs = w8_s[i];
        D.q = descs[i].q;
        D.s = descs[i].s;
        D.x = descs[i].x;
        D.y = descs[i].y;
        D.K = descs[i].K;
        D.ldx = descs[i].ldx;
        D.ldy = descs[i].ldy;
        D.N = static_cast<int32_t>(descs[i].N);
        D.nb = static_cast<int32_t>(descs[i].K / 32);
        D.S = plans[i].S;
        D.bps = plans[i].bps;
        D.tiles = plans[i].tiles;
        D.item_begin = items;
        if (plans[i].S > 1) {
            D.part = reinterpret_cast<float *>(plan_base + plans[i].part_off);
            D.tickets = reinterpret_cast<uint32_t *>(plan_base + plans[i].ticket_off);
        } else {
            D.part = nullptr;
            D.tickets = nullptr;
        }
        items += plans[i].tiles * plans[i].S;
    }
    p.status = dev_status;
    p.count = count;
    p.M = M;
    p.total_items = items;
    if (items == 0) return Q8_OK;

    if (variant == Q8_VARIANT_AUTO) variant = (M == 1) ? Q8_VARIANT_SIMT : Q8_VARIANT_MMA;
    if (variant == Q8_VARIANT_BATCH_INVARIANT) variant = Q8_VARIANT_MMA;
    if (variant == Q8_VARIANT_W8A8) {
        if (M <= 8) return run<8, Q8_VARIANT_W8A8>(p, di, stream, chained);
        if (M <= 16) return run<16, Q8_VARIANT_W8A8>(p, di, stream, chained);
        return run<32, Q8_VARIANT_W8A8>(p, di, stream, chained);
    }

    if (variant == Q8_VARIANT_MMA) {
        if (M <= 8) return run<8, Q8_VARIANT_MMA>(p, di, stream, chained);
        if (M <= 16) return run<16, Q8_VARIANT_MMA>(p, di, stream, chained);
        return run<32, Q8_VARIANT_MMA>(p, di, stream, chained);
    }
    if (M <= 1) return run<1, Q8_VARIANT_SIMT>(p, di, stream, chained);
    if (M <= 2) return run<2, Q8_VARIANT_SIMT>(p, di, stream, chained);
    if (M <= 4) return run<4, Q8_VARIANT_SIMT>(p, di, stream, chained);
    if (M <= 8) return run<8, Q8_VARIANT_SIMT>(p, di, stream, chained);
    if (M <= 16) return run<16, Q8_VARIANT_SIMT>(p, di, stream, chained);
    return run<32, Q8_VARIANT_SIMT>(p, di, stream, chained);
}

}  // namespace q8
